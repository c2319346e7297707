"""NVFP4 experts, through the C ABI.

* moe_quantize_nvfp4: packed E2M1 codes, E4M3 block scales and fp32 row
  scales bit-exact against the oracle's NVFP4 quantizer, on rows that hit
  zeros, negative zero, code ties, saturation, subnormal block scales and
  blocks whose scale rounds to zero; the block-scale padding is zero.
* moe_layer_forward_nvfp4: weights quantized with moe_quantize_nvfp4;
  routing bit-exact (it is the bf16 router), y against the oracle's NVFP4
  layer, which quantizes the same bf16 weights and tokens itself and rounds
  H through bf16 and NVFP4 as the GPU does. Codes of x and W agree bit for
  bit (first test); an H element near an E2M1 or block-scale rounding
  boundary may round the other way when the fp32 and fp64 sums differ,
  which the 2e-2 bar covers. The shapes cover K tails inside a 256-element
  block, partial N tiles, shared experts, capacity drops, the split-K path
  at two batch sizes, decode-sized batches and the full Mixtral- and
  DeepSeek-V3-shaped layers.
"""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth
from gpu_common import (BF16_TOL, capacity_of, cfg_of, grouped_tiles, host, margin_inputs,
                        oracle_routing, oracle_rows, rel_inf, sample_rows, segment_edge_rows)

pytestmark = pytest.mark.gpu


def quantize(t):
    rows = t.shape[0] if t.dim() == 2 else t.shape[0] * t.shape[1]
    cols = t.shape[-1]
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=t.device)
    sf = torch.full((rows, moe.moe_nvfp4_scale_stride(cols)), 0xFF, dtype=torch.uint8,
                    device=t.device)
    sc = torch.empty(rows, dtype=torch.float32, device=t.device)
    moe.moe_quantize_nvfp4(t.reshape(rows, cols), q, sf, sc)
    return q, sf, sc


def unpack(q):
    """One E2M1 code per element from the packed [rows, cols/2] bytes."""
    q = q.cpu().numpy()
    out = np.empty((q.shape[0], 2 * q.shape[1]), np.uint8)
    out[:, 0::2] = q & 0x0F
    out[:, 1::2] = q >> 4
    return out


def test_scale_stride():
    assert moe.moe_nvfp4_scale_stride(4096) == 256
    assert moe.moe_nvfp4_scale_stride(320) == 32
    assert moe.moe_nvfp4_scale_stride(16) == 16
    assert moe.moe_nvfp4_scale_stride(0) == 0


# 300 rows take the block-a-row kernel, 1300 the warp-a-row one
@pytest.mark.parametrize("n_rows", [300, 1300])
def test_quantize_nvfp4_is_bit_exact(oracle, n_rows):
    g = torch.Generator(device="cuda").manual_seed(7)
    m = torch.randn(n_rows, 320, generator=g, device="cuda") * 3
    m[0] = 0.0
    m[1] = -0.0
    # a block of E2M1 ties and saturation against a block max of 6
    m[2, :16] = torch.tensor([6, 5, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25,
                              -5, -3.5, -0.25, 7, 0, -0.0, 4.5, 1e-3])
    m[3] *= 2.0 ** -20          # tiny row: codes from a large 2688 / amax
    m[4] *= 2.0 ** 20
    m[5, ::3] = 0.0
    m[6, 16:] *= 1e-5           # blocks far below the row max: subnormal block scales
    m[9, 16:] *= 3e-5
    m[7, 32:] *= 1e-7           # ... and block scales that round to zero
    m[8, :16] = -0.0            # a zero block in a nonzero row
    x = m.to(torch.bfloat16)
    q, sf, sc = quantize(x)
    torch.cuda.synchronize()
    rq, rbs, rsc = oracle.quantize_rows_nvfp4(host(x))
    assert np.array_equal(sc.cpu().numpy(), rsc)
    nb = x.shape[1] // 16
    sfh = sf.cpu().numpy()
    assert np.array_equal(sfh[:, :nb], rbs)
    assert not sfh[:, nb:].any(), "block-scale padding must be zero"
    assert np.array_equal(unpack(q), rq)
    # the cases above do reach every E2M1 code and subnormal block scales
    assert set(np.unique(rq).tolist()) == set(range(16))
    assert (rbs[rbs > 0] < 8).any()


class Nvfp4Run:
    def __init__(self, w, inp):
        self.cfg = cfg_of(w)
        T, N, k = w.T, w.n_experts, w.top_k
        self.wq = [quantize(inp[n]) for n in ("w_gate", "w_up", "w_down")]
        self.y = torch.full((T, w.d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        self.tw = torch.zeros((T, k), device="cuda")
        self.counts = torch.full((N,), -1, dtype=torch.int32, device="cuda")
        self.ps = torch.empty(N, device="cuda")
        self.ws = moe.workspace(self.cfg, "layer_nvfp4")
        self.inp = inp

    def __call__(self):
        i = self.inp
        (gq, gsf, gs), (uq, usf, us), (dq, dsf, ds) = self.wq
        moe.moe_layer_forward_nvfp4(self.cfg, i["x"], i["w_router"], i["logit_bias"],
                                    i["sel_bias"], gq, gsf, gs, uq, usf, us, dq, dsf, ds, self.y,
                                    self.idx, self.tw, self.counts, self.ps, self.ws)
        return self


def check_nvfp4(oracle, w, rows=None):
    inp = margin_inputs(w, oracle)
    run = Nvfp4Run(w, inp)()
    assert moe.moe_stream_status(run.ws) == 0
    r64, idx, tw, counts, ps = oracle_routing(oracle, w, inp)
    assert np.array_equal(run.idx.cpu().numpy(), idx)
    assert np.array_equal(run.counts.cpu().numpy(), counts)
    rows = list(range(w.T)) if rows is None else rows(idx) if callable(rows) else rows
    ref = oracle_rows(oracle, w, inp, idx, tw, rows, nvfp4=True)
    got = run.y.float().cpu().numpy()[rows]
    assert not np.isnan(got).any()
    err = rel_inf(got, ref)
    print(f"{w.name}: NVFP4 rel-inf error {err:.3e}")
    assert err <= BF16_TOL, err
    return err, counts


SMALL = [
    synth.Workload("nvf4_mix_small", T=512, d_model=512, n_experts=8, top_k=2, d_ff=1024,
                   seed=61),
    synth.Workload("nvf4_dsv3_small", T=256, d_model=256, n_experts=64, top_k=8, d_ff=256,
                   n_shared=1, gate_mode=1, sel_bias=True, seed=62),
    synth.Workload("nvf4_decode_small", T=3, d_model=512, n_experts=8, top_k=2, d_ff=512,
                   seed=63),
    synth.Workload("nvf4_decode_shared", T=17, d_model=256, n_experts=16, top_k=4, d_ff=384,
                   n_shared=2, seed=64),
    synth.Workload("nvf4_capacity", T=1024, d_model=256, n_experts=128, top_k=8, d_ff=256,
                   zipf_s=1.2, capacity_factor=1.0, seed=65),
    # K tails inside a 256-element block (320 = 256 + 64, 448 = 256 + 192)
    # and partial N tiles of both projections
    synth.Workload("nvf4_ragged_k", T=300, d_model=320, n_experts=8, top_k=2, d_ff=448, seed=66),
    # split-K: fewer tiles than two waves and 16 K blocks of 256 in both
    # projections, so both write fp32 partial rows (T = 8 and T = 96)
    synth.Workload("nvf4_split_k", T=8, d_model=4096, n_experts=8, top_k=2, d_ff=4096,
                   n_shared=1, seed=67),
    synth.Workload("nvf4_split_k_prefill", T=96, d_model=4096, n_experts=8, top_k=2, d_ff=2048,
                   n_shared=1, seed=73),
    # decode-sized batches: segments of 1 to 64 rows (a 40-row shared
    # segment; routed segments of more than 32 rows) with K tails and partial
    # feature tiles
    synth.Workload("nvf4_decode_ragged_k", T=40, d_model=320, n_experts=8, top_k=2, d_ff=448,
                   n_shared=1, seed=74),
    synth.Workload("nvf4_decode_t64_small", T=64, d_model=512, n_experts=4, top_k=2, d_ff=512,
                   seed=75),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_layer_nvfp4_small(oracle, w):
    check_nvfp4(oracle, w)


# A large batch with a shared expert that reads x, and a K tail in the gate/up
# projection (2176 = 8*256 + 128)
LARGE = synth.Workload("nvf4_large_shared_k_tail", T=4096, d_model=2176, n_experts=8, top_k=2,
                      d_ff=1024, n_shared=1, seed=70)
FULL = [synth.MIXTRAL_PREFILL, synth.MIXTRAL_DECODE[0], synth.MIXTRAL_DECODE[3],
        synth.DEEPSEEK_V3, LARGE]


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_layer_nvfp4_full_size(oracle, w):
    check_nvfp4(oracle, w, lambda idx: segment_edge_rows(idx, w.n_experts, capacity_of(w),
                                                          n_random=8, seed=w.seed, max_experts=8))


def test_layer_nvfp4_multi_tile_every_row(oracle):
    """NVFP4 on 1-CTA tiles with every CTA running >= 3 tiles of each
    projection (persistent walk, the single accumulator's phase flips, the
    scale buffers' reuse across tiles); y compared on every token."""
    w = synth.Workload("nvf4_multi_tile", T=8192, d_model=1024, n_experts=8, top_k=2,
                       d_ff=1024, seed=65)
    _, counts = check_nvfp4(oracle, w)
    gu, dn = grouped_tiles(counts, w.T, w.n_shared, w.d_model, w.d_ff, 128)
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    assert gu >= 3 * grid and dn >= 3 * grid, (gu, dn, grid)


def test_layer_nvfp4_refuses_unsupported_shapes():
    for d, f in ((320, 200), (200, 256), (128, 256), (256, 128)):
        w = synth.Workload("nvf4_bad", T=4, d_model=d, n_experts=4, top_k=2, d_ff=f, seed=68)
        assert moe.workspace_size(cfg_of(w), "layer_nvfp4") == 0


@pytest.mark.parametrize("w,nrows", [
    (synth.Workload("nvf4_block_pattern", T=384, d_model=512, n_experts=8, top_k=2, d_ff=768,
                    n_shared=1, seed=69), None),
    (LARGE.replace(name="nvf4_block_pattern_large", seed=71), 96),
    (synth.Workload("nvf4_block_pattern_decode", T=48, d_model=512, n_experts=4, top_k=2,
                    d_ff=768, n_shared=1, seed=72), None),
], ids=lambda v: v.name if hasattr(v, "name") else str(v))
def test_layer_nvfp4_block_scale_pattern(oracle, w, nrows):
    """Expert weights whose 16-element blocks differ by up to 2^8 from one
    row and block to the next, so that a block scale applied to the wrong
    row or K block of either operand would be far outside the bar. Routing
    is untouched (the router weights are not changed)."""
    inp = margin_inputs(w, oracle)
    for name in ("w_gate", "w_up", "w_down"):
        t = inp[name]
        rows = torch.arange(t.shape[1], device=t.device).view(1, -1, 1)
        blocks = torch.arange(t.shape[2] // 16, device=t.device).view(1, 1, -1)
        expo = ((rows * 7 + blocks * 3) % 9 - 4).float()
        f = torch.exp2(expo).repeat_interleave(16, dim=2)
        inp[name] = (t.float() * f).to(t.dtype)
    run = Nvfp4Run(w, inp)()
    assert moe.moe_stream_status(run.ws) == 0
    _, idx, tw, _, _ = oracle_routing(oracle, w, inp)
    assert np.array_equal(run.idx.cpu().numpy(), idx)
    rows = list(range(w.T)) if nrows is None else sample_rows(w.T, nrows, seed=w.seed)
    ref = oracle_rows(oracle, w, inp, idx, tw, rows, nvfp4=True)
    err = rel_inf(run.y.float().cpu().numpy()[rows], ref)
    print(f"{w.name}: NVFP4 rel-inf error {err:.3e}")
    assert err <= BF16_TOL, err
