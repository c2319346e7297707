"""FP8 (E4M3) experts, through the C ABI.

* moe_quantize_fp8: codes and row scales bit-exact against the oracle's
  E4M3 quantizer, on rows that hit zeros, negative zero, ties, saturation and
  subnormal codes.
* moe_layer_forward_fp8: weights quantized with moe_quantize_fp8; routing
  bit-exact (it is the bf16 router), y against the oracle's FP8 layer, which
  quantizes the same bf16 weights and tokens itself and rounds H through
  bf16 and E4M3 as the GPU does. Codes of x and W agree bit for bit (first
  test); an H element near an E4M3 rounding boundary may round the other
  way when the fp32 and fp64 sums differ, which the 2e-2 bar covers.
"""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth
from gpu_common import (BF16_TOL, capacity_of, cfg_of, grouped_tiles, host, margin_inputs,
                        oracle_routing, oracle_rows, rel_inf, segment_edge_rows)

pytestmark = pytest.mark.gpu


def quantize(t):
    rows = t.shape[0] if t.dim() == 2 else t.shape[0] * t.shape[1]
    cols = t.shape[-1]
    q = torch.empty((rows, cols), dtype=torch.uint8, device=t.device)
    sc = torch.empty(rows, dtype=torch.float32, device=t.device)
    moe.moe_quantize_fp8(t.reshape(rows, cols), q, sc)
    return q, sc


# 300 rows take the block-a-row kernel, 1300 the warp-a-row one
@pytest.mark.parametrize("n_rows", [300, 1300])
def test_quantize_fp8_is_bit_exact(oracle, n_rows):
    g = torch.Generator(device="cuda").manual_seed(5)
    m = torch.randn(n_rows, 264, generator=g, device="cuda") * 3
    m[0] = 0.0
    m[1] = -0.0
    m[2, :8] = torch.tensor([448, 464, 1e4, -1e4, 2 ** -9, 2 ** -11, 1.0625, -1.1875])
    m[3] *= 2.0 ** -20          # tiny row: codes from a large 448 / amax
    m[4] *= 2.0 ** 20
    m[5, ::3] = 0.0
    x = m.to(torch.bfloat16)
    q, sc = quantize(x)
    torch.cuda.synchronize()
    rq, rsc = oracle.quantize_rows_e4m3(host(x))
    assert np.array_equal(sc.cpu().numpy(), rsc)
    assert np.array_equal(q.cpu().numpy(), rq)


class Fp8Run:
    def __init__(self, w, inp):
        self.cfg = cfg_of(w)
        T, N, k = w.T, w.n_experts, w.top_k
        self.wq = [quantize(inp[n]) for n in ("w_gate", "w_up", "w_down")]
        self.y = torch.full((T, w.d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        self.tw = torch.zeros((T, k), device="cuda")
        self.counts = torch.full((N,), -1, dtype=torch.int32, device="cuda")
        self.ps = torch.empty(N, device="cuda")
        self.ws = moe.workspace(self.cfg, "layer_fp8")
        self.inp = inp

    def __call__(self):
        i = self.inp
        (gq, gs), (uq, us), (dq, ds) = self.wq
        moe.moe_layer_forward_fp8(self.cfg, i["x"], i["w_router"], i["logit_bias"], i["sel_bias"],
                                  gq, gs, uq, us, dq, ds, self.y, self.idx, self.tw, self.counts,
                                  self.ps, self.ws)
        return self


def check_fp8(oracle, w, rows=None):
    inp = margin_inputs(w, oracle)
    run = Fp8Run(w, inp)()
    assert moe.moe_stream_status(run.ws) == 0
    r64, idx, tw, counts, ps = oracle_routing(oracle, w, inp)
    assert np.array_equal(run.idx.cpu().numpy(), idx)
    assert np.array_equal(run.counts.cpu().numpy(), counts)
    rows = list(range(w.T)) if rows is None else rows(idx) if callable(rows) else rows
    ref = oracle_rows(oracle, w, inp, idx, tw, rows, fp8=True)
    got = run.y.float().cpu().numpy()[rows]
    assert not np.isnan(got).any()
    err = rel_inf(got, ref)
    print(f"{w.name}: FP8 rel-inf error {err:.3e}")
    assert err <= BF16_TOL, err
    return err, counts


SMALL = [
    synth.Workload("fp8_mix_small", T=512, d_model=512, n_experts=8, top_k=2, d_ff=1024, seed=51),
    synth.Workload("fp8_dsv3_small", T=256, d_model=256, n_experts=64, top_k=8, d_ff=256,
                   n_shared=1, gate_mode=1, sel_bias=True, seed=52),
    synth.Workload("fp8_decode_small", T=3, d_model=512, n_experts=8, top_k=2, d_ff=512, seed=53),
    synth.Workload("fp8_decode_shared", T=17, d_model=256, n_experts=16, top_k=4, d_ff=384,
                   n_shared=2, seed=54),
    synth.Workload("fp8_capacity", T=1024, d_model=256, n_experts=128, top_k=8, d_ff=128,
                   zipf_s=1.2, capacity_factor=1.0, seed=55),
    synth.Workload("fp8_ragged_k", T=300, d_model=208, n_experts=8, top_k=2, d_ff=144, seed=56),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_layer_fp8_small(oracle, w):
    check_fp8(oracle, w)


FULL = [synth.MIXTRAL_PREFILL, synth.MIXTRAL_DECODE[0], synth.MIXTRAL_DECODE[3], synth.DEEPSEEK_V3,
        # CTA-pair tiles: >= 384 pairs per expert and no K split possible
        # (fp32 partial rows of either projection would exceed 64 MB)
        synth.Workload("fp8_pair_tiles", T=4096, d_model=2176, n_experts=8, top_k=2, d_ff=1024,
                       n_shared=1, seed=58, tiles=2),
        # weight-stationary CTA pairs: 256 experts of ~200 rows, a K tail
        synth.Workload("fp8_weight_pair_tiles", T=4096, d_model=1600, n_experts=256, top_k=8,
                       d_ff=512, n_shared=1, gate_mode=1, sel_bias=True, seed=59, tiles=3)]


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_layer_fp8_full_size(oracle, w):
    check_fp8(oracle, w, lambda idx: segment_edge_rows(idx, w.n_experts, capacity_of(w),
                                                        n_random=8, seed=w.seed, max_experts=8))


def test_layer_fp8_pair_multi_tile_every_row(oracle):
    """E4M3 on CTA pairs with every pair running >= 3 tiles of each
    projection (persistent walk, both accumulators); y compared on every
    token."""
    w = synth.Workload("fp8_multi_tile_pair", T=16384, d_model=512, n_experts=8, top_k=2,
                       d_ff=1024, seed=64, tiles=2)
    _, counts = check_fp8(oracle, w)
    gu, dn = grouped_tiles(counts, w.T, w.n_shared, w.d_model, w.d_ff, 256)
    grid = torch.cuda.get_device_properties(0).multi_processor_count // 2
    assert gu >= 3 * grid and dn >= 3 * grid, (gu, dn, grid)


def test_layer_fp8_refuses_unaligned_rows():
    w = synth.Workload("fp8_bad", T=4, d_model=200, n_experts=4, top_k=2, d_ff=64, seed=57)
    assert moe.workspace_size(cfg_of(w), "layer_fp8") == 0
