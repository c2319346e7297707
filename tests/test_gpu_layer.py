"""The whole layer (moe_layer_forward) against the oracle.

* The tiny fp32 layer and reduced-size bf16 layers of each workload family:
  every token checked; routing, counts bit-exact; gate weights within
  GATE_TOL; y within 1e-5 (fp32) or 2e-2 (bf16) of max |y_ref|.
* The full-size workloads (Mixtral-8x7B prefill and decode, DeepSeek-V3,
  Zipf-imbalanced) in the configuration the benchmark times: routing of
  every token bit-exact, statistics within fp32 rounding, y checked on
  sampled tokens (the oracle computes them one by one).
"""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth
from gpu_common import (BF16_TOL, F32_TOL, GATE_TOL, LayerRun, capacity_of, grouped_tiles,
                        margin_inputs, oracle_routing, oracle_rows, rel_inf, segment_edge_rows)

pytestmark = pytest.mark.gpu

SMALL = [
    synth.TINY,
    synth.Workload("mix_small", T=512, d_model=512, n_experts=8, top_k=2, d_ff=1024, seed=21),
    synth.Workload("dsv3_small", T=256, d_model=256, n_experts=256, top_k=8, d_ff=256, n_shared=1,
                   gate_mode=1, sel_bias=True, seed=22),
    synth.Workload("zipf_small", T=1024, d_model=256, n_experts=128, top_k=8, d_ff=128,
                   zipf_s=1.2, seed=23),
    synth.Workload("decode_small", T=3, d_model=512, n_experts=8, top_k=2, d_ff=512, seed=24),
    synth.Workload("f32_shared", T=100, d_model=48, n_experts=6, top_k=3, d_ff=64, n_shared=2,
                   dtype="f32", gate_mode=1, sel_bias=True, seed=25),
    # expert capacity: hot experts drop their later pairs
    synth.Workload("zipf_small_capacity", T=1024, d_model=256, n_experts=128, top_k=8, d_ff=128,
                   zipf_s=1.2, capacity_factor=1.0, seed=26),
    synth.Workload("mix_small_capacity", T=512, d_model=512, n_experts=8, top_k=2, d_ff=1024,
                   capacity_factor=0.75, seed=27),
    synth.Workload("dsv3_small_capacity_shared", T=256, d_model=256, n_experts=64, top_k=8,
                   d_ff=256, n_shared=1, gate_mode=1, sel_bias=True, capacity_factor=0.5,
                   seed=28),
    synth.Workload("f32_capacity", T=100, d_model=48, n_experts=6, top_k=3, d_ff=64, n_shared=1,
                   dtype="f32", capacity_factor=0.6, seed=29),
    # decode-sized batches: the whole layer in one cooperative kernel
    synth.Workload("decode_fused_shared_renorm", T=5, d_model=256, n_experts=16, top_k=4,
                   d_ff=256, n_shared=2, gate_mode=1, sel_bias=True, seed=30),
    synth.Workload("decode_fused_capacity", T=8, d_model=512, n_experts=4, top_k=2, d_ff=512,
                   capacity_factor=0.5, seed=31),
    synth.Workload("decode_fused_32_experts_top8", T=8, d_model=256, n_experts=32, top_k=8,
                   d_ff=256, seed=32),
    synth.Workload("decode_fused_zipf_single_token", T=1, d_model=768, n_experts=8, top_k=2,
                   d_ff=1280, zipf_s=1.2, seed=33),
    synth.Workload("decode_fused_single_token_shared_renorm", T=1, d_model=512, n_experts=32,
                   top_k=8, d_ff=768, n_shared=2, gate_mode=1, sel_bias=True, seed=34),
    synth.Workload("decode_fused_single_token_capacity", T=1, d_model=256, n_experts=4, top_k=2,
                   d_ff=512, capacity_factor=0.1, seed=35),
]


def check_layer(oracle, w, rows=None):
    inp = margin_inputs(w, oracle)
    run = LayerRun(w, inp)()
    assert run.status() == 0
    r64, idx, tw, counts, ps = oracle_routing(oracle, w, inp)
    assert np.array_equal(run.topk_idx.cpu().numpy(), idx)
    assert np.array_equal(run.counts.cpu().numpy(), counts)
    assert np.abs(run.topk_w.cpu().numpy() - tw).max() <= GATE_TOL
    assert np.allclose(run.prob_sum.cpu().numpy(), ps, rtol=1e-4, atol=1e-4)
    rows = list(range(w.T)) if rows is None else rows(idx) if callable(rows) else rows
    ref = oracle_rows(oracle, w, inp, idx, tw, rows)
    got = run.y.float().cpu().numpy()[rows]
    assert not np.isnan(got).any()
    tol = BF16_TOL if w.dtype == "bf16" else F32_TOL
    err = rel_inf(got, ref)
    assert err <= tol, err
    return run, err


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_layer_small(oracle, w):
    check_layer(oracle, w)


def test_layer_is_deterministic(oracle):
    w = SMALL[2]
    inp = margin_inputs(w, oracle)
    a = LayerRun(w, inp)()
    ya = a.y.clone()
    a()
    assert torch.equal(ya.view(torch.int16), a.y.view(torch.int16))


def test_layer_empty_batch():
    w = synth.MIXTRAL_PREFILL.replace(T=0, d_model=64, d_ff=128)
    inp = synth.make_inputs(w, "cuda")
    run = LayerRun(w, inp)()
    assert run.status() == 0
    assert run.counts.cpu().tolist() == [0] * w.n_experts


FULL = [synth.MIXTRAL_PREFILL, *synth.MIXTRAL_DECODE, synth.DEEPSEEK_V3, synth.ZIPF,
        synth.ZIPF_CAPACITY,
        # the large layers on the 256-row CTA-pair tiling, which the library
        # does not pick for them
        synth.DEEPSEEK_V3.replace(name="deepseek_v3_moe_pair_tiles", tiles=2),
        synth.ZIPF.replace(name="zipf_imbalanced_pair_tiles", tiles=2),
        synth.MIXTRAL_PREFILL.replace(name="mixtral_8x7b_prefill_pair_tiles", tiles=2)]


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_layer_full_size(oracle, w):
    """Routing of every token bit-exact; y on the owners of the first and the
    last row of every expert segment (so every segment's last, partial M
    tile is compared) and on 16 other tokens."""
    run, err = check_layer(oracle, w, lambda idx: segment_edge_rows(
        idx, w.n_experts, capacity_of(w), n_random=16, seed=w.seed, max_experts=64))
    print(f"{w.name}: rel-inf error on segment-edge and sampled tokens = {err:.3e}")


# Shapes whose grouped GEMMs give every CTA (or CTA pair) at least three
# tiles, so the persistent walk, both TMEM accumulators and their phase flips
# all run; y is compared against the oracle on every token.
MULTI_TILE = [
    # CTA pairs, 256-row tiles: ~1024 gate/up and ~256 down tiles
    (synth.Workload("multi_tile_pair", T=16384, d_model=512, n_experts=8, top_k=2, d_ff=1024,
                    seed=61, tiles=2), 256),
    # the same layer on weight-stationary CTA pairs (the library's choice):
    # ~512 gate/up and ~256 down tiles of 256 features x 256 tokens
    (synth.Workload("multi_tile_weight_pair", T=16384, d_model=512, n_experts=8, top_k=2,
                    d_ff=1024, seed=61), 256),
    # 1-CTA, 128-row tiles over ~256-row segments, a shared expert, both
    # DeepSeek-V3 routing options
    (synth.Workload("multi_tile_1cta_shared", T=4096, d_model=768, n_experts=64, top_k=4,
                    d_ff=512, n_shared=1, gate_mode=1, sel_bias=True, seed=62, tiles=1), 128),
    # a layer of ~256-row segments on weight-stationary CTA pairs (256
    # features x <= 256 tokens a tile), and a 256-expert layer of ~128-row
    # segments on them
    (synth.Workload("multi_tile_weight_pair_shared", T=4096, d_model=768, n_experts=64,
                    top_k=4, d_ff=768, n_shared=1, gate_mode=1, sel_bias=True, seed=62,
                    tiles=3), 256),
    (synth.Workload("multi_tile_weight_pair_256_experts", T=4096, d_model=1024, n_experts=256,
                    top_k=8, d_ff=512, n_shared=1, gate_mode=1, sel_bias=True, seed=66,
                    tiles=3), 256),
]


@pytest.mark.parametrize("w,tile_m", MULTI_TILE, ids=lambda v: getattr(v, "name", str(v)))
def test_layer_multi_tile_every_row(oracle, w, tile_m):
    run, err = check_layer(oracle, w)
    counts = run.counts.cpu().tolist()
    gu, dn = grouped_tiles(counts, w.T, w.n_shared, w.d_model, w.d_ff, tile_m)
    if w.tiles in (0, 3):  # weight-stationary pairs: 256 features a tile in both projections
        gu = gu * ((w.d_ff + 255) // 256) // ((w.d_ff + 127) // 128)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid = sms // 2 if tile_m == 256 else sms
    assert gu >= 3 * grid and dn >= 3 * grid, (gu, dn, grid)
    print(f"{w.name}: {gu} gate/up and {dn} down tiles over {grid} CTAs; rel-inf error {err:.3e}")


def test_layer_decode_split_k_every_row(oracle):
    """T = 64 with d_ff = 4096: swap-AB decode tiles, each projection split
    along K so that every CTA runs >= 3 (tile, split) units; y compared on
    every token."""
    w = synth.Workload("multi_unit_decode_splitk", T=64, d_model=1024, n_experts=8, top_k=2,
                       d_ff=4096, seed=63)
    run, err = check_layer(oracle, w)
    print(f"{w.name}: rel-inf error {err:.3e}")


def test_layer_replays_from_a_cuda_graph(oracle):
    """moe_layer_forward only enqueues stream-ordered work (no host syncs or
    allocations), so it can be captured in a CUDA graph; replays must give
    the eager result bit for bit, for a mid-sized batch (1-CTA tiles with a K
    split), a decode-sized one (swap-AB decode tiles, split-K) and one on
    weight-stationary CTA pairs."""
    for w in (synth.Workload("graph_prefill", T=2048, d_model=512, n_experts=4, top_k=2,
                             d_ff=512, seed=41),
              synth.Workload("graph_decode", T=2, d_model=1024, n_experts=8, top_k=2,
                             d_ff=2048, seed=42),
              synth.Workload("graph_weight_pair", T=2048, d_model=512, n_experts=4, top_k=2,
                             d_ff=512, seed=44, tiles=3)):
        inp = margin_inputs(w, oracle)
        run = LayerRun(w, inp)()
        torch.cuda.synchronize()
        eager = run.y.clone()
        run.y.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=cap):
            i = inp
            moe.moe_layer_forward(run.cfg, i["x"], i["w_router"], i["logit_bias"], i["sel_bias"],
                                  i["w_gate"], i["w_up"], i["w_down"], run.y, run.topk_idx,
                                  run.topk_w, run.counts, run.prob_sum, run.ws, cap)
        for _ in range(2):
            run.y.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(run.y.view(torch.int16), eager.view(torch.int16)), w.name


def test_decode_barrier_timeout_is_reported(oracle):
    """The single-token layer kernel's grid barriers are bounded waits. With
    one arrival withheld (an arrival no CTA makes) every wait runs out after
    1 ms: the kernel records MOE_ERR_TIMEOUT and returns, the host reads it
    from the status word, and the context stays usable -- the next call with
    the default setting succeeds and matches the oracle."""
    w = synth.Workload("barrier_timeout", T=1, d_model=512, n_experts=8, top_k=2, d_ff=1024,
                       seed=43)
    inp = margin_inputs(w, oracle)
    run = LayerRun(w, inp)()
    assert run.status() == 0
    moe.moe_set_decode_barrier_test(1, 1_000_000)
    try:
        run()
        assert run.status() == moe.MOE_ERR_TIMEOUT
    finally:
        moe.moe_set_decode_barrier_test(0, 0)
    check_layer(oracle, w)


# The row gather fused into the gate/up GEMM (weight-stationary pairs): the
# tensor cores get the same operand values as from x_perm, so y must equal
# the separate-gather layer's bit for bit, and the oracle within the bar.
FUSED_GATHER = [
    synth.Workload("fused_gather_dsv3_small", T=256, d_model=256, n_experts=256, top_k=8,
                   d_ff=256, n_shared=1, gate_mode=1, sel_bias=True, seed=22, tiles=3),
    # a K tail (d_model = 200: the last 64-wide K block is part zero-fill),
    # a shared expert, ragged segments
    synth.Workload("fused_gather_k_tail_shared", T=700, d_model=200, n_experts=6, top_k=2,
                   d_ff=136, n_shared=1, seed=45, tiles=3),
    synth.Workload("fused_gather_capacity", T=1024, d_model=256, n_experts=128, top_k=8,
                   d_ff=128, zipf_s=1.2, capacity_factor=1.0, seed=26, tiles=3),
    synth.Workload("fused_gather_multi_tile", T=16384, d_model=512, n_experts=8, top_k=2,
                   d_ff=1024, seed=61),
]


@pytest.mark.parametrize("w", FUSED_GATHER, ids=lambda w: w.name)
def test_layer_fused_gather(oracle, w):
    fused, err = check_layer(oracle, w.replace(gather=2))
    inp = fused.inp
    plain = LayerRun(w.replace(gather=1), inp)()
    assert plain.status() == 0
    assert torch.equal(fused.y.view(torch.int16), plain.y.view(torch.int16)), w.name
    print(f"{w.name}: fused gather rel-inf error {err:.3e}, equal to the separate gather")


def test_layer_fused_gather_full_size_deepseek(oracle):
    w = synth.DEEPSEEK_V3.replace(name="deepseek_v3_moe_fused_gather", gather=2)
    run, err = check_layer(oracle, w, lambda idx: segment_edge_rows(
        idx, w.n_experts, capacity_of(w), n_random=16, seed=w.seed, max_experts=64))
    plain = LayerRun(w.replace(gather=1), run.inp)()
    assert plain.status() == 0
    assert torch.equal(run.y.view(torch.int16), plain.y.view(torch.int16))


@pytest.mark.parametrize("w", [
    synth.Workload("splitk_combine_decode", T=8, d_model=1024, n_experts=8, top_k=2, d_ff=2048,
                   seed=46),
    synth.Workload("splitk_combine_decode_shared", T=40, d_model=512, n_experts=16, top_k=4,
                   d_ff=1536, n_shared=1, gate_mode=1, sel_bias=True, seed=47),
    synth.Workload("splitk_combine_1cta", T=300, d_model=768, n_experts=8, top_k=2, d_ff=1024,
                   capacity_factor=0.8, seed=48),
], ids=lambda w: w.name)
def test_layer_split_down_reduced_into_y_matches_separate_kernels(oracle, w):
    """In the layer forward a down projection split along K is summed
    straight into y (the split-K reduction and the combine in one kernel).
    The same routing through the separate entry points (moe_permute,
    moe_grouped_swiglu with its own reduction, moe_combine) must give y bit
    for bit, and y must match the oracle."""
    run, err = check_layer(oracle, w)
    cfg = run.cfg
    T, d, N, k = w.T, w.d_model, w.n_experts, w.top_k
    P = T * k
    dev = "cuda"
    inp = run.inp
    off = torch.empty(N + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(P, dtype=torch.int32, device=dev)
    inv = torch.empty(P, dtype=torch.int32, device=dev)
    xp = torch.empty(max(P, 128), d, dtype=torch.bfloat16, device=dev)
    wsp = moe.workspace(cfg, "permute")
    moe.moe_permute(cfg, inp["x"], run.topk_idx, off, sp, inv, xp, wsp)
    yp = torch.empty(P + w.n_shared * T, d, dtype=torch.bfloat16, device=dev)
    wsg = moe.workspace(cfg, "grouped")
    moe.moe_grouped_swiglu(cfg, xp, inp["x"], off, sp, run.topk_w, inp["w_gate"], inp["w_up"],
                           inp["w_down"], yp, wsg)
    y2 = torch.empty_like(run.y)
    moe.moe_combine(cfg, yp, inv, None, y2)
    assert moe.moe_stream_status(wsg) == 0
    assert torch.equal(run.y.view(torch.int16), y2.view(torch.int16)), w.name
