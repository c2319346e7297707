"""Capacity overflow rerouted in rounds (moe_reroute, moe_config.overflow)
against the oracle's reading of "Keeping the experts busy" (the extras are
dropped or rerouted).

* moe_reroute on seeded fp32 scores (ties, selection biases, NaN, a Zipf
  offset; one to many blocks, up to 256 experts; the full Zipf-imbalanced
  shape): the assignment and the round count bit-exact against
  oracle.reroute on the same scores.
* moe_permute given the assignment (-1 for dropped pairs): offsets, rows and
  inv_pos bit-exact against oracle.permute.
* The layers with overflow = reroute (bf16, FP8, NVFP4) on reduced sizes
  whose tokens have every key at least 1e-3 from every other, so that both
  sides rank all experts alike: routing bit-exact, y of every token within
  the tolerances of the other layer tests.
* The full Zipf-imbalanced layer with its 1.25x capacity rerouted: the
  layer's y equals, bit for bit, the same step run as separate calls
  (router, moe_reroute, moe_permute, moe_grouped_swiglu, moe_combine), and
  its assignment satisfies the reading's invariants.
"""
import math

import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth
from gpu_common import (BF16_TOL, GATE_TOL, LayerRun, capacity_of, cfg_of, host, margin_inputs,
                        oracle_routing, oracle_rows, rel_inf)

pytestmark = pytest.mark.gpu


def gpu_route(cfg, logits, sel_bias):
    """topk_idx from the library's router on given scores (logits_in)."""
    T, N, k = cfg.T, cfg.n_experts, cfg.top_k
    dev = logits.device
    idx = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    tw = torch.zeros((T, k), dtype=torch.float32, device=dev)
    counts = torch.zeros(N, dtype=torch.int32, device=dev)
    ps = torch.zeros(N, dtype=torch.float32, device=dev)
    ws = moe.workspace(cfg, "router", dev)
    moe.moe_router_topk(cfg, None, None, None, sel_bias, logits, None, idx, tw, counts, ps, ws)
    assert moe.moe_stream_status(ws) == 0
    return idx


def gpu_reroute(cfg, logits, sel_bias, idx):
    dev = logits.device
    assign = torch.full((cfg.T, cfg.top_k), -9, dtype=torch.int32, device=dev)
    rounds = torch.full((1,), -1, dtype=torch.int32, device=dev)
    ws = moe.workspace(cfg, "reroute", dev)
    moe.moe_reroute(cfg, logits, sel_bias, idx, assign, rounds, ws)
    st = moe.moe_stream_status(ws)
    return assign, int(rounds.item()), st


def scores(T, N, seed, zipf=0.0, nans=0):
    r = synth.random_logits(T, N, seed, ties=True)
    if zipf > 0:
        r = r + torch.tensor([-zipf * math.log(e + 1) for e in range(N)], dtype=torch.float32)
    if nans:
        g = torch.Generator().manual_seed(seed + 1)
        pos = torch.randint(0, T * N, (nans,), generator=g)
        r.view(-1)[pos] = float("nan")
    return r


# (T, N, k, capacity factor, selection bias, Zipf offset s, NaN scores)
CASES = [
    (1, 8, 2, 0.5, False, 0.0, 0),
    (7, 4, 2, 1.0, True, 0.0, 0),
    (100, 3, 1, 1.0, False, 1.2, 0),
    (333, 16, 4, 0.75, True, 1.2, 0),
    (2048, 32, 8, 1.0, False, 0.8, 0),
    (5000, 64, 6, 1.25, True, 1.2, 0),
    (3000, 256, 8, 1.0, True, 0.5, 0),
    (1500, 40, 3, 0.9, False, 1.0, 300),      # NaN scores rank below every number
    (4096, 8, 2, 0.25, False, 0.0, 0),        # heavy overflow: most pairs dropped
    (16384, 128, 8, 1.25, False, 1.2, 0),     # the Zipf-imbalanced shape and capacity
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "T{}_N{}_k{}_cf{}".format(*c[:4]))
def test_reroute_matches_oracle(oracle, case):
    T, N, k, cf, bias, zipf, nans = case
    r = scores(T, N, seed=T + N + k, zipf=zipf, nans=nans)
    sb = (torch.rand(N, generator=torch.Generator().manual_seed(N)) * 0.2 - 0.1) if bias else None
    C = moe.capacity_for(cf, T, k, N)
    cfg = moe.config(T=T, d_model=64, n_experts=N, top_k=k, d_ff=64, capacity=C,
                     overflow=moe.MOE_OVERFLOW_REROUTE)
    rd = r.cuda()
    sbd = None if sb is None else sb.cuda()
    sbn = None if sb is None else sb.numpy()
    ref_idx, _, _, _ = oracle.route(r.numpy(), k, sel_bias=sbn)
    if nans == 0:  # (the oracle's top-k does not define an order for NaN keys)
        assert np.array_equal(gpu_route(cfg, rd, sbd).cpu().numpy(), ref_idx)
    # both sides reroute from the oracle's top-k on the same scores
    assign, rounds, st = gpu_reroute(cfg, rd, sbd, torch.from_numpy(ref_idx).cuda())
    assert st == 0
    ref, ref_rounds = oracle.reroute(r.numpy(), ref_idx, C, sel_bias=sbn)
    assert np.array_equal(assign.cpu().numpy(), ref)
    assert rounds == ref_rounds
    print(f"T={T} N={N} k={k} C={C}: {rounds} rounds, "
          f"{int((ref != ref_idx).sum())} pairs moved or dropped")


def test_reroute_without_cap_and_empty(oracle):
    T, N, k = 300, 16, 4
    r = scores(T, N, seed=5)
    cfg = moe.config(T=T, d_model=64, n_experts=N, top_k=k, d_ff=64, capacity=0)
    idx = gpu_route(cfg, r.cuda(), None)
    assign, rounds, st = gpu_reroute(cfg, r.cuda(), None, idx)
    assert st == 0 and rounds == 0 and torch.equal(assign, idx)
    cfg0 = moe.config(T=0, d_model=64, n_experts=N, top_k=k, d_ff=64, capacity=3)
    e = torch.empty(0, N, device="cuda")
    assign, rounds, st = gpu_reroute(cfg0, e, None, torch.empty(0, k, dtype=torch.int32,
                                                                device="cuda"))
    assert st == 0 and rounds == 0


def test_reroute_reports_bad_expert_index(oracle):
    """An index outside [0, N) sets MOE_ERR_DEVICE_CHECK; its pair is dropped
    and nothing is written out of bounds."""
    T, N, k = 64, 8, 2
    r = scores(T, N, seed=6)
    cfg = moe.config(T=T, d_model=64, n_experts=N, top_k=k, d_ff=64, capacity=8)
    idx = gpu_route(cfg, r.cuda(), None)
    idx[3, 1] = N + 5
    idx[9, 0] = -4
    assign, rounds, st = gpu_reroute(cfg, r.cuda(), None, idx)
    assert st == moe.MOE_ERR_DEVICE_CHECK
    a = assign.cpu().numpy()
    assert a[3, 1] == -1 and a[9, 0] == -1
    assert ((a >= -1) & (a < N)).all()


def test_permute_takes_the_assignment(oracle):
    T, N, k, d = 2500, 32, 4, 64
    r = scores(T, N, seed=7, zipf=1.2)
    C = moe.capacity_for(0.5, T, k, N)  # tight: some pairs find no room
    ref_idx, _, _, _ = oracle.route(r.numpy(), k)
    a, _ = oracle.reroute(r.numpy(), ref_idx, C)
    assert (a == -1).any()
    assign = torch.from_numpy(a).cuda()
    x = torch.randn(T, d, device="cuda").to(torch.bfloat16)
    pc = moe.config(T=T, d_model=d, n_experts=N, top_k=k, d_ff=64)
    off = torch.empty(N + 1, dtype=torch.int32, device="cuda")
    sp = torch.full((T * k,), -5, dtype=torch.int32, device="cuda")
    inv = torch.full((T * k,), -5, dtype=torch.int32, device="cuda")
    xp = torch.zeros(T * k, d, dtype=torch.bfloat16, device="cuda")
    ws = moe.workspace(pc, "permute")
    moe.moe_permute(pc, x, assign, off, sp, inv, xp, ws)
    assert moe.moe_stream_status(ws) == 0
    ro, rsp, rinv = oracle.permute(a, N)
    assert np.array_equal(off.cpu().numpy(), ro)
    assert np.array_equal(sp.cpu().numpy()[:ro[N]], rsp)
    assert np.array_equal(inv.cpu().numpy(), rinv)
    rows = torch.as_tensor(rsp // k, device="cuda", dtype=torch.long)
    assert torch.equal(xp[:ro[N]], x[rows])


SMALL = [
    synth.Workload("reroute_zipf_small", T=1200, d_model=512, n_experts=16, top_k=4, d_ff=768,
                   zipf_s=1.2, capacity_factor=1.0, overflow=1, seed=61),
    synth.Workload("reroute_shared_renorm_bias", T=700, d_model=256, n_experts=12, top_k=3,
                   d_ff=512, n_shared=1, gate_mode=1, sel_bias=True, zipf_s=0.8,
                   capacity_factor=0.8, overflow=1, seed=62),
    synth.Workload("reroute_tight_drops", T=400, d_model=256, n_experts=8, top_k=2, d_ff=256,
                   zipf_s=1.5, capacity_factor=0.5, overflow=1, seed=63),
    synth.Workload("reroute_weight_pair_tiles", T=2048, d_model=512, n_experts=8, top_k=2,
                   d_ff=1024, zipf_s=1.0, capacity_factor=1.1, overflow=1, tiles=3, seed=64),
    synth.Workload("reroute_one_cta_tiles", T=900, d_model=256, n_experts=10, top_k=2,
                   d_ff=512, zipf_s=1.2, capacity_factor=0.9, overflow=1, tiles=1, seed=65),
    synth.Workload("reroute_small_batch", T=6, d_model=256, n_experts=8, top_k=2, d_ff=256,
                   zipf_s=2.0, capacity_factor=1.0, overflow=1, seed=66),
]


def oracle_assign(oracle, w, inp, idx):
    lb = None if inp["logit_bias"] is None else inp["logit_bias"].double().cpu().numpy()
    _, r32 = oracle.router_logits(host(inp["x"]), host(inp["w_router"]), lb)
    assign, rounds = oracle.reroute(r32, idx, capacity_of(w), sel_bias=host(inp["sel_bias"]))
    return assign, rounds


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("quant", ["bf16", "fp8", "nvfp4"])
def test_layer_reroute_small(oracle, w, quant):
    if quant != "bf16" and w.d_model % 16:
        pytest.skip("quantized layers need d_model % 16 == 0")
    inp = margin_inputs(w, oracle, all_keys=True)
    r64, idx, tw, counts, ps = oracle_routing(oracle, w, inp)
    assign, rounds = oracle_assign(oracle, w, inp, idx)
    moved = (assign != idx) & (assign >= 0)
    assert moved.any(), "the case is meant to reroute some pairs"
    if quant == "bf16":
        run = LayerRun(w, inp)()
        st = run.status()
        y, gidx, gtw = run.y, run.topk_idx, run.topk_w
    else:
        y, gidx, gtw, st = quantized_layer(w, inp, quant)
    assert st == 0
    assert np.array_equal(gidx.cpu().numpy(), idx)
    assert np.abs(gtw.cpu().numpy() - tw).max() <= GATE_TOL
    rows = list(range(w.T))
    ref = oracle_rows(oracle, w, inp, idx, tw, rows, assign=assign, fp8=quant == "fp8",
                      nvfp4=quant == "nvfp4")
    got = y.float().cpu().numpy()
    assert not np.isnan(got).any()
    err = rel_inf(got, ref)
    print(f"{w.name} {quant}: {rounds} rounds, {int(moved.sum())} pairs moved, "
          f"{int((assign < 0).sum())} dropped, rel-inf error {err:.3e}")
    assert err <= BF16_TOL, err


def quantized_layer(w, inp, quant):
    """moe_layer_forward_fp8 / _nvfp4 with the weights quantized by the
    library (the helpers of the FP8 and NVFP4 tests): (y, topk_idx, topk_w,
    status)."""
    from test_gpu_fp8 import quantize as quantize_fp8
    from test_gpu_nvfp4 import quantize as quantize_nvfp4
    cfg = cfg_of(w)
    T, k = w.T, w.top_k
    dev = inp["x"].device
    y = torch.full((T, w.d_model), float("nan"), dtype=torch.bfloat16, device=dev)
    idx = torch.full((T, k), -1, dtype=torch.int32, device=dev)
    tw = torch.zeros((T, k), dtype=torch.float32, device=dev)
    names = ("w_gate", "w_up", "w_down")
    if quant == "fp8":
        q = [quantize_fp8(inp[n]) for n in names]
        ws = moe.workspace(cfg, "layer_fp8", dev)
        moe.moe_layer_forward_fp8(cfg, inp["x"], inp["w_router"], inp["logit_bias"],
                                  inp["sel_bias"], *q[0], *q[1], *q[2], y, idx, tw, None, None,
                                  ws)
    else:
        q = [quantize_nvfp4(inp[n]) for n in names]
        ws = moe.workspace(cfg, "layer_nvfp4", dev)
        moe.moe_layer_forward_nvfp4(cfg, inp["x"], inp["w_router"], inp["logit_bias"],
                                    inp["sel_bias"], *q[0], *q[1], *q[2], y, idx, tw, None, None,
                                    ws)
    return y, idx, tw, moe.moe_stream_status(ws)


def test_layer_reroute_full_size_is_the_composed_step():
    """The Zipf-imbalanced layer with its 1.25x capacity rerouted, as the
    benchmark times it: y equals the same step run as separate calls, bit for
    bit, and the assignment keeps the reading's invariants (no expert over
    capacity, distinct experts per token, the cut's pairs in place, a drop
    only when every expert the token does not hold is full)."""
    w = synth.ZIPF_REROUTE
    inp = synth.make_inputs(w, "cuda")
    run = LayerRun(w, inp)()
    assert run.status() == 0
    cfg = cfg_of(w)
    T, N, k, d = w.T, w.n_experts, w.top_k, w.d_model
    C = capacity_of(w)
    dev = inp["x"].device
    logits = torch.empty(T, N, dtype=torch.float32, device=dev)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, k, dtype=torch.float32, device=dev)
    counts = torch.empty(N, dtype=torch.int32, device=dev)
    ps = torch.empty(N, dtype=torch.float32, device=dev)
    rws = moe.workspace(cfg, "router", dev)
    moe.moe_router_topk(cfg, inp["x"], inp["w_router"], inp["logit_bias"], inp["sel_bias"], None,
                        logits, idx, tw, counts, ps, rws)
    assert moe.moe_stream_status(rws) == 0
    assert torch.equal(idx, run.topk_idx)
    assign, rounds, st = gpu_reroute(cfg, logits, inp["sel_bias"], idx)
    assert st == 0
    pc = cfg_of(w.replace(capacity_factor=0.0, overflow=0))
    off = torch.empty(N + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    xp = torch.empty(T * k, d, dtype=torch.bfloat16, device=dev)
    pws = moe.workspace(pc, "permute", dev)
    moe.moe_permute(pc, inp["x"], assign, off, sp, inv, xp, pws)
    assert moe.moe_stream_status(pws) == 0
    yp = torch.empty(T * k, d, dtype=torch.bfloat16, device=dev)
    gws = moe.workspace(pc, "grouped", dev)
    moe.moe_grouped_swiglu(pc, xp, None, off, sp, tw, inp["w_gate"], inp["w_up"], inp["w_down"],
                           yp, gws)
    assert moe.moe_stream_status(gws) == 0
    y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    moe.moe_combine(pc, yp, inv, None, y)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), run.y.view(torch.int16))
    a, i0 = assign.cpu().numpy(), idx.cpu().numpy()
    load = np.bincount(a[a >= 0], minlength=N)
    assert (load <= C).all()
    rank, seen = np.empty(T * k, np.int64), np.zeros(N, np.int64)
    for p, e in enumerate(i0.ravel()):  # the cut: each expert's first C pairs
        rank[p], seen[e] = seen[e], seen[e] + 1
    keep = (rank < C).reshape(T, k)
    assert (a[keep] == i0[keep]).all()
    for t in np.nonzero((a < 0).any(axis=1))[0]:
        hold = set(i0[t].tolist()) | set(a[t][a[t] >= 0].tolist())
        assert all(load[e] == C for e in range(N) if e not in hold)
    for t in range(T):
        got = a[t][a[t] >= 0]
        assert len(set(got.tolist())) == got.size
    moved = int(((a != i0) & (a >= 0)).sum())
    print(f"{w.name}: C={C}, {rounds} rounds, {moved} pairs rerouted, "
          f"{int((a < 0).sum())} dropped")
    assert moved > 0
