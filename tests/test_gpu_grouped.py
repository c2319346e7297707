"""K3/K4 (and K7) parity: every expert's SwiGLU FFN over its ragged row
segment, gate-weighted, against the oracle's expert on the same rows.

Shapes span several 128-row tiles, ragged segment ends, empty experts, a
K not a multiple of the 64-wide K block, an output width not a multiple of
the tile width, a shared expert, and batches small enough that tiles are
split along K (decode). The oracle's own grouping (rows in
expert order) decides which pair each output row belongs to."""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth
from gpu_common import BF16_TOL, F32_TOL, host, rel_inf
from test_gpu_permute import random_idx

pytestmark = pytest.mark.gpu

CASES = [
    # name, T, d, N, k, d_ff, shared, dtype, skew
    ("ragged_5x", 300, 256, 5, 2, 384, 0, "bf16", 0.0),
    ("shared", 200, 128, 6, 3, 256, 1, "bf16", 0.0),
    ("one_token", 1, 512, 8, 2, 1024, 0, "bf16", 0.0),
    ("k_n_tails", 130, 200, 3, 2, 136, 1, "bf16", 0.0),
    ("hot_expert", 1000, 256, 4, 1, 128, 0, "bf16", 6.0),
    ("many_experts", 600, 128, 64, 4, 128, 2, "bf16", 1.2),
    # few tiles: the K dimension is split across CTAs and the partials summed
    ("splitk_decode_T1", 1, 4096, 8, 2, 14336, 0, "bf16", 0.0),
    ("splitk_T5_shared", 5, 1024, 8, 2, 2048, 1, "bf16", 0.0),
    ("splitk_ragged_k", 20, 1000, 16, 4, 520, 0, "bf16", 0.0),
    # large segments (>= 384 rows per expert on average): 256-row tiles on CTA pairs
    ("pair_tiles", 2000, 256, 4, 2, 384, 0, "bf16", 0.0),
    ("pair_ragged_shared", 1500, 200, 3, 2, 136, 1, "bf16", 0.0),
    ("pair_skewed", 3000, 128, 8, 2, 256, 0, "bf16", 1.5),
    ("f32", 64, 64, 4, 2, 128, 0, "f32", 0.0),
    ("f32_shared", 90, 40, 5, 2, 48, 1, "f32", 0.0),
]


# The same shapes with a named tiling: 256-row CTA pairs, and weight-stationary
# CTA pairs (token tiles cut to multiples of 16 rows), whatever the library
# would choose for them.
FORCED = [c + (t,) for c in CASES if c[7] == "bf16" for t in (2, 3)]


@pytest.mark.parametrize("name,T,d,N,k,d_ff,s,dtype,skew,tiles", FORCED,
                         ids=[f"{c[0]}-tiles{c[-1]}" for c in FORCED])
def test_grouped_swiglu_tilings_match_oracle(oracle, name, T, d, N, k, d_ff, s, dtype, skew, tiles):
    test_grouped_swiglu_matches_oracle(oracle, name, T, d, N, k, d_ff, s, dtype, skew, tiles)


@pytest.mark.parametrize("name,T,d,N,k,d_ff,s,dtype,skew", CASES, ids=[c[0] for c in CASES])
def test_grouped_swiglu_matches_oracle(oracle, name, T, d, N, k, d_ff, s, dtype, skew, tiles=0):
    w = synth.Workload(name, T=T, d_model=d, n_experts=N, top_k=k, d_ff=d_ff, n_shared=s,
                       dtype=dtype, seed=T + d)
    inp = synth.make_inputs(w, "cuda")
    idx = random_idx(T, N, k, seed=T, skew=skew)
    gw = np.random.default_rng(T).uniform(0.05, 1.0, (T, k)).astype(np.float32)
    cfg = moe.config(T=T, d_model=d, n_experts=N, top_k=k, d_ff=d_ff, n_shared=s,
                     dtype=moe.MOE_BF16 if dtype == "bf16" else moe.MOE_F32, tiles=tiles)
    P = T * k
    dev = "cuda"
    off = torch.empty(N + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(P, dtype=torch.int32, device=dev)
    inv = torch.empty(P, dtype=torch.int32, device=dev)
    xp = torch.empty(P, d, dtype=w.torch_dtype, device=dev)
    ws = moe.workspace(cfg, "permute")
    moe.moe_permute(cfg, inp["x"], torch.from_numpy(idx).cuda(), off, sp, inv, xp, ws)
    assert moe.moe_stream_status(ws) == 0
    yp = torch.full((P + s * T, d), float("nan"), dtype=w.torch_dtype, device=dev)
    wsg = moe.workspace(cfg, "grouped")
    moe.moe_grouped_swiglu(cfg, xp, inp["x"] if s else None, off, sp, torch.from_numpy(gw).cuda(),
                           inp["w_gate"], inp["w_up"], inp["w_down"], yp, wsg)
    assert moe.moe_stream_status(wsg) == 0
    got = yp.float().cpu().numpy()

    # Oracle: each routed row r holds pair p = r_sp[r] (the oracle's grouping).
    _, r_sp, _ = oracle.permute(idx, N)
    xh = host(inp["x"])
    wg, wu, wd = host(inp["w_gate"]), host(inp["w_up"]), host(inp["w_down"])
    ref = np.empty((P + s * T, d))
    xrow = lambda t: xh[t].astype(np.float64) if xh.dtype != np.uint16 else \
        (xh[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for r in range(P):
        p = r_sp[r]
        t, slot = divmod(int(p), k)
        e = idx[t, slot]
        ref[r] = gw[t, slot] * oracle.expert_swiglu(xrow(t), wg[e], wu[e], wd[e])
    for j in range(s):
        for t in range(T):
            ref[P + j * T + t] = oracle.expert_swiglu(xrow(t), wg[N + j], wu[N + j], wd[N + j])
    tol = BF16_TOL if dtype == "bf16" else F32_TOL
    assert not np.isnan(got).any()
    assert rel_inf(got, ref) <= tol, rel_inf(got, ref)
    # every segment on its own scale as well
    r_off = np.concatenate([[0], np.cumsum(np.bincount(idx.ravel(), minlength=N))])
    for e in range(N):
        a, b = r_off[e], r_off[e + 1]
        if b > a:
            assert rel_inf(got[a:b], ref[a:b]) <= tol, (e, rel_inf(got[a:b], ref[a:b]))


def test_bad_offsets_are_reported():
    """Offsets that decrease are caught on the device: the status word says so
    and no GEMM tile runs."""
    T, d, N, k, d_ff = 64, 64, 4, 2, 128
    cfg = moe.config(T=T, d_model=d, n_experts=N, top_k=k, d_ff=d_ff)
    w = synth.Workload("bad", T=T, d_model=d, n_experts=N, top_k=k, d_ff=d_ff, seed=1)
    inp = synth.make_inputs(w, "cuda")
    xp = torch.zeros(T * k, d, dtype=torch.bfloat16, device="cuda")
    off = torch.tensor([0, 50, 20, 100, 128], dtype=torch.int32, device="cuda")
    yp = torch.full((T * k, d), 7.0, dtype=torch.bfloat16, device="cuda")
    ws = moe.workspace(cfg, "grouped")
    moe.moe_grouped_swiglu(cfg, xp, None, off, None, None, inp["w_gate"], inp["w_up"], inp["w_down"],
                           yp, ws)
    assert moe.moe_stream_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    assert (yp.float() == 7.0).all()
