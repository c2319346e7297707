"""K1 parity: router scores, top-k, gate weights and statistics against the
oracle, through the C ABI.

* Given fp32 scores (parity mode, with many exact ties in scores and keys):
  indices and counts bit-exact, weights and probability sums within fp32
  rounding.
* From x and W_r (the fused router GEMM): indices bit-exact on inputs with
  an order margin >= 1e-3; scores within fp32 accumulation error.
"""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth
from gpu_common import GATE_TOL, SCORE_TOL, cfg_of, host, margin_inputs, oracle_routing

pytestmark = pytest.mark.gpu


def run_router(cfg, x=None, w=None, logit_bias=None, sel_bias=None, logits_in=None):
    T, N, k = cfg.T, cfg.n_experts, cfg.top_k
    dev = "cuda"
    out = dict(
        logits=torch.full((T, N), float("nan"), device=dev),
        idx=torch.full((T, k), -1, dtype=torch.int32, device=dev),
        w=torch.full((T, k), float("nan"), device=dev),
        counts=torch.full((N,), -5, dtype=torch.int32, device=dev),
        prob_sum=torch.full((N,), float("nan"), device=dev),
    )
    ws = moe.workspace(cfg, "router", dev)
    moe.moe_router_topk(cfg, x, w, logit_bias, sel_bias, logits_in, out["logits"], out["idx"],
                        out["w"], out["counts"], out["prob_sum"], ws)
    assert moe.moe_stream_status(ws) == 0
    return {k_: v.cpu() for k_, v in out.items()}


PARITY_CASES = [
    # T, N, k, gate_mode, sel_bias
    (1, 4, 2, 0, False),
    (3, 8, 2, 1, False),
    (17, 8, 2, 0, True),
    (64, 4, 2, 0, False),
    (50, 1, 1, 0, False),
    (40, 8, 8, 1, True),      # k = N
    (77, 33, 3, 0, True),     # N not a multiple of 32
    (1000, 128, 8, 0, False),
    (333, 256, 8, 1, True),
    (4096, 256, 8, 1, True),
    (2049, 64, 6, 0, True),
]


@pytest.mark.parametrize("T,N,k,mode,use_sb", PARITY_CASES)
def test_routing_given_scores_is_bit_exact(oracle, T, N, k, mode, use_sb):
    logits = synth.random_logits(T, N, seed=T * 1000 + N, ties=True)
    sb = None
    if use_sb:
        sb = synth.random_logits(1, N, seed=N + 7, ties=True)[0] * 0.05
        sb[::3] = 0.0  # exact key ties through the bias too
    cfg = moe.config(T=T, d_model=8, n_experts=N, top_k=k, d_ff=8, gate_mode=mode)
    got = run_router(cfg, logits_in=logits.cuda(), sel_bias=None if sb is None else sb.cuda())
    idx, tw, counts, ps = oracle.route(logits.numpy(), k, mode, None if sb is None else sb.numpy())
    assert np.array_equal(got["idx"].numpy(), idx)
    assert np.array_equal(got["counts"].numpy(), counts)
    assert np.array_equal(got["logits"].numpy(), logits.numpy())
    assert np.abs(got["w"].numpy() - tw).max() <= 2e-6
    assert np.allclose(got["prob_sum"].numpy(), ps, rtol=1e-4, atol=1e-4)


def test_routing_is_deterministic():
    T, N, k = 4096, 256, 8
    logits = synth.random_logits(T, N, seed=5).cuda()
    cfg = moe.config(T=T, d_model=8, n_experts=N, top_k=k, d_ff=8, gate_mode=1)
    a = run_router(cfg, logits_in=logits)
    b = run_router(cfg, logits_in=logits)
    for key in a:
        assert torch.equal(a[key], b[key]), key


GEMM_CASES = [
    synth.Workload("r_small_f32", T=129, d_model=64, n_experts=4, top_k=2, d_ff=8, dtype="f32", seed=11),
    synth.Workload("r_mix", T=300, d_model=256, n_experts=8, top_k=2, d_ff=8, seed=12),
    synth.Workload("r_dsv3", T=200, d_model=512, n_experts=256, top_k=8, d_ff=8, gate_mode=1,
                   sel_bias=True, seed=13),
    synth.Workload("r_zipf", T=257, d_model=1024, n_experts=128, top_k=8, d_ff=8, zipf_s=1.2, seed=14),
    synth.Workload("r_n40", T=65, d_model=136, n_experts=40, top_k=5, d_ff=8, dtype="f32", seed=15),
    # bf16 with more than 32 experts: the tensor-core router. Ragged expert
    # count, K not a multiple of the 64-wide K block, partial token tiles,
    # one token, and more than 32 token tiles (block sums reduced separately).
    synth.Workload("r_tc_n33", T=130, d_model=136, n_experts=33, top_k=3, d_ff=8, sel_bias=True,
                   seed=16),
    synth.Workload("r_tc_one_token", T=1, d_model=64, n_experts=129, top_k=8, d_ff=8, gate_mode=1,
                   seed=17),
    synth.Workload("r_tc_n200_many_tiles", T=4500, d_model=200, n_experts=200, top_k=6, d_ff=8,
                   zipf_s=1.2, seed=18),
    synth.DEEPSEEK_V3.replace(name="r_dsv3_full_size", d_ff=8),   # d_model = 7168
    # bf16 with up to 32 experts and at least 256 tokens: the mma.sync kernel
    # (16-token tiles, the warps splitting d_model); below 256 tokens the
    # warp kernel, one to eight warps per token group.
    synth.Workload("r_warp_many_groups", T=4000, d_model=4096, n_experts=8, top_k=2, d_ff=8,
                   seed=19),
    # two 8-expert column tiles, four of their rows past N; 65 vectors a row
    # (a partial 32-element chunk); an odd T (the last tile holds 13 tokens)
    synth.Workload("r_stream_n12_ragged_d", T=2301, d_model=520, n_experts=12, top_k=3, d_ff=8,
                   gate_mode=1, sel_bias=True, seed=26),
    synth.Workload("r_warp_one_expert", T=2100, d_model=256, n_experts=1, top_k=1, d_ff=8, seed=21),
    synth.Workload("r_warp_n32", T=9000, d_model=256, n_experts=32, top_k=8, d_ff=8, seed=22),
    synth.Workload("r_warp_n16_grid_stride", T=19500, d_model=128, n_experts=16, top_k=4, d_ff=8,
                   seed=23),
    synth.Workload("r_warp_decode", T=1, d_model=4096, n_experts=8, top_k=2, d_ff=8, seed=24),
    synth.Workload("r_warp_n20", T=129, d_model=520, n_experts=20, top_k=5, d_ff=8,
                   gate_mode=1, sel_bias=True, zipf_s=1.2, seed=25),
]


@pytest.mark.parametrize("w", GEMM_CASES, ids=lambda w: w.name)
def test_router_gemm_routes_like_the_oracle(oracle, w):
    inp = margin_inputs(w, oracle)
    cfg = cfg_of(w)
    got = run_router(cfg, inp["x"], inp["w_router"], inp["logit_bias"], inp["sel_bias"])
    r64, idx, tw, counts, ps = oracle_routing(oracle, w, inp)
    assert np.array_equal(got["idx"].numpy(), idx)
    assert np.array_equal(got["counts"].numpy(), counts)
    assert np.abs(got["logits"].numpy() - r64).max() <= SCORE_TOL
    assert np.abs(got["w"].numpy() - tw).max() <= GATE_TOL
    assert np.allclose(got["prob_sum"].numpy(), ps, rtol=1e-4, atol=1e-4)


@pytest.mark.parametrize("N,k,mode,T", [(64, 8, 1, 300), (256, 8, 0, 300), (48, 5, 0, 300),
                                        (8, 2, 0, 300), (8, 2, 0, 2500), (32, 6, 1, 2500)])
def test_router_gemm_breaks_exact_ties_by_index(oracle, N, k, mode, T):
    """Small-integer x and W_r make every product and sum exact in fp32, so
    the scores computed on the tensor cores equal the oracle's bit for bit
    and tie often (many experts share a score); duplicated router rows and a
    selection bias on a 1/4 grid add exact key ties. Selection must keep the
    lower expert index on every tie, as the oracle does."""
    d = 256
    g = torch.Generator().manual_seed(N * 31 + k)
    x = torch.randint(-2, 3, (T, d), generator=g).to(torch.bfloat16)
    base = torch.randint(-1, 2, (max(N // 4, 1), d), generator=g)
    W = base.repeat(4, 1)[:N][torch.randperm(N, generator=g)].to(torch.bfloat16)
    sb = (torch.randint(-2, 3, (N,), generator=g).float() * 0.25)
    sb[::2] = 0.0
    cfg = moe.config(T=T, d_model=d, n_experts=N, top_k=k, d_ff=8, dtype=moe.MOE_BF16,
                     gate_mode=mode)
    got = run_router(cfg, x.cuda(), W.cuda(), None, sb.cuda())
    r64, r32 = oracle.router_logits(host(x), host(W), None)
    assert np.array_equal(got["logits"].numpy(), r32)
    idx, tw, counts, ps = oracle.route(r32, k, mode, sb.numpy())
    assert np.array_equal(got["idx"].numpy(), idx)
    assert np.array_equal(got["counts"].numpy(), counts)
    assert np.abs(got["w"].numpy() - tw).max() <= 2e-6
    assert np.allclose(got["prob_sum"].numpy(), ps, rtol=1e-4, atol=1e-4)


def test_router_empty_batch():
    cfg = moe.config(T=0, d_model=64, n_experts=8, top_k=2, d_ff=8)
    counts = torch.full((8,), 7, dtype=torch.int32, device="cuda")
    ps = torch.full((8,), 3.0, device="cuda")
    e = torch.empty(0, device="cuda")
    ei = torch.empty(0, dtype=torch.int32, device="cuda")
    ws = moe.workspace(cfg, "router")
    moe.moe_router_topk(cfg, e, e, None, None, None, None, ei, e, counts, ps, ws)
    assert moe.moe_stream_status(ws) == 0
    assert counts.cpu().tolist() == [0] * 8 and ps.cpu().tolist() == [0.0] * 8


def test_balance_stats_match_oracle(oracle):
    T, N, k = 1000, 64, 4
    logits = synth.random_logits(T, N, seed=3, ties=False)
    cfg = moe.config(T=T, d_model=8, n_experts=N, top_k=k, d_ff=8)
    got = run_router(cfg, logits_in=logits.cuda())
    f = torch.empty(N, device="cuda")
    P = torch.empty(N, device="cuda")
    aux = torch.empty(1, device="cuda")
    moe.moe_balance_stats(N, T, k, got["counts"].cuda(), got["prob_sum"].cuda(), 0.01, f, P, aux)
    _, _, counts, ps = oracle.route(logits.numpy(), k)
    fr, Pr, auxr = oracle.balance_stats(counts, ps, T, k, 0.01)
    assert np.allclose(f.cpu().numpy(), fr, rtol=1e-6)
    assert np.allclose(P.cpu().numpy(), Pr, rtol=1e-4)
    assert abs(aux.item() - auxr) <= 1e-4 * auxr


def test_nan_scores_keep_indices_valid(oracle):
    """A NaN score ranks below every number: indices stay in range and
    distinct, and tokens without NaN route exactly as the oracle does."""
    T, N, k = 200, 64, 6
    logits = synth.random_logits(T, N, seed=9, ties=False)
    nan_rows = [3, 50, 51, 199]
    logits[3, :] = float("nan")          # a token with no number at all
    logits[50, ::2] = float("nan")
    logits[51, 5] = float("nan")
    logits[199, 60:] = float("nan")
    cfg = moe.config(T=T, d_model=8, n_experts=N, top_k=k, d_ff=8)
    got = run_router(cfg, logits_in=logits.cuda())
    idx = got["idx"].numpy()
    assert ((idx >= 0) & (idx < N)).all()
    assert all(len(set(row)) == k for row in idx.tolist())
    assert idx[3].tolist() == list(range(k))       # all -inf: lowest indices
    assert not np.isnan(logits[50, idx[50]].numpy()).any()
    ok = [t for t in range(T) if t not in nan_rows]
    ref_idx, ref_w, _, _ = oracle.route(logits.numpy()[ok], k)
    assert np.array_equal(idx[ok], ref_idx)
    assert np.abs(got["w"].numpy()[ok] - ref_w).max() <= 2e-6
    assert int(got["counts"].numpy().sum()) == T * k
