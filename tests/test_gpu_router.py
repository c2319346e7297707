"""K1 parity: router scores, top-k, gate weights and statistics against the
oracle, through the C ABI.

* Given fp32 scores (parity mode, with many exact ties in scores and keys):
  indices and counts bit-exact, weights and probability sums within fp32
  rounding.
* From x and W_r (the fused router GEMM): indices bit-exact on inputs with
  a selection margin >= 1e-3; scores within fp32 accumulation error.
"""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth
from gpu_common import cfg_of, host, margin_inputs, oracle_routing

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
]


@pytest.mark.parametrize("w", GEMM_CASES, ids=lambda w: w.name)
def test_router_gemm_routes_like_the_oracle(oracle, w):
    inp = margin_inputs(w, oracle)
    cfg = cfg_of(w)
    got = run_router(cfg, inp["x"], inp["w_router"], inp["logit_bias"], inp["sel_bias"])
    r64, idx, tw, counts, ps = oracle_routing(oracle, w, inp)
    assert np.array_equal(got["idx"].numpy(), idx)
    assert np.array_equal(got["counts"].numpy(), counts)
    assert np.abs(got["logits"].numpy() - r64).max() <= 1e-4
    assert np.abs(got["w"].numpy() - tw).max() <= 1e-5
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
