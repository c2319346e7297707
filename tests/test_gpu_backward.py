"""The layer backward (moe_layer_backward) against the oracle's gradient.

The loss is sum(dy * y) + aux_grad * aux with the routing held fixed; the
oracle differentiates its own forward in fp64 (pinned by finite
differences and autograd on the CPU).

* Reduced-size layers of each family (shared experts, both gate modes,
  capacity cuts, the tensor-core router, a single token, experts that take
  no token, dimensions that are not multiples of the tiles): every gradient
  in full against the oracle's, max |g - g_ref| / max |g_ref| <= 2e-2 per
  tensor (bf16 intermediates: H, the pre-activations, dO, da | db, dA;
  fp32 sums). Experts that took no token have exactly zero gradients.
* dy = 0: only the balance term; dx and dW_r against the oracle's balance
  gradient, the expert gradients exactly zero.
* Two calls give the same bits.
* Full-size Mixtral-8x7B and DeepSeek-V3 layers: dx rows of sampled tokens,
  rows of dW_g and dW_u and columns of dW_d of sampled experts against the
  oracle's sampled gradient; dW_r and dx with dy = 0 against the oracle's
  balance gradient over all tokens.
"""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth
from gpu_common import BF16_TOL, capacity_of, cfg_of, host, margin_inputs, rel_inf, sample_rows

pytestmark = pytest.mark.gpu

ALPHA = 0.01

SMALL = [
    synth.Workload("bwd_mix_small", T=256, d_model=256, n_experts=8, top_k=2, d_ff=512, seed=41),
    synth.Workload("bwd_shared_renorm_capacity", T=200, d_model=128, n_experts=6, top_k=3,
                   d_ff=192, n_shared=1, gate_mode=1, sel_bias=True, capacity_factor=0.75,
                   seed=42),
    synth.Workload("bwd_tc_router", T=160, d_model=256, n_experts=64, top_k=4, d_ff=128, seed=43),
    synth.Workload("bwd_single_token", T=1, d_model=128, n_experts=8, top_k=2, d_ff=128, seed=44),
    synth.Workload("bwd_empty_experts", T=8, d_model=128, n_experts=32, top_k=1, d_ff=128,
                   seed=45),
    synth.Workload("bwd_zipf", T=512, d_model=256, n_experts=32, top_k=4, d_ff=256, zipf_s=1.2,
                   seed=46),
    synth.Workload("bwd_ragged_dims", T=77, d_model=200, n_experts=4, top_k=2, d_ff=320,
                   n_shared=2, seed=47),
    synth.Workload("bwd_zipf_reroute", T=300, d_model=128, n_experts=8, top_k=2, d_ff=192,
                   zipf_s=1.2, capacity_factor=1.0, overflow=1, seed=48),
]


def f64(t):
    """Exact fp64 copy of a bf16 / fp32 device tensor."""
    return t.double().cpu().numpy()


class BwdRun:
    def __init__(self, w, inp, dy, aux_grad=1.0):
        self.cfg = cfg_of(w)
        E = w.n_experts + w.n_shared
        dev = inp["x"].device
        nan = float("nan")
        self.dx = torch.full((w.T, w.d_model), nan, device=dev)
        self.dwr = torch.full((w.n_experts, w.d_model), nan, device=dev)
        self.dwg = torch.full((E, w.d_ff, w.d_model), nan, device=dev)
        self.dwu = torch.full((E, w.d_ff, w.d_model), nan, device=dev)
        self.dwd = torch.full((E, w.d_model, w.d_ff), nan, device=dev)
        self.ws = moe.workspace(self.cfg, "backward", dev)
        self.inp, self.dy, self.aux_grad = inp, dy, aux_grad

    def __call__(self):
        i = self.inp
        moe.moe_layer_backward(self.cfg, i["x"], i["w_router"], i["logit_bias"], i["sel_bias"],
                               i["w_gate"], i["w_up"], i["w_down"], self.dy, ALPHA,
                               self.aux_grad, self.dx, self.dwr, self.dwg, self.dwu, self.dwd,
                               self.ws)
        assert moe.moe_stream_status(self.ws) == 0
        return self


def oracle_full(oracle, w, inp, dy, aux_grad):
    lb = None if inp["logit_bias"] is None else f64(inp["logit_bias"])
    return oracle.layer_backward(host(inp["x"]), host(inp["w_router"]), host(inp["w_gate"]),
                                 host(inp["w_up"]), host(inp["w_down"]), w.top_k, f64(dy),
                                 gate_mode=w.gate_mode, logit_bias=lb,
                                 sel_bias=host(inp["sel_bias"]), n_shared=w.n_shared,
                                 capacity=capacity_of(w), alpha=ALPHA, aux_grad=aux_grad,
                                 reroute=bool(w.overflow))


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_backward_small(oracle, w):
    inp = margin_inputs(w, oracle, all_keys=bool(w.overflow))
    dy = synth.make_grad_output(w)
    aux_grad = 10.0
    run = BwdRun(w, inp, dy, aux_grad)()
    ref = oracle_full(oracle, w, inp, dy, aux_grad)
    got = dict(dx=run.dx, dw_router=run.dwr, dw_gate=run.dwg, dw_up=run.dwu, dw_down=run.dwd)
    for key, t in got.items():
        g = t.cpu().numpy()
        assert not np.isnan(g).any(), key
        err = rel_inf(g, ref[key])
        assert err <= BF16_TOL, (key, err)
    # experts that took no token: exactly zero, as the oracle's
    for key in ("dw_gate", "dw_up", "dw_down"):
        idle = [e for e in range(ref[key].shape[0]) if not ref[key][e].any()]
        for e in idle:
            assert not got[key][e].any().item(), (key, e)
    if w.name == "bwd_empty_experts":
        assert idle, "the case is meant to leave experts without tokens"


def test_backward_balance_term_alone(oracle):
    w = SMALL[2]
    inp = margin_inputs(w, oracle)
    dy = torch.zeros(w.T, w.d_model, dtype=torch.bfloat16, device="cuda")
    run = BwdRun(w, inp, dy, aux_grad=100.0)()
    dx, dwr = oracle.balance_backward(host(inp["x"]), host(inp["w_router"]), w.top_k,
                                      gate_mode=w.gate_mode, alpha=ALPHA, aux_grad=100.0)
    assert rel_inf(run.dx.cpu().numpy(), dx) <= BF16_TOL
    assert rel_inf(run.dwr.cpu().numpy(), dwr) <= BF16_TOL
    for t in (run.dwg, run.dwu, run.dwd):
        assert not t.any().item()


def test_backward_is_deterministic(oracle):
    w = SMALL[1]
    inp = margin_inputs(w, oracle)
    dy = synth.make_grad_output(w)
    run = BwdRun(w, inp, dy)()
    first = [t.clone() for t in (run.dx, run.dwr, run.dwg, run.dwu, run.dwd)]
    run()
    for a, b in zip(first, (run.dx, run.dwr, run.dwg, run.dwu, run.dwd)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


FULL = [synth.MIXTRAL_PREFILL, synth.DEEPSEEK_V3]


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_backward_full_size_sampled(oracle, w):
    inp = margin_inputs(w, oracle)
    dy = synth.make_grad_output(w)
    run = BwdRun(w, inp, dy)()
    N, S = w.n_experts, w.n_shared
    lb = None if inp["logit_bias"] is None else f64(inp["logit_bias"])
    xh, wrh, sbh = host(inp["x"]), host(inp["w_router"]), host(inp["sel_bias"])
    # routing decides which experts the sampled tokens need
    _, r32 = oracle.router_logits(xh, wrh, lb)
    idx, _, counts, _ = oracle.route(r32, w.top_k, w.gate_mode, sbh)
    toks = sample_rows(w.T, 3, seed=5)
    busiest = int(np.argmax(counts))
    col_experts = sorted({0, busiest, N - 1} | ({N} if S else set()))
    cols = [(e, j) for e in col_experts for j in (0, w.d_ff // 2 + 3, w.d_ff - 1)]
    need = set(idx[toks].ravel().tolist()) | set(range(N, N + S)) | set(col_experts)
    experts = {e: (host(inp["w_gate"][e]), host(inp["w_up"][e]), host(inp["w_down"][e]))
               for e in sorted(need)}
    ref = oracle.backward_samples(xh, wrh, experts, N, w.top_k, f64(dy), tokens=toks,
                                  columns=cols, gate_mode=w.gate_mode, logit_bias=lb,
                                  sel_bias=sbh, n_shared=S, capacity=capacity_of(w), alpha=ALPHA,
                                  aux_grad=1.0)
    assert rel_inf(run.dx[toks].cpu().numpy(), ref["dx_rows"]) <= BF16_TOL
    e_idx = torch.tensor([e for e, _ in cols], device="cuda")
    j_idx = torch.tensor([j for _, j in cols], device="cuda")
    assert rel_inf(run.dwg[e_idx, j_idx].cpu().numpy(), ref["dw_gate_rows"]) <= BF16_TOL
    assert rel_inf(run.dwu[e_idx, j_idx].cpu().numpy(), ref["dw_up_rows"]) <= BF16_TOL
    assert rel_inf(run.dwd[e_idx, :, j_idx].cpu().numpy(), ref["dw_down_cols"]) <= BF16_TOL
    # the balance term over every token: dy = 0
    run.dy = torch.zeros_like(dy)
    run()
    dx, dwr = oracle.balance_backward(xh, wrh, w.top_k, gate_mode=w.gate_mode, logit_bias=lb,
                                      sel_bias=sbh, alpha=ALPHA, aux_grad=1.0)
    assert rel_inf(run.dx.cpu().numpy(), dx) <= BF16_TOL
    assert rel_inf(run.dwr.cpu().numpy(), dwr) <= BF16_TOL
