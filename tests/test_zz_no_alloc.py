"""moe_router_topk_noalloc, the router entry point for callers that cannot
allocate device memory or pass a workspace (a runtime whose memory planner
assigns all device memory in advance, or a plugin slot that passes only
inputs and outputs): its scratch is a fixed array of the library's own
device memory. Checked through the C ABI on two calls in a row (the second
reuses the array the first left behind): against moe_router_topk, the
workspace entry point, and against the oracle's routing (indices and counts
bit-exact on inputs with the top-k order margin), with the array's status
word read back after each call. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth
from gpu_common import GATE_TOL, margin_inputs, oracle_routing

pytestmark = pytest.mark.gpu


def _outputs(T, N, k, dev="cuda"):
    return dict(logits=torch.full((T, N), float("nan"), device=dev),
                idx=torch.full((T, k), -1, dtype=torch.int32, device=dev),
                w=torch.full((T, k), float("nan"), device=dev),
                counts=torch.full((N,), -5, dtype=torch.int32, device=dev),
                prob_sum=torch.full((N,), float("nan"), device=dev))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(cfg, inp, o, stream):
    return moe.lib().moe_router_topk_noalloc(
        ctypes.byref(cfg), _p(inp["x"]), _p(inp["w_router"]), _p(inp["logit_bias"]),
        _p(inp["sel_bias"]), None, _p(o["logits"]), _p(o["idx"]), _p(o["w"]), _p(o["counts"]),
        _p(o["prob_sum"]), ctypes.c_void_p(stream.cuda_stream))


def _call_ws(cfg, inp, o, stream):
    ws = moe.workspace(cfg, "router")
    rc = moe.lib().moe_router_topk(
        ctypes.byref(cfg), _p(inp["x"]), _p(inp["w_router"]), _p(inp["logit_bias"]),
        _p(inp["sel_bias"]), None, _p(o["logits"]), _p(o["idx"]), _p(o["w"]), _p(o["counts"]),
        _p(o["prob_sum"]), _p(ws), ctypes.c_size_t(ws.numel()), ctypes.c_void_p(stream.cuda_stream))
    return rc


WORKLOADS = [
    synth.Workload("na_dsv3", T=2000, d_model=512, n_experts=256, top_k=8, d_ff=8, gate_mode=1,
                   sel_bias=True, seed=31),
    synth.Workload("na_mix", T=4096, d_model=1024, n_experts=8, top_k=2, d_ff=8, seed=32),
]


def test_noalloc_router_matches_workspace_router_twice(oracle):
    stream = torch.cuda.current_stream()
    for w in WORKLOADS:  # two calls in a row on the shared static scratch
        inp = margin_inputs(w, oracle)
        cfg = moe.config(T=w.T, d_model=w.d_model, n_experts=w.n_experts, top_k=w.top_k,
                         d_ff=w.d_ff, gate_mode=w.gate_mode)
        a, b = _outputs(w.T, w.n_experts, w.top_k), _outputs(w.T, w.n_experts, w.top_k)
        assert _call_noalloc(cfg, inp, a, stream) == moe.MOE_OK
        assert moe.moe_router_topk_noalloc_status(stream) == moe.MOE_OK, w.name
        assert _call_ws(cfg, inp, b, stream) == moe.MOE_OK
        torch.cuda.synchronize()
        for key in ("idx", "counts"):
            assert torch.equal(a[key], b[key]), (w.name, key)
        for key in ("logits", "w", "prob_sum"):
            assert not torch.isnan(a[key]).any()
            assert np.allclose(a[key].cpu().numpy(), b[key].cpu().numpy(), rtol=1e-6, atol=1e-6), \
                (w.name, key)
        # the oracle's routing of the same tokens: indices and counts bit-exact
        _, idx, tw, counts, ps = oracle_routing(oracle, w, inp)
        assert np.array_equal(a["idx"].cpu().numpy(), idx), w.name
        assert np.array_equal(a["counts"].cpu().numpy(), counts), w.name
        assert np.abs(a["w"].cpu().numpy() - tw).max() <= GATE_TOL, w.name
        assert np.allclose(a["prob_sum"].cpu().numpy(), ps, rtol=1e-4, atol=1e-4), w.name


def test_noalloc_router_rejects_calls_beyond_its_scratch():
    N, k = 256, 8
    T = 33 * 1024  # needs 256 + 8 * ceil(T / 64) * 256 bytes > 1 MiB
    cfg = moe.config(T=T, d_model=64, n_experts=N, top_k=k, d_ff=8)
    o = _outputs(1, N, k)
    before = moe.launch_count()
    rc = moe.lib().moe_router_topk_noalloc(
        ctypes.byref(cfg), _p(o["logits"]), _p(o["logits"]), None, None, None, None, _p(o["idx"]),
        _p(o["w"]), _p(o["counts"]), _p(o["prob_sum"]), None)
    assert rc == moe.MOE_ERR_WORKSPACE
    assert moe.launch_count() == before


@pytest.mark.parametrize("N,k,T_max", [(8, 2, 1048320), (32, 4, 262080), (256, 8, 32704)])
def test_noalloc_router_limit_is_exact(N, k, T_max):
    """The largest accepted batch matches the documented bound (256 + 8*B*N
    bytes of the 1 MiB array): T_max runs, T_max + 1 is refused unlaunched.
    Scores are given (logits_in), the path whose block count sets B."""
    stream = torch.cuda.current_stream()
    logits = torch.zeros((T_max + 1, N), device="cuda")
    o = _outputs(T_max + 1, N, k)
    for T, ok in ((T_max, True), (T_max + 1, False)):
        cfg = moe.config(T=T, d_model=64, n_experts=N, top_k=k, d_ff=8)
        before = moe.launch_count()
        rc = moe.lib().moe_router_topk_noalloc(
            ctypes.byref(cfg), None, None, None, None, _p(logits), None, _p(o["idx"]), _p(o["w"]),
            _p(o["counts"]), _p(o["prob_sum"]), ctypes.c_void_p(stream.cuda_stream))
        if ok:
            assert rc == moe.MOE_OK
            assert moe.moe_router_topk_noalloc_status(stream) == moe.MOE_OK
            assert int(o["counts"].sum().item()) == T * k
        else:
            assert rc == moe.MOE_ERR_WORKSPACE
            assert moe.launch_count() == before
