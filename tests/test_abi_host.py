"""The C ABI library loads and exports every symbol include/moe.h declares,
and its host-side checks behave as the header states. CPU only: no call here
reaches a CUDA API (every case is rejected before the first one)."""
import ctypes
import os
import re

import pytest

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.lib()


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_layer_entry_points():
    names = declared()
    for n in ("moe_router_topk", "moe_permute", "moe_grouped_swiglu", "moe_combine",
              "moe_layer_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(moe.exported_symbols()) == names


def cfg(**kw):
    base = dict(T=64, d_model=64, n_experts=4, top_k=2, d_ff=128, n_shared=0,
                dtype=moe.MOE_BF16, gate_mode=0)
    base.update(kw)
    return moe.config(**base)


@pytest.mark.parametrize("kw,rc", [
    ({}, moe.MOE_OK),
    ({"T": 0}, moe.MOE_OK),
    ({"T": -1}, moe.MOE_ERR_INVALID_ARG),
    ({"top_k": 5}, moe.MOE_ERR_INVALID_ARG),
    ({"top_k": 0}, moe.MOE_ERR_INVALID_ARG),
    ({"dtype": 7}, moe.MOE_ERR_INVALID_ARG),
    ({"gate_mode": 2}, moe.MOE_ERR_INVALID_ARG),
    ({"n_experts": 300, "top_k": 2}, moe.MOE_ERR_UNSUPPORTED),
    ({"n_experts": 16, "top_k": 9}, moe.MOE_ERR_UNSUPPORTED),
    ({"n_shared": 5}, moe.MOE_ERR_UNSUPPORTED),
    ({"d_model": 60}, moe.MOE_ERR_UNSUPPORTED),
    ({"d_ff": 100}, moe.MOE_ERR_UNSUPPORTED),
    ({"T": 1 << 28, "top_k": 4}, moe.MOE_ERR_UNSUPPORTED),
    ({"capacity": 1}, moe.MOE_OK),
    ({"capacity": -1}, moe.MOE_ERR_INVALID_ARG),
])
def test_check_config(lib, kw, rc):
    assert moe.check_config(cfg(**kw)) == rc
    assert lib.moe_check_config(None) == moe.MOE_ERR_INVALID_ARG


def test_workspace_sizes(lib):
    for kind in ("layer", "router", "permute", "grouped"):
        a = moe.workspace_size(cfg(), kind)
        b = moe.workspace_size(cfg(T=4096), kind)
        assert a > 0 and a % 256 == 0 and b >= a, kind
        assert moe.workspace_size(cfg(T=-1), kind) == 0
    # The layer workspace holds x_perm, y_perm and the hidden rows at least.
    c = cfg(T=4096, d_model=4096, n_experts=8, top_k=2, d_ff=14336)
    P = 4096 * 2
    assert moe.workspace_size(c) >= 2 * P * 4096 * 2 + P * 14336 * 2
    # backward: bf16 with d_ff a multiple of 64 only; it holds H, a | b, da | db
    assert moe.workspace_size(cfg(dtype=moe.MOE_F32), "backward") == 0
    assert moe.workspace_size(cfg(d_ff=96), "backward") == 0
    assert moe.workspace_size(c, "backward") >= 5 * P * 14336 * 2


def test_status_strings(lib):
    for rc in range(0, -8, -1):
        assert moe.status_string(rc) and moe.status_string(rc) != "unknown status"
    assert moe.status_string(-99) == "unknown status"


def _P(v):
    return ctypes.c_void_p(v)


def test_host_rejections_launch_nothing(lib):
    """Null outputs, misaligned pointers and short workspaces are refused on
    the host before any CUDA call (fake addresses are never dereferenced)."""
    c = cfg()
    before = moe.launch_count()
    A = 0x10000  # 256-byte aligned fake device address
    args = [_P(A)] * 10
    # null topk_idx
    a = list(args)
    a[6] = None
    assert lib.moe_router_topk(ctypes.byref(c), *a, _P(A), 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    # misaligned x
    a = list(args)
    a[0] = _P(A + 2)
    a[4] = None  # logits_in unset so x is needed
    a[2] = None
    assert lib.moe_router_topk(ctypes.byref(c), *a, _P(A), 1 << 20, None) == moe.MOE_ERR_MISALIGNED
    # logits_in together with logit_bias
    a = list(args)
    assert lib.moe_router_topk(ctypes.byref(c), *a, _P(A), 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    # workspace too small / misaligned
    a = list(args)
    a[2] = None
    assert lib.moe_router_topk(ctypes.byref(c), *a, _P(A), 16, None) == moe.MOE_ERR_WORKSPACE
    assert lib.moe_router_topk(ctypes.byref(c), *a, _P(A + 16), 1 << 20, None) == moe.MOE_ERR_MISALIGNED
    # permute: null outputs, bad config
    assert lib.moe_permute(ctypes.byref(c), _P(A), _P(A), None, _P(A), _P(A), _P(A), _P(A), 1 << 20,
                           None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_permute(ctypes.byref(cfg(top_k=9)), _P(A), _P(A), _P(A), _P(A), _P(A), _P(A),
                           _P(A), 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    # grouped: topk_w without sorted_pair; short workspace
    assert lib.moe_grouped_swiglu(ctypes.byref(c), _P(A), None, _P(A), None, _P(A), _P(A), _P(A),
                                  _P(A), _P(A), _P(A), 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_grouped_swiglu(ctypes.byref(c), _P(A), None, _P(A), _P(A), _P(A), _P(A), _P(A),
                                  _P(A), _P(A), _P(A), 64, None) == moe.MOE_ERR_WORKSPACE
    # shared experts need x
    assert lib.moe_grouped_swiglu(ctypes.byref(cfg(n_shared=1)), _P(A), None, _P(A), _P(A), _P(A),
                                  _P(A), _P(A), _P(A), _P(A), _P(A), 1 << 30,
                                  None) == moe.MOE_ERR_INVALID_ARG
    # combine / layer: null output
    assert lib.moe_combine(ctypes.byref(c), _P(A), _P(A), None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward(ctypes.byref(c), _P(A), _P(A), None, None, _P(A), _P(A), _P(A),
                                 None, None, None, None, None, _P(A), 1 << 30,
                                 None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward(ctypes.byref(c), _P(A), _P(A), None, None, _P(A), _P(A), _P(A),
                                 _P(A + 8), None, None, None, None, _P(A), 1 << 30,
                                 None) == moe.MOE_ERR_MISALIGNED
    # backward: fp32 and d_ff not a multiple of 64 are not built; null and
    # misaligned outputs; a short workspace
    F = ctypes.c_float
    bw = [_P(A)] * 2 + [None, None] + [_P(A)] * 4
    outs = [_P(A)] * 5
    assert lib.moe_layer_backward(ctypes.byref(cfg(dtype=moe.MOE_F32)), *bw, F(0.01), F(1.0),
                                  *outs, _P(A), 1 << 40, None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_layer_backward(ctypes.byref(cfg(d_ff=96)), *bw, F(0.01), F(1.0), *outs, _P(A),
                                  1 << 40, None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_layer_backward(ctypes.byref(c), *bw, F(0.01), F(1.0), None, *outs[1:], _P(A),
                                  1 << 40, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_backward(ctypes.byref(c), *bw, F(0.01), F(1.0), _P(A + 4), *outs[1:],
                                  _P(A), 1 << 40, None) == moe.MOE_ERR_MISALIGNED
    assert lib.moe_layer_backward(ctypes.byref(c), *bw, F(0.01), F(1.0), *outs, _P(A), 64,
                                  None) == moe.MOE_ERR_WORKSPACE
    # balance stats: bad sizes
    assert lib.moe_balance_stats(0, 4, 1, _P(A), _P(A), ctypes.c_float(0.01), _P(A), _P(A), _P(A),
                                 None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_stream_status(None, None) == moe.MOE_ERR_INVALID_ARG
    assert moe.launch_count() == before


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """The product binding has no fallback: a missing library is an error."""
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(moe, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        moe.lib()


def test_capacity_for():
    """ceil(factor * T * k / N), at least 1."""
    assert moe.capacity_for(1.25, 16384, 8, 128) == 1280
    assert moe.capacity_for(1.0, 10, 1, 3) == 4
    assert moe.capacity_for(0.01, 4, 1, 8) == 1
