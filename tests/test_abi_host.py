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
    ({"capacity": 4, "overflow": moe.MOE_OVERFLOW_REROUTE}, moe.MOE_OK),
    ({"overflow": moe.MOE_OVERFLOW_REROUTE}, moe.MOE_OK),  # no capacity: nothing to reroute
    ({"overflow": 2}, moe.MOE_ERR_INVALID_ARG),
    ({"overflow": -1}, moe.MOE_ERR_INVALID_ARG),
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


def test_reroute_workspace_sizes(lib):
    """moe_reroute's workspace grows with the tokens and experts and is 0 for
    an invalid configuration. The layer carves the router scores and the
    reroute assignment only when it reroutes (capacity set and overflow =
    MOE_OVERFLOW_REROUTE), so its workspace is larger exactly then."""
    a = moe.workspace_size(cfg(capacity=8), "reroute")
    b = moe.workspace_size(cfg(T=4096, capacity=8), "reroute")
    c = moe.workspace_size(cfg(T=4096, n_experts=128, top_k=8, capacity=8), "reroute")
    assert a > 0 and a % 256 == 0 and b > a and c > b
    assert moe.workspace_size(cfg(overflow=3), "reroute") == 0
    drop = moe.workspace_size(cfg(T=4096, capacity=8))
    rr = moe.workspace_size(cfg(T=4096, capacity=8, overflow=moe.MOE_OVERFLOW_REROUTE))
    uncapped = moe.workspace_size(cfg(T=4096, overflow=moe.MOE_OVERFLOW_REROUTE))
    assert rr > drop and uncapped == moe.workspace_size(cfg(T=4096))


def test_reroute_host_rejections_launch_nothing(lib):
    """moe_reroute refuses null inputs or outputs, misaligned pointers, a bad
    configuration and a short or misaligned workspace on the host, before any
    CUDA call (fake addresses are never dereferenced)."""
    c = cfg(capacity=8, overflow=moe.MOE_OVERFLOW_REROUTE)
    before = moe.launch_count()
    A = 0x10000
    need = moe.workspace_size(c, "reroute")

    def call(conf=c, logits=A, sel=None, idx=A, assign=A, rounds=None, ws=A, nbytes=need):
        return lib.moe_reroute(ctypes.byref(conf), _P(logits), _P(sel), _P(idx), _P(assign),
                               _P(rounds), _P(ws), nbytes, None)

    assert call(logits=None) == moe.MOE_ERR_INVALID_ARG
    assert call(idx=None) == moe.MOE_ERR_INVALID_ARG
    assert call(assign=None) == moe.MOE_ERR_INVALID_ARG
    assert call(logits=A + 4) == moe.MOE_ERR_MISALIGNED
    assert call(sel=A + 8) == moe.MOE_ERR_MISALIGNED
    assert call(rounds=A + 2) == moe.MOE_ERR_MISALIGNED
    assert call(conf=cfg(overflow=5)) == moe.MOE_ERR_INVALID_ARG
    assert call(nbytes=need - 256) == moe.MOE_ERR_WORKSPACE
    assert call(ws=A + 16) == moe.MOE_ERR_MISALIGNED
    assert call(ws=None) == moe.MOE_ERR_INVALID_ARG
    assert moe.launch_count() == before


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


def test_quantized_layers_host_rejections(lib):
    """FP8 and NVFP4 entry points: sizes, shapes, null and misaligned
    pointers and short workspaces are refused on the host, before any CUDA
    call (fake addresses are never dereferenced)."""
    before = moe.launch_count()
    A = 0x10000
    ok = cfg(T=64, d_model=256, n_experts=4, top_k=2, d_ff=256)
    # workspace sizes: zero for what is not supported
    assert moe.workspace_size(ok, "layer_fp8") > 0
    assert moe.workspace_size(ok, "layer_nvfp4") > 0
    assert moe.workspace_size(cfg(dtype=moe.MOE_F32, d_model=256, d_ff=256), "layer_nvfp4") == 0
    assert moe.workspace_size(cfg(d_model=256, d_ff=320), "layer_nvfp4") > 0
    for d, f in ((256, 200), (200, 256), (128, 256), (256, 128)):
        assert moe.workspace_size(cfg(d_model=d, d_ff=f), "layer_nvfp4") == 0, (d, f)
    # scale stride: cols / 16 rounded up to 16 bytes
    assert [moe.moe_nvfp4_scale_stride(c) for c in (16, 256, 320, 4096, 14336, 0, -16)] == \
        [16, 16, 32, 256, 896, 0, 0]
    # quantizers
    for fn in (lib.moe_quantize_fp8,):
        assert fn(4, 12, _P(A), _P(A), _P(A), None) == moe.MOE_ERR_INVALID_ARG      # cols % 8
        assert fn(4, 16, None, _P(A), _P(A), None) == moe.MOE_ERR_INVALID_ARG
        assert fn(4, 16, _P(A + 8), _P(A), _P(A), None) == moe.MOE_ERR_MISALIGNED
        assert fn(0, 16, None, None, None, None) == moe.MOE_OK                      # nothing to do
    q4 = lib.moe_quantize_nvfp4
    assert q4(4, 24, _P(A), _P(A), _P(A), _P(A), None) == moe.MOE_ERR_INVALID_ARG   # cols % 16
    assert q4(-1, 32, _P(A), _P(A), _P(A), _P(A), None) == moe.MOE_ERR_INVALID_ARG
    assert q4(4, 32, _P(A), _P(A), None, _P(A), None) == moe.MOE_ERR_INVALID_ARG    # no scales
    assert q4(4, 32, _P(A), _P(A), _P(A + 4), _P(A), None) == moe.MOE_ERR_MISALIGNED
    assert q4(0, 32, None, None, None, None, None) == moe.MOE_OK
    # the NVFP4 layer: fp32, unsupported shapes, null weights, short workspace
    w9 = [_P(A)] * 9
    tail = [_P(A), None, None, None, None]  # y, topk_idx, topk_w, counts, prob_sum
    L = lib.moe_layer_forward_nvfp4
    assert L(ctypes.byref(cfg(dtype=moe.MOE_F32, d_model=256, d_ff=256)), _P(A), _P(A), None, None,
             *w9, *tail, _P(A), 1 << 40, None) == moe.MOE_ERR_UNSUPPORTED
    assert L(ctypes.byref(cfg(d_model=256, d_ff=192)), _P(A), _P(A), None, None, *w9, *tail,
             _P(A), 1 << 40, None) == moe.MOE_ERR_UNSUPPORTED
    bad = list(w9)
    bad[4] = None  # wu_sf
    assert L(ctypes.byref(ok), _P(A), _P(A), None, None, *bad, *tail, _P(A), 1 << 40,
             None) == moe.MOE_ERR_INVALID_ARG
    bad = list(w9)
    bad[7] = _P(A + 8)  # wd_sf
    assert L(ctypes.byref(ok), _P(A), _P(A), None, None, *bad, *tail, _P(A), 1 << 40,
             None) == moe.MOE_ERR_MISALIGNED
    assert L(ctypes.byref(ok), _P(A), _P(A), None, None, *w9, *tail, _P(A), 64,
             None) == moe.MOE_ERR_WORKSPACE
    # the FP8 layer
    w6 = [_P(A)] * 6
    F8 = lib.moe_layer_forward_fp8
    assert F8(ctypes.byref(cfg(dtype=moe.MOE_F32, d_model=256, d_ff=256)), _P(A), _P(A), None, None,
              *w6, *tail, _P(A), 1 << 40, None) == moe.MOE_ERR_UNSUPPORTED
    bad = list(w6)
    bad[1] = None
    assert F8(ctypes.byref(ok), _P(A), _P(A), None, None, *bad, *tail, _P(A), 1 << 40,
              None) == moe.MOE_ERR_INVALID_ARG
    assert F8(ctypes.byref(ok), _P(A), _P(A), None, None, *w6, *tail, _P(A), 64,
              None) == moe.MOE_ERR_WORKSPACE
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
