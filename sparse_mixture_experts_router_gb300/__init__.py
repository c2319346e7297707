"""Python binding of libmoe.so, the sparse top-k MoE FFN layer forward for
one GB300 (sm_103a).

Argument marshalling only: every function below checks nothing itself, takes
torch tensors (or None), passes their device pointers and sizes to the C ABI
of the same name (``include/moe.h``) on the current CUDA stream, and raises
:class:`MoeError` on a non-zero status. All computation runs in the library's
CUDA kernels; there is no CPU fallback. If ``libmoe.so`` has not been built,
the first call raises instead of computing anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_MISALIGNED = -3
MOE_ERR_WORKSPACE = -4
MOE_ERR_CUDA = -5
MOE_ERR_TIMEOUT = -6
MOE_ERR_DEVICE_CHECK = -7

MOE_F32, MOE_BF16 = 0, 1
MOE_GATE_TOPK_SOFTMAX, MOE_GATE_ALL_SOFTMAX_RENORM = 0, 1
MOE_TILES_AUTO, MOE_TILES_CTA, MOE_TILES_PAIR, MOE_TILES_WEIGHT_PAIR = 0, 1, 2, 3
MOE_GATHER_AUTO, MOE_GATHER_KERNEL, MOE_GATHER_FUSED = 0, 1, 2
MOE_OVERFLOW_DROP, MOE_OVERFLOW_REROUTE = 0, 1


class MoeError(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn}: status {status} ({text})")
        self.status = status


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("gate_mode", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("tiles", ctypes.c_int32),
                ("gather", ctypes.c_int32), ("overflow", ctypes.c_int32)]

    def __repr__(self):
        return "moe_config(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


def config(T, d_model, n_experts, top_k, d_ff, n_shared=0, dtype=MOE_BF16,
           gate_mode=MOE_GATE_TOPK_SOFTMAX, capacity=0, tiles=0, gather=0,
           overflow=MOE_OVERFLOW_DROP) -> moe_config:
    return moe_config(T, d_model, n_experts, top_k, n_shared, d_ff, dtype, gate_mode, capacity,
                      tiles, gather, overflow)


def capacity_for(factor: float, T: int, top_k: int, n_experts: int) -> int:
    """Expert capacity from a capacity factor: ceil(factor * T * k / N), the
    even share of the T*k pairs times the factor (at least 1)."""
    import math
    return max(1, math.ceil(factor * T * top_k / n_experts))


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_I = ctypes.c_int
_CFG = ctypes.POINTER(moe_config)
_SIGS = {
    "moe_version": (_I, []),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_cuda_error": (_I, []),
    "moe_check_config": (_I, [_CFG]),
    "moe_router_workspace_size": (_SZ, [_CFG]),
    "moe_permute_workspace_size": (_SZ, [_CFG]),
    "moe_grouped_workspace_size": (_SZ, [_CFG]),
    "moe_workspace_size": (_SZ, [_CFG]),
    "moe_router_topk": (_I, [_CFG] + [_P] * 10 + [_P, _SZ, _P]),
    "moe_router_topk_noalloc": (_I, [_CFG] + [_P] * 10 + [_P]),
    "moe_router_topk_noalloc_status": (_I, [_P]),
    "moe_permute": (_I, [_CFG] + [_P] * 6 + [_P, _SZ, _P]),
    "moe_grouped_swiglu": (_I, [_CFG] + [_P] * 9 + [_P, _SZ, _P]),
    "moe_combine": (_I, [_CFG, _P, _P, _P, _P, _P]),
    "moe_reroute_workspace_size": (_SZ, [_CFG]),
    "moe_reroute": (_I, [_CFG] + [_P] * 5 + [_P, _SZ, _P]),
    "moe_layer_forward": (_I, [_CFG] + [_P] * 12 + [_P, _SZ, _P]),
    "moe_quantize_fp8": (_I, [ctypes.c_int64, ctypes.c_int32, _P, _P, _P, _P]),
    "moe_workspace_size_fp8": (_SZ, [_CFG]),
    "moe_layer_forward_fp8": (_I, [_CFG] + [_P] * 15 + [_P, _SZ, _P]),
    "moe_nvfp4_scale_stride": (ctypes.c_int32, [ctypes.c_int32]),
    "moe_quantize_nvfp4": (_I, [ctypes.c_int64, ctypes.c_int32, _P, _P, _P, _P, _P]),
    "moe_workspace_size_nvfp4": (_SZ, [_CFG]),
    "moe_layer_forward_nvfp4": (_I, [_CFG] + [_P] * 18 + [_P, _SZ, _P]),
    "moe_balance_stats": (_I, [ctypes.c_int32] * 3 + [_P, _P, ctypes.c_float, _P, _P, _P, _P]),
    "moe_workspace_size_backward": (_SZ, [_CFG]),
    "moe_layer_backward": (_I, [_CFG] + [_P] * 8 + [ctypes.c_float, ctypes.c_float] + [_P] * 5
                           + [_P, _SZ, _P]),
    "moe_stream_status": (_I, [_P, _P]),
    "moe_set_decode_barrier_test": (None, [ctypes.c_int32, ctypes.c_uint64]),
    "moe_profile_enable": (None, [_I]),
    "moe_profile_collect": (_I, [_P, _P, _I]),
    "moe_profile_kernel_name": (ctypes.c_char_p, [_I]),
    "moe_launch_count": (ctypes.c_uint64, []),
}

_lock = threading.Lock()
_lib = None


def lib():
    """The loaded libmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` "
                    "(there is no fallback implementation)")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
            _lib = l
    return _lib


def exported_symbols():
    return list(_SIGS)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn, rc):
    if rc != MOE_OK:
        raise MoeError(fn, rc, status_string(rc))


def status_string(rc: int) -> str:
    return lib().moe_status_string(rc).decode()


def check_config(cfg: moe_config) -> int:
    return lib().moe_check_config(ctypes.byref(cfg))


def workspace_size(cfg: moe_config, kind: str = "layer") -> int:
    fn = {"layer": "moe_workspace_size", "router": "moe_router_workspace_size",
          "permute": "moe_permute_workspace_size", "grouped": "moe_grouped_workspace_size",
          "layer_fp8": "moe_workspace_size_fp8", "layer_nvfp4": "moe_workspace_size_nvfp4",
          "backward": "moe_workspace_size_backward", "reroute": "moe_reroute_workspace_size"}[kind]
    return int(getattr(lib(), fn)(ctypes.byref(cfg)))


def workspace(cfg: moe_config, kind: str = "layer", device="cuda"):
    """A caller-owned workspace tensor of the size the library asks for."""
    import torch
    n = workspace_size(cfg, kind)
    if n == 0:
        raise MoeError("workspace_size", check_config(cfg), "invalid configuration")
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_router_topk(cfg, x, w_router, logit_bias, sel_bias, logits_in, logits_out, topk_idx,
                    topk_w, counts, prob_sum, ws, stream=None):
    _check("moe_router_topk", lib().moe_router_topk(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(sel_bias),
        _ptr(logits_in), _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
        _ptr(prob_sum), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def moe_router_topk_noalloc(cfg, x, w_router, logit_bias, sel_bias, logits_in, logits_out,
                            topk_idx, topk_w, counts, prob_sum, stream=None):
    _check("moe_router_topk_noalloc", lib().moe_router_topk_noalloc(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(sel_bias),
        _ptr(logits_in), _ptr(logits_out), _ptr(topk_idx), _ptr(topk_w), _ptr(counts),
        _ptr(prob_sum), _stream(stream)))


def moe_router_topk_noalloc_status(stream=None):
    """Synchronises the stream and returns the device-side status of the last
    moe_router_topk_noalloc call (0, or a negative MOE_ERR_* code)."""
    return lib().moe_router_topk_noalloc_status(_stream(stream))


def moe_reroute(cfg, logits, sel_bias, topk_idx, assign, rounds, ws, stream=None):
    _check("moe_reroute", lib().moe_reroute(
        ctypes.byref(cfg), _ptr(logits), _ptr(sel_bias), _ptr(topk_idx), _ptr(assign),
        _ptr(rounds), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def moe_permute(cfg, x, topk_idx, expert_offsets, sorted_pair, inv_pos, x_perm, ws, stream=None):
    _check("moe_permute", lib().moe_permute(
        ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(expert_offsets), _ptr(sorted_pair),
        _ptr(inv_pos), _ptr(x_perm), _ptr(ws), ws.numel() if ws is not None else 0,
        _stream(stream)))


def moe_grouped_swiglu(cfg, x_perm, x, expert_offsets, sorted_pair, topk_w, w_gate, w_up, w_down,
                       y_perm, ws, stream=None):
    _check("moe_grouped_swiglu", lib().moe_grouped_swiglu(
        ctypes.byref(cfg), _ptr(x_perm), _ptr(x), _ptr(expert_offsets), _ptr(sorted_pair),
        _ptr(topk_w), _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(y_perm), _ptr(ws),
        ws.numel() if ws is not None else 0, _stream(stream)))


def moe_combine(cfg, y_perm, inv_pos, topk_w, y, stream=None):
    _check("moe_combine", lib().moe_combine(
        ctypes.byref(cfg), _ptr(y_perm), _ptr(inv_pos), _ptr(topk_w), _ptr(y), _stream(stream)))


def moe_quantize_fp8(src, q, scale, stream=None):
    """Row-wise E4M3 codes and fp32 scales of a [rows, cols] bf16 tensor."""
    rows, cols = src.shape[0], src.numel() // max(1, src.shape[0])
    _check("moe_quantize_fp8", lib().moe_quantize_fp8(rows, cols, _ptr(src), _ptr(q), _ptr(scale),
                                                      _stream(stream)))


def moe_layer_forward_fp8(cfg, x, w_router, logit_bias, sel_bias, wg_q, wg_scale, wu_q, wu_scale,
                          wd_q, wd_scale, y, topk_idx, topk_w, counts, prob_sum, ws, stream=None):
    _check("moe_layer_forward_fp8", lib().moe_layer_forward_fp8(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(sel_bias),
        _ptr(wg_q), _ptr(wg_scale), _ptr(wu_q), _ptr(wu_scale), _ptr(wd_q), _ptr(wd_scale),
        _ptr(y), _ptr(topk_idx), _ptr(topk_w), _ptr(counts), _ptr(prob_sum), _ptr(ws),
        ws.numel() if ws is not None else 0, _stream(stream)))


def moe_nvfp4_scale_stride(cols):
    """Bytes of one row of NVFP4 block scales for rows of `cols` elements."""
    return int(lib().moe_nvfp4_scale_stride(int(cols)))


def moe_quantize_nvfp4(src, q, sf, scale, stream=None):
    """Row-wise NVFP4 of a [rows, cols] bf16 tensor: packed E2M1 codes
    [rows, cols/2], E4M3 block scales [rows, moe_nvfp4_scale_stride(cols)] and
    fp32 row scales [rows]."""
    rows, cols = src.shape[0], src.numel() // max(1, src.shape[0])
    _check("moe_quantize_nvfp4", lib().moe_quantize_nvfp4(rows, cols, _ptr(src), _ptr(q), _ptr(sf),
                                                          _ptr(scale), _stream(stream)))


def moe_layer_forward_nvfp4(cfg, x, w_router, logit_bias, sel_bias, wg_q, wg_sf, wg_scale, wu_q,
                            wu_sf, wu_scale, wd_q, wd_sf, wd_scale, y, topk_idx, topk_w, counts,
                            prob_sum, ws, stream=None):
    _check("moe_layer_forward_nvfp4", lib().moe_layer_forward_nvfp4(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(sel_bias),
        _ptr(wg_q), _ptr(wg_sf), _ptr(wg_scale), _ptr(wu_q), _ptr(wu_sf), _ptr(wu_scale),
        _ptr(wd_q), _ptr(wd_sf), _ptr(wd_scale), _ptr(y), _ptr(topk_idx), _ptr(topk_w),
        _ptr(counts), _ptr(prob_sum), _ptr(ws), ws.numel() if ws is not None else 0,
        _stream(stream)))


def moe_layer_forward(cfg, x, w_router, logit_bias, sel_bias, w_gate, w_up, w_down, y, topk_idx,
                      topk_w, counts, prob_sum, ws, stream=None):
    _check("moe_layer_forward", lib().moe_layer_forward(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(sel_bias),
        _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(y), _ptr(topk_idx), _ptr(topk_w),
        _ptr(counts), _ptr(prob_sum), _ptr(ws), ws.numel() if ws is not None else 0,
        _stream(stream)))


def moe_layer_backward(cfg, x, w_router, logit_bias, sel_bias, w_gate, w_up, w_down, dy, alpha,
                       aux_grad, dx, dw_router, dw_gate, dw_up, dw_down, ws, stream=None):
    _check("moe_layer_backward", lib().moe_layer_backward(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(logit_bias), _ptr(sel_bias),
        _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(dy), ctypes.c_float(alpha),
        ctypes.c_float(aux_grad), _ptr(dx), _ptr(dw_router), _ptr(dw_gate), _ptr(dw_up),
        _ptr(dw_down), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def moe_balance_stats(n_experts, T, top_k, counts, prob_sum, alpha, f, P, aux, stream=None):
    _check("moe_balance_stats", lib().moe_balance_stats(
        n_experts, T, top_k, _ptr(counts), _ptr(prob_sum), ctypes.c_float(alpha), _ptr(f), _ptr(P),
        _ptr(aux), _stream(stream)))


def moe_stream_status(ws, stream=None) -> int:
    return int(lib().moe_stream_status(_ptr(ws), _stream(stream)))


def moe_set_decode_barrier_test(withhold: int, limit_ns: int) -> None:
    lib().moe_set_decode_barrier_test(int(withhold), int(limit_ns))


def profile_kernel_names() -> list:
    out = []
    for i in range(32):
        name = lib().moe_profile_kernel_name(i).decode()
        if not name:
            break
        out.append(name)
    return out


def profile_enable(on: bool = True, kernels=None):
    """Bracket launches with CUDA events: every kernel kind, or only those
    named in ``kernels`` (names as in profile_collect)."""
    if not on:
        mask = 0
    elif kernels is None:
        mask = -1
    else:
        names = profile_kernel_names()
        mask = 0
        for k in kernels:
            mask |= 1 << names.index(k)
    lib().moe_profile_enable(mask)


def profile_collect() -> dict:
    """{kernel name: (total ms, launches)} of the launches since the last
    collect while profiling was on (synchronises on the last event)."""
    n = 32
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int32 * n)()
    k = lib().moe_profile_collect(ms, cnt, n)
    out = {}
    for i in range(k):
        name = lib().moe_profile_kernel_name(i).decode()
        if cnt[i]:
            out[name] = (float(ms[i]), int(cnt[i]))
    return out


def launch_count() -> int:
    return int(lib().moe_launch_count())


def version() -> int:
    return int(lib().moe_version())
