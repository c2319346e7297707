"""CPU fp64 oracle for the sparse top-k MoE FFN layer forward.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product library
(``sparse_mixture_experts_router_gb300``) never imports it and shares no code
with it.

This module is argument marshalling around ``moe_oracle.c`` (numpy arrays in,
numpy arrays out); all arithmetic lives in the C file, which states the
definition it follows for every function, citing the pages by title and
section. Stored bf16 inputs are passed as their uint16 bit patterns and are
widened exactly inside the C code.

Parity unpinned: the SwiGLU expert at realistic sizes (no printed value on the
pages; pinned only by reduction to library routines and by brute force on
tiny inputs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2
GATE_TOPK_SOFTMAX, GATE_ALL_SOFTMAX_RENORM = 0, 1

_P = ctypes.c_void_p
_I = ctypes.c_int


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle C file into a shared library (gcc, OpenMP, -O2,
    strict IEEE arithmetic: no fast-math, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    lib.oracle_num_threads.restype = _I
    lib.oracle_softmax.argtypes = [_I, _P, _P]
    lib.oracle_topk.argtypes = [_I, _I, _P, _P]
    lib.oracle_gates.argtypes = [_I, _I, _I, _P, _P, _P]
    lib.oracle_router_logits.argtypes = [_I, _I, _I, _I, _P, _I, _P, _P, _P, _P]
    lib.oracle_route.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P]
    lib.oracle_capacity_keep.argtypes = [_I, _I, _I, _P, _I, _P]
    lib.oracle_permute.argtypes = [_I, _I, _I, _P, _I, _P, _P, _P]
    lib.oracle_reroute.restype = _I
    lib.oracle_reroute.argtypes = [_I, _I, _I, _P, _P, _P, _I, _P]
    lib.oracle_expert_swiglu.argtypes = [_I, _I, _I, _P, _P, _P, _P, _P]
    lib.oracle_gated_sum.argtypes = [_I, _I, _P, _P, _P]
    lib.oracle_layer_rows.restype = _I
    lib.oracle_layer_rows.argtypes = [_I, _I, _I, _I, _I, _I, _I, _P, _I,
                                      _P, _P, _P, _P, _P, _P, _I, _I, _P, _P]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode_scan.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode_scan.argtypes = [ctypes.c_float]
    lib.oracle_quantize_rows_e4m3.argtypes = [_I, _I, _I, _P, _P, _P]
    lib.oracle_e2m1_decode.restype = ctypes.c_double
    lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_encode.restype = ctypes.c_uint8
    lib.oracle_e2m1_encode.argtypes = [ctypes.c_float]
    lib.oracle_e2m1_encode_scan.restype = ctypes.c_uint8
    lib.oracle_e2m1_encode_scan.argtypes = [ctypes.c_float]
    lib.oracle_quantize_rows_nvfp4.argtypes = [_I, _I, _I, _P, _P, _P, _P]
    lib.oracle_balance_loss.restype = ctypes.c_double
    lib.oracle_balance_loss.argtypes = [_I, _P, _P, ctypes.c_double]
    lib.oracle_balance_stats.restype = ctypes.c_double
    lib.oracle_balance_stats.argtypes = [_I, _I, _I, _P, _P, ctypes.c_double,
                                         _P, _P]
    lib.oracle_selection_margin.argtypes = [_I, _I, _I, _P, _P, _P]
    lib.oracle_order_margin.argtypes = [_I, _I, _I, _P, _P, _P]
    _D = ctypes.c_double
    lib.oracle_layer_backward.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P,
                                          _P, _P, _P, _P, _P, _D, _D, _P, _P, _P, _P, _P]
    lib.oracle_layer_backward.restype = None
    lib.oracle_backward_samples.argtypes = [_I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _I, _P, _P,
                                            _P, _P, _P, _P, _P, _D, _D, _I, _P, _P, _I, _P, _P,
                                            _P, _P, _P]
    lib.oracle_backward_samples.restype = _I
    lib.oracle_balance_backward.argtypes = [_I, _I, _I, _I, _I, _I, _P, _I, _P, _P, _P, _D, _D,
                                            _P, _P]
    lib.oracle_balance_backward.restype = None
    return lib


def load(path: str | None = None):
    """Load (compiling first if needed) the oracle library. ``path`` loads a
    specific build instead (used by the planted-mistake tests)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                compile_oracle()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


def _stored(a):
    """(dtype code, contiguous array) of a stored input: float32, float64, or
    uint16 holding bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return F32, a
    if a.dtype == np.float64:
        return F64, a
    if a.dtype == np.uint16:
        return BF16, a
    raise TypeError(f"oracle inputs are float32, float64 or bf16 bits (uint16), got {a.dtype}")


class Oracle:
    """Thin marshalling layer over one loaded oracle library."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def softmax(self, r):
        r = _c(r, np.float64)
        p = np.empty_like(r)
        self.lib.oracle_softmax(r.size, _ptr(r), _ptr(p))
        return p

    def topk(self, key, k):
        key = _c(key, np.float32)
        idx = np.empty(k, np.int32)
        self.lib.oracle_topk(key.size, k, _ptr(key), _ptr(idx))
        return idx

    def gates(self, r, idx, mode=GATE_TOPK_SOFTMAX):
        r = _c(r, np.float64)
        idx = _c(idx, np.int32)
        g = np.empty(idx.size, np.float64)
        self.lib.oracle_gates(r.size, idx.size, mode, _ptr(r), _ptr(idx), _ptr(g))
        return g

    def router_logits(self, x, w_router, logit_bias=None):
        """(r64 [T,N] fp64, r32 [T,N] fp32)."""
        xd, x = _stored(x)
        wd, w = _stored(w_router)
        T, d = x.shape
        N = w.shape[0]
        assert w.shape[1] == d
        lb = None if logit_bias is None else _c(logit_bias, np.float64)
        r64 = np.empty((T, N), np.float64)
        r32 = np.empty((T, N), np.float32)
        self.lib.oracle_router_logits(T, d, N, xd, _ptr(x), wd, _ptr(w), _ptr(lb),
                                      _ptr(r64), _ptr(r32))
        return r64, r32

    def route(self, r32, k, gate_mode=GATE_TOPK_SOFTMAX, sel_bias=None):
        """(topk_idx [T,k] int32, topk_w [T,k] fp64, counts [N] int32,
        prob_sum [N] fp64) from fp32 router scores."""
        r32 = _c(r32, np.float32)
        T, N = r32.shape
        sb = None if sel_bias is None else _c(sel_bias, np.float32)
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float64)
        counts = np.empty(N, np.int32)
        prob_sum = np.empty(N, np.float64)
        self.lib.oracle_route(T, N, k, gate_mode, _ptr(r32), _ptr(sb), _ptr(idx),
                              _ptr(w), _ptr(counts), _ptr(prob_sum))
        return idx, w, counts, prob_sum

    def capacity_keep(self, topk_idx, N, capacity):
        """keep [T*k] uint8: 1 for a pair its expert keeps under the capacity."""
        topk_idx = _c(topk_idx, np.int32)
        T, k = topk_idx.shape
        keep = np.empty(T * k, np.uint8)
        self.lib.oracle_capacity_keep(T, k, N, _ptr(topk_idx), int(capacity), _ptr(keep))
        return keep

    def permute(self, topk_idx, N, capacity=0):
        """(offsets [N+1], sorted_pair [rows], inv_pos [T*k]) int32; rows =
        offsets[N] kept pairs, inv_pos -1 for a dropped pair."""
        topk_idx = _c(topk_idx, np.int32)
        T, k = topk_idx.shape
        offsets = np.empty(N + 1, np.int32)
        sp = np.empty(T * k, np.int32)
        inv = np.empty(T * k, np.int32)
        self.lib.oracle_permute(T, k, N, _ptr(topk_idx), int(capacity), _ptr(offsets), _ptr(sp),
                                _ptr(inv))
        return offsets, sp[:offsets[N]], inv

    def reroute(self, r32, topk_idx, capacity, sel_bias=None):
        """(assign [T,k] int32, rounds): the expert each pair runs on when
        capacity overflow is rerouted in rounds (-1: dropped), and the number
        of rounds after the capacity cut."""
        r32 = _c(r32, np.float32)
        topk_idx = _c(topk_idx, np.int32)
        T, N = r32.shape
        k = topk_idx.shape[1]
        sb = None if sel_bias is None else _c(sel_bias, np.float32)
        assign = np.empty((T, k), np.int32)
        rounds = self.lib.oracle_reroute(T, k, N, _ptr(r32), _ptr(sb), _ptr(topk_idx),
                                         int(capacity), _ptr(assign))
        return assign, int(rounds)

    def expert_swiglu(self, x_row, wg, wu, wd):
        wdt, wg = _stored(wg)
        wdt2, wu = _stored(wu)
        wdt3, wd = _stored(wd)
        assert wdt == wdt2 == wdt3
        d_ff, d = wg.shape
        x_row = _c(x_row, np.float64)
        out = np.empty(d, np.float64)
        self.lib.oracle_expert_swiglu(d, d_ff, wdt, _ptr(wg), _ptr(wu), _ptr(wd),
                                      _ptr(x_row), _ptr(out))
        return out

    def gated_sum(self, G, E):
        G = _c(G, np.float64)
        E = _c(E, np.float64).reshape(G.size, -1)
        y = np.empty(E.shape[1], np.float64)
        self.lib.oracle_gated_sum(G.size, E.shape[1], _ptr(G), _ptr(E), _ptr(y))
        return y

    def e4m3_decode(self, code):
        return float(self.lib.oracle_e4m3_decode(int(code)))

    def e4m3_encode(self, v, scan=False):
        f = self.lib.oracle_e4m3_encode_scan if scan else self.lib.oracle_e4m3_encode
        return int(f(float(v)))

    def quantize_rows_e4m3(self, m):
        """(codes [rows, cols] uint8, scales [rows] fp32) of a stored matrix:
        one scale fp32(amax/448) per row, codes E4M3(fp32(v/scale))."""
        dt, m = _stored(m)
        rows, cols = m.shape
        q = np.empty((rows, cols), np.uint8)
        sc = np.empty(rows, np.float32)
        self.lib.oracle_quantize_rows_e4m3(rows, cols, dt, _ptr(m), _ptr(q), _ptr(sc))
        return q, sc

    def e2m1_decode(self, code):
        return float(self.lib.oracle_e2m1_decode(int(code)))

    def e2m1_encode(self, v, scan=False):
        f = self.lib.oracle_e2m1_encode_scan if scan else self.lib.oracle_e2m1_encode
        return int(f(float(v)))

    def quantize_rows_nvfp4(self, m):
        """(codes [rows, cols] uint8 (one E2M1 code per element), block scale
        codes [rows, cols/16] uint8 (E4M3), row scales [rows] fp32) of a
        stored matrix whose column count is a multiple of 16."""
        dt, m = _stored(m)
        rows, cols = m.shape
        assert cols % 16 == 0
        q = np.empty((rows, cols), np.uint8)
        bs = np.empty((rows, cols // 16), np.uint8)
        sc = np.empty(rows, np.float32)
        self.lib.oracle_quantize_rows_nvfp4(rows, cols, dt, _ptr(m), _ptr(q), _ptr(bs), _ptr(sc))
        return q, bs, sc

    def nvfp4_values(self, q, bs, sc):
        """fp64 values of an NVFP4 matrix (codes, block scales, row scales)."""
        e2 = np.array([self.e2m1_decode(c) for c in range(16)])
        e4 = np.array([self.e4m3_decode(c) for c in range(256)])
        return e2[q] * np.repeat(e4[bs], 16, axis=1) * sc.astype(np.float64)[:, None]

    def layer_rows(self, x, experts, topk_idx, topk_w, rows, N, n_shared=0, keep=None,
                   fp8=False, nvfp4=False):
        """y [len(rows), d] fp64 for the listed tokens. ``experts`` maps an
        expert index (0..N+n_shared-1; shared ones last) to its (wg, wu, wd)
        stored arrays; experts no listed token uses may be absent. ``keep``
        ([T*k] uint8, from capacity_keep) marks the pairs that run; a dropped
        pair adds nothing. ``fp8`` evaluates the experts in E4M3 with row
        scales (tokens, weight output channels and H rows quantized);
        ``nvfp4`` in NVFP4 (E2M1 codes, E4M3 scales of 16-element blocks and
        fp32 row scales, the same rows quantized)."""
        assert not (fp8 and nvfp4)
        xd, x = _stored(x)
        T, d = x.shape
        topk_idx = _c(topk_idx, np.int32)
        topk_w = _c(topk_w, np.float64)
        k = topk_idx.shape[1]
        rows = _c(rows, np.int32)
        E = N + n_shared
        refs = []  # the stored arrays, alive until the call returns
        tabs = [(_P * E)(), (_P * E)(), (_P * E)()]
        wdt = None
        d_ff = None
        for e, mats in experts.items():
            for j, m in enumerate(mats):
                dt, m = _stored(m)
                wdt = dt if wdt is None else wdt
                assert dt == wdt
                refs.append(m)
                tabs[j][e] = m.ctypes.data
            d_ff = mats[0].shape[0]
        y = np.empty((rows.size, d), np.float64)
        keep = None if keep is None else _c(keep, np.uint8)
        rc = self.lib.oracle_layer_rows(T, d, d_ff, N, k, n_shared, xd, _ptr(x), wdt,
                                        tabs[0], tabs[1], tabs[2], _ptr(topk_idx),
                                        _ptr(topk_w), _ptr(keep), 2 if nvfp4 else int(bool(fp8)), rows.size,
                                        _ptr(rows), _ptr(y))
        if rc != 0:
            raise ValueError("oracle_layer_rows: a token needs an expert that was not supplied")
        return y

    def selection_margin(self, r64, k, sel_bias=None):
        """Per-token gap between the k-th and (k+1)-th largest fp64 key."""
        r64 = _c(r64, np.float64)
        T, N = r64.shape
        sb = None if sel_bias is None else _c(sel_bias, np.float32)
        m = np.empty(T, np.float64)
        self.lib.oracle_selection_margin(T, N, k, _ptr(r64), _ptr(sb), _ptr(m))
        return m

    def order_margin(self, r64, k, sel_bias=None):
        """Per-token smallest gap between neighbours among the k+1 largest
        fp64 keys (all N keys when k = N)."""
        r64 = _c(r64, np.float64)
        T, N = r64.shape
        sb = None if sel_bias is None else _c(sel_bias, np.float32)
        m = np.empty(T, np.float64)
        self.lib.oracle_order_margin(T, N, k, _ptr(r64), _ptr(sb), _ptr(m))
        return m

    def balance_loss(self, f, P, alpha=0.01):
        f = _c(f, np.float64)
        P = _c(P, np.float64)
        return float(self.lib.oracle_balance_loss(f.size, _ptr(f), _ptr(P), alpha))

    def balance_stats(self, counts, prob_sum, T, k, alpha=0.01):
        """(f, P, aux)."""
        counts = _c(counts, np.int32)
        prob_sum = _c(prob_sum, np.float64)
        N = counts.size
        f = np.empty(N, np.float64)
        P = np.empty(N, np.float64)
        aux = self.lib.oracle_balance_stats(N, T, k, _ptr(counts), _ptr(prob_sum),
                                            alpha, _ptr(f), _ptr(P))
        return f, P, float(aux)

    # ---- composition: the full layer for a token subset ---------------------
    def layer(self, x, w_router, wg, wu, wd, k, gate_mode=GATE_TOPK_SOFTMAX,
              logit_bias=None, sel_bias=None, n_shared=0, rows=None, capacity=0, fp8=False,
              nvfp4=False, reroute=False):
        """Full forward: router scores for all tokens, routing for all tokens,
        expert outputs for ``rows`` (all tokens when None), with an expert
        capacity (0 = none) whose overflow is dropped, or rerouted
        (``reroute``, see ``reroute``). wg/wu/wd are the stacked
        [N+n_shared, ...] stored arrays (or dicts expert -> array). Returns a
        dict with r32, topk_idx, topk_w, counts, prob_sum, keep, assign (the
        expert each pair runs on, -1 if dropped), rounds, y."""
        _, r32 = self.router_logits(x, w_router, logit_bias)
        idx, w, counts, prob_sum = self.route(r32, k, gate_mode, sel_bias)
        N = r32.shape[1]
        T = r32.shape[0]
        if reroute:
            assign, rounds = self.reroute(r32, idx, capacity, sel_bias)
            keep = (assign.ravel() >= 0).astype(np.uint8)
        else:
            keep = self.capacity_keep(idx, N, capacity)
            assign = np.where(keep.reshape(idx.shape) != 0, idx, -1).astype(np.int32)
            rounds = 0
        if rows is None:
            rows = np.arange(T, dtype=np.int32)
        rows = np.asarray(rows, np.int32)
        run = np.where(assign >= 0, assign, idx).astype(np.int32)  # dropped: keep says so
        need = sorted(set(run[rows].ravel().tolist()) | set(range(N, N + n_shared)))
        experts = {e: (wg[e], wu[e], wd[e]) for e in need}
        y = self.layer_rows(x, experts, run, w, rows, N, n_shared, keep, fp8, nvfp4)
        return dict(r32=r32, topk_idx=idx, topk_w=w, counts=counts,
                    prob_sum=prob_sum, keep=keep, assign=assign, rounds=rounds, y=y, rows=rows)

    def _bwd_inputs(self, x, w_router, wg, wu, wd, k, dy, logit_bias, sel_bias):
        xd, x = _stored(x)
        wdt, w_router = _stored(w_router)
        mats = []
        for m in (wg, wu, wd):
            dt, m = _stored(m)
            assert dt == wdt, "weights share one stored type"
            mats.append(m)
        T, d = x.shape
        N = w_router.shape[0]
        E, d_ff = mats[0].shape[0], mats[0].shape[1]
        lb = None if logit_bias is None else _c(logit_bias, np.float64)
        sb = None if sel_bias is None else _c(sel_bias, np.float32)
        dy = _c(dy, np.float64)
        assert dy.shape == (T, d)
        return xd, x, wdt, w_router, mats, T, d, N, E, d_ff, lb, sb, dy

    def layer_backward(self, x, w_router, wg, wu, wd, k, dy, gate_mode=GATE_TOPK_SOFTMAX,
                       logit_bias=None, sel_bias=None, n_shared=0, capacity=0, alpha=0.01,
                       aux_grad=1.0, reroute=False):
        """Gradients of sum(dy * y) + aux_grad * aux for all tokens (routing
        held fixed; capacity overflow dropped, or rerouted with ``reroute``): dict of dx [T,d], dw_router [N,d], dw_gate / dw_up
        [E,d_ff,d], dw_down [E,d,d_ff], fp64. Stacked weight arrays, shared
        experts last (E = N + n_shared)."""
        (xd, x, wdt, w_router, mats, T, d, N, E, d_ff, lb, sb,
         dy) = self._bwd_inputs(x, w_router, wg, wu, wd, k, dy, logit_bias, sel_bias)
        assert E == N + n_shared
        out = dict(dx=np.empty((T, d)), dw_router=np.empty((N, d)),
                   dw_gate=np.empty((E, d_ff, d)), dw_up=np.empty((E, d_ff, d)),
                   dw_down=np.empty((E, d, d_ff)))
        self.lib.oracle_layer_backward(
            T, d, d_ff, N, k, n_shared, gate_mode, capacity, int(bool(reroute)), xd, _ptr(x), wdt,
            _ptr(w_router), _ptr(lb), _ptr(sb), _ptr(mats[0]), _ptr(mats[1]), _ptr(mats[2]), _ptr(dy),
            float(alpha), float(aux_grad), _ptr(out["dx"]), _ptr(out["dw_router"]),
            _ptr(out["dw_gate"]), _ptr(out["dw_up"]), _ptr(out["dw_down"]))
        return out

    def backward_samples(self, x, w_router, experts, N, k, dy, tokens=(), columns=(),
                         gate_mode=GATE_TOPK_SOFTMAX, logit_bias=None, sel_bias=None,
                         n_shared=0, capacity=0, alpha=0.01, aux_grad=1.0, reroute=False):
        """The same gradients at sampled places: dx rows of ``tokens``; for
        each (e, j) of ``columns`` the row j of dw_gate[e] and dw_up[e] and
        the column j of dw_down[e] (each length d). ``experts`` maps an
        expert index (shared ones after the N routed) to its stored
        (wg, wu, wd); experts no sample needs may be absent."""
        xd, x = _stored(x)
        wdt, w_router = _stored(w_router)
        T, d = x.shape
        E = N + n_shared
        refs = []
        tabs = [(_P * E)(), (_P * E)(), (_P * E)()]
        d_ff = None
        for e, mats in experts.items():
            for j, m in enumerate(mats):
                dt, m = _stored(m)
                assert dt == wdt, "weights share one stored type"
                refs.append(m)
                tabs[j][e] = m.ctypes.data
            d_ff = mats[0].shape[0]
        lb = None if logit_bias is None else _c(logit_bias, np.float64)
        sb = None if sel_bias is None else _c(sel_bias, np.float32)
        dy = _c(dy, np.float64)
        toks = _c(list(tokens), np.int32)
        cols = np.asarray(list(columns), np.int32).reshape(-1, 2)
        we, wj = _c(cols[:, 0], np.int32), _c(cols[:, 1], np.int32)
        out = dict(dx_rows=np.empty((toks.size, d)), dw_gate_rows=np.empty((we.size, d)),
                   dw_up_rows=np.empty((we.size, d)), dw_down_cols=np.empty((we.size, d)))
        rc = self.lib.oracle_backward_samples(
            T, d, d_ff, N, k, n_shared, gate_mode, capacity, int(bool(reroute)), xd, _ptr(x), wdt,
            _ptr(w_router), _ptr(lb), _ptr(sb), tabs[0], tabs[1], tabs[2], _ptr(dy), float(alpha),
            float(aux_grad), toks.size, _ptr(toks), _ptr(out["dx_rows"]), we.size, _ptr(we),
            _ptr(wj), _ptr(out["dw_gate_rows"]), _ptr(out["dw_up_rows"]),
            _ptr(out["dw_down_cols"]))
        if rc != 0:
            raise ValueError("oracle_backward_samples: a sample needs an expert not supplied")
        return out

    def balance_backward(self, x, w_router, k, gate_mode=GATE_TOPK_SOFTMAX, logit_bias=None,
                         sel_bias=None, alpha=0.01, aux_grad=1.0):
        """dx [T,d] and dw_router [N,d] when dy = 0 (the balance term alone)."""
        xd, x = _stored(x)
        wdt, w_router = _stored(w_router)
        T, d = x.shape
        N = w_router.shape[0]
        lb = None if logit_bias is None else _c(logit_bias, np.float64)
        sb = None if sel_bias is None else _c(sel_bias, np.float32)
        dx = np.empty((T, d))
        dwr = np.empty((N, d))
        self.lib.oracle_balance_backward(T, d, N, k, gate_mode, xd, _ptr(x), wdt, _ptr(w_router),
                                         _ptr(lb), _ptr(sb), float(alpha), float(aux_grad),
                                         _ptr(dx), _ptr(dwr))
        return dx, dwr
