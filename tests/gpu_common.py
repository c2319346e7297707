"""Helpers of the GPU parity tests: seeded inputs with the top-k margin
guarantee, calls through the C ABI, host copies for the oracle, and the
error measures the tolerances are stated in.

Expected values come only from the oracle run on the generated inputs; no
output of the CUDA library is ever fed to the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import sparse_mixture_experts_router_gb300 as moe
from sparse_mixture_experts_router_gb300 import synth

MIN_MARGIN = 1e-3   # order margin of generated tokens (fp64 keys): fixes the
                    # top-k set and its order against fp32 score rounding
BF16_TOL = 2e-2     # max |y - y_ref| / max |y_ref|, bf16 weights and activations
F32_TOL = 1e-5      # same measure, fp32 layers
# Router scores computed from x and W_r are fp32 sums of d_model products;
# the tensor cores and the CUDA cores add them in another order than the
# oracle (fp64, rounded once), which moves a score by up to ~1e-4 at
# d_model = 7168. Gate weights are a softmax of the scores: for either gate
# mode, sum_j |dg_i/dr_j| <= 2 g_i (1 - g_i) <= 1/2, so a score error of
# SCORE_TOL moves a weight by at most SCORE_TOL / 2.
SCORE_TOL = 1e-4
GATE_TOL = SCORE_TOL / 2


def capacity_of(w: synth.Workload) -> int:
    return moe.capacity_for(w.capacity_factor, w.T, w.top_k, w.n_experts) \
        if w.capacity_factor > 0 else 0


def cfg_of(w: synth.Workload) -> moe.moe_config:
    return moe.config(T=w.T, d_model=w.d_model, n_experts=w.n_experts, top_k=w.top_k,
                      d_ff=w.d_ff, n_shared=w.n_shared,
                      dtype=moe.MOE_BF16 if w.dtype == "bf16" else moe.MOE_F32,
                      gate_mode=w.gate_mode, capacity=capacity_of(w), tiles=w.tiles,
                      gather=w.gather, overflow=w.overflow)


def host(t):
    """numpy copy of a device tensor in the form the oracle reads (bf16 as
    uint16 bit patterns); None stays None."""
    if t is None:
        return None
    return synth.bf16_bits(t)


def margin_inputs(w: synth.Workload, oracle, device="cuda", max_rounds=30, all_keys=False):
    """Workload inputs whose tokens all have an order margin >= 1e-3: the
    k+1 largest keys (all N with all_keys, which capacity rerouting ranks)
    are pairwise at least 1e-3 apart, so the kept set and its order do not
    depend on how the scores are rounded (tokens below it are redrawn from
    fresh N(0,1) draws)."""
    inp = synth.make_inputs(w, device)
    W = host(inp["w_router"])
    lb = None if inp["logit_bias"] is None else inp["logit_bias"].double().cpu().numpy()
    sb = host(inp["sel_bias"])
    rows = np.arange(w.T)
    for rnd in range(max_rounds):
        xs = host(inp["x"][torch.as_tensor(rows, device=inp["x"].device)])
        r64, _ = oracle.router_logits(xs, W, lb)
        m = oracle.order_margin(r64, w.n_experts - 1 if all_keys else w.top_k, sb)
        bad = rows[m < MIN_MARGIN]
        if bad.size == 0:
            return inp
        synth.redraw_rows(inp["x"], bad.tolist(), w.seed, rnd)
        rows = bad
    raise RuntimeError("could not reach the order margin")


def oracle_routing(oracle, w, inp):
    """Routing of all tokens by the oracle: (r64, topk_idx, topk_w, counts, prob_sum)."""
    lb = None if inp["logit_bias"] is None else inp["logit_bias"].double().cpu().numpy()
    r64, r32 = oracle.router_logits(host(inp["x"]), host(inp["w_router"]), lb)
    idx, tw, counts, ps = oracle.route(r32, w.top_k, w.gate_mode, host(inp["sel_bias"]))
    return r64, idx, tw, counts, ps


_HOST_WEIGHTS = []  # [(device tensors, host copies)] of the last workload


def host_weights(inp):
    """Host copies (oracle form) of the three expert weight tensors, made
    once per set of device tensors: one copy each rather than one per
    expert and batch of tokens. The cache holds the device tensors it was
    made from, so their memory cannot be reused by other tensors while it
    is cached."""
    dev = tuple(inp[n] for n in ("w_gate", "w_up", "w_down"))
    if not (_HOST_WEIGHTS and all(a is b for a, b in zip(_HOST_WEIGHTS[0][0], dev))):
        _HOST_WEIGHTS.clear()
        _HOST_WEIGHTS.append((dev, tuple(host(t) for t in dev)))
    return _HOST_WEIGHTS[0][1]


def oracle_rows(oracle, w, inp, idx, tw, rows, max_experts=40, fp8=False, nvfp4=False,
                assign=None):
    """Oracle layer output for the listed tokens. The oracle gets only the
    experts those tokens use, a batch of tokens at a time: FP8 and NVFP4
    quantize every expert they are given, so a batch is limited to
    max_experts; bf16 and fp32 take all tokens in one batch. ``assign`` (the
    oracle's rerouted experts, -1 dropped) replaces the capacity cut."""
    rows = [int(r) for r in rows]
    xh = host(inp["x"])
    wg, wu, wd = host_weights(inp)
    if assign is None:
        keep = oracle.capacity_keep(idx, w.n_experts, capacity_of(w))
    else:
        keep = (np.asarray(assign).ravel() >= 0).astype(np.uint8)
        idx = np.where(np.asarray(assign) >= 0, assign, idx).astype(np.int32)
    out = np.empty((len(rows), w.d_model), np.float64)
    shared = list(range(w.n_experts, w.n_experts + w.n_shared))
    limit = max_experts if (fp8 or nvfp4) else w.n_experts + w.n_shared
    i = 0
    while i < len(rows):
        batch, need = [], set(shared)
        while i < len(rows):
            cand = need | set(idx[rows[i]].tolist())
            if batch and len(cand) > limit:
                break
            need = cand
            batch.append(rows[i])
            i += 1
        experts = {e: (wg[e], wu[e], wd[e]) for e in sorted(need)}
        y = oracle.layer_rows(xh, experts, idx, tw, batch, w.n_experts, w.n_shared, keep, fp8,
                              nvfp4)
        out[i - len(batch):i] = y
    return out


class LayerRun:
    """Device outputs of one moe_layer_forward call."""

    def __init__(self, w: synth.Workload, inp: dict, device="cuda"):
        self.cfg = cfg_of(w)
        T, N, k = w.T, w.n_experts, w.top_k
        self.y = torch.full((T, w.d_model), float("nan"), dtype=w.torch_dtype, device=device)
        self.topk_idx = torch.full((T, k), -1, dtype=torch.int32, device=device)
        self.topk_w = torch.zeros((T, k), dtype=torch.float32, device=device)
        self.counts = torch.full((N,), -1, dtype=torch.int32, device=device)
        self.prob_sum = torch.full((N,), float("nan"), dtype=torch.float32, device=device)
        self.ws = moe.workspace(self.cfg, "layer", device)
        self.inp = inp

    def __call__(self):
        i = self.inp
        moe.moe_layer_forward(self.cfg, i["x"], i["w_router"], i["logit_bias"], i["sel_bias"],
                              i["w_gate"], i["w_up"], i["w_down"], self.y, self.topk_idx,
                              self.topk_w, self.counts, self.prob_sum, self.ws)
        return self

    def status(self):
        return moe.moe_stream_status(self.ws)


def rel_inf(y, ref):
    """max |y - ref| / max |ref| over all elements."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(y - ref).max() / (den if den > 0 else 1.0))


def sample_rows(T, n, seed=0):
    """n token rows including the first and the last."""
    if T <= n:
        return list(range(T))
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, T - 1), size=n - 2, replace=False)
    return sorted([0, T - 1] + mid.tolist())


def segment_edge_rows(idx, n_experts, capacity=0, n_random=8, seed=0, max_experts=None):
    """Token rows whose outputs cover both ends of expert segments: the owner
    of each routed expert's first row and of its last kept row (the row of
    the segment's last, usually partial, M tile), plus n_random other
    tokens, first and last token included. Rows inside a segment are in
    ascending token order, so an expert's first and last rows belong to the
    smallest and the largest token that chose it (with a capacity C, the
    C-th smallest). max_experts, when given, takes that many experts evenly
    spread over [0, N) instead of all of them."""
    idx = np.asarray(idx)
    T = idx.shape[0]
    rows = set(sample_rows(T, max(2, n_random), seed=seed))
    experts = range(n_experts)
    if max_experts is not None and max_experts < n_experts:
        experts = sorted(set(np.linspace(0, n_experts - 1, max_experts).round().astype(int)))
    for e in experts:
        toks = np.nonzero((idx == e).any(axis=1))[0]
        if toks.size == 0:
            continue
        last = toks.size - 1 if capacity <= 0 else min(toks.size, capacity) - 1
        rows.add(int(toks[0]))
        rows.add(int(toks[last]))
    return sorted(rows)


def grouped_tiles(counts, T, n_shared, d_model, d_ff, tile_m):
    """Work tiles of the two grouped GEMMs when every segment is cut into
    tile_m-row tiles: (gate/up tiles of 128 SwiGLU columns, down tiles of
    256 output columns)."""
    mt = sum((int(c) + tile_m - 1) // tile_m for c in counts)
    mt += n_shared * ((T + tile_m - 1) // tile_m)
    return mt * ((d_ff + 127) // 128), mt * ((d_model + 255) // 256)
