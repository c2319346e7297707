"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function takes an :class:`oracle.Oracle` and raises
``AssertionError`` when the oracle disagrees with:

* values the pages print for a worked example (``tests/golden/*.json``, each
  with its citation),
* closed forms worked out by hand in the pin,
* special cases that reduce to a library routine (numpy / torch fp64 matmul,
  ``torch.nn.functional.silu``, ``torch.topk`` on distinct keys), or
* brute force on tiny inputs (every expert evaluated densely, unselected ones
  given weight zero).

``test_oracle_pins.py`` runs them against the real oracle;
``test_oracle_mutations.py`` runs them against builds of the oracle with one
planted mistake each and checks that some pin fails for every mistake.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- the pages --
def pin_worked_example_top2_of_4(o):
    """Mixture of experts and speculative decoding, 'Following one token
    through an MoE layer': scores -> kept experts -> weights -> blend."""
    g = golden("worked_example_top2_of_4.json")
    tol = g["tolerance"]
    r32 = np.array([g["scores"]], np.float32)
    idx, w, counts, _ = o.route(r32, g["k"], gate_mode=0)
    assert idx[0].tolist() == g["kept_experts_0_based"], idx
    assert np.allclose(w[0], g["top2_softmax_weights"], atol=tol), w
    idx2, w2, _, _ = o.route(r32, g["k"], gate_mode=1)
    assert idx2[0].tolist() == g["kept_experts_0_based"]
    assert np.allclose(w2[0], g["top2_softmax_weights"], atol=tol), w2
    p = o.softmax(np.array(g["scores"]))
    assert np.allclose(p[g["kept_experts_0_based"]], g["all_expert_softmax_of_kept"], atol=tol), p
    y = o.gated_sum(w[0], np.array(g["expert_outputs_of_kept"]))
    assert np.allclose(y, g["blend"], atol=tol), y
    assert counts.tolist() == [1, 0, 1, 0]


def pin_dense_and_sparse_4_experts(o):
    """Mixture of Experts and Guided Decoding: dense softmax over 4 gate
    scores, and the sparse top-2 weights with zeros elsewhere."""
    g = golden("dense_and_sparse_4_experts.json")
    s = np.array(g["scores"])
    p = o.softmax(s)
    assert np.allclose(p, g["dense_softmax_printed"], atol=g["dense_softmax_tolerance"]), p
    idx, w, _, _ = o.route(np.array([s], np.float32), g["k"], gate_mode=0)
    dense = np.zeros(s.size)
    dense[idx[0]] = w[0]
    assert np.allclose(dense, g["sparse_weights_printed"], atol=g["sparse_tolerance"]), dense


def pin_gated_sum_3_experts(o):
    """Mixture of Experts and Guided Decoding: 0.5*2 + 0.3*4 + 0.2*0 = 2.2."""
    g = golden("gated_sum_3_experts.json")
    y = o.gated_sum(np.array(g["gates"]), np.array(g["expert_outputs"])[:, None])
    assert abs(y[0] - g["output"]) <= g["tolerance"], y


def pin_balance_loss_n4(o):
    """Balanced routing gives 1.0*alpha, the collapsed one 2.8*alpha, both
    from the printed f and P and realised as actual routings of 4 tokens."""
    g = golden("balance_loss_n4.json")
    a, tol = g["alpha"], g["tolerance"]
    for case in ("balanced", "collapsed"):
        c = g[case]
        loss = o.balance_loss(c["f"], c["P"], a)
        assert abs(loss - c["loss_over_alpha"] * a) <= tol, (case, loss)
    # Realised: token t strongly prefers expert t (k = 1); by symmetry every
    # expert gets one token and mean probability exactly 1/4.
    r = np.full((4, 4), -3.0, np.float32)
    np.fill_diagonal(r, 2.0)
    idx, _, counts, ps = o.route(r, 1)
    f, P, aux = o.balance_stats(counts, ps, 4, 1, a)
    assert idx[:, 0].tolist() == [0, 1, 2, 3]
    assert np.allclose(f, 0.25, atol=1e-15) and np.allclose(P, 0.25, atol=1e-9)
    assert abs(aux - 1.0 * a) <= 1e-9, aux
    # Collapsed: every token has softmax [0.7, 0.1, 0.1, 0.1] and picks 0.
    r = np.tile(np.log(np.array([0.7, 0.1, 0.1, 0.1])), (4, 1)).astype(np.float32)
    idx, _, counts, ps = o.route(r, 1)
    f, P, aux = o.balance_stats(counts, ps, 4, 1, a)
    assert idx[:, 0].tolist() == [0, 0, 0, 0]
    assert np.allclose(f, [1, 0, 0, 0]) and np.allclose(P, [0.7, 0.1, 0.1, 0.1], atol=1e-6)
    assert abs(aux - 2.8 * a) <= 1e-7, aux


# ------------------------------------------------------------- closed forms --
def pin_renormalised_all_softmax_equals_topk_softmax(o):
    """Softmax over all N then renormalising the kept k equals the softmax
    over the kept k (exact identity; equal up to rounding)."""
    rng = _rng(1)
    r = rng.normal(0, 2, (50, 16)).astype(np.float32)
    for k in (1, 2, 5, 16):
        i0, w0, _, _ = o.route(r, k, gate_mode=0)
        i1, w1, _, _ = o.route(r, k, gate_mode=1)
        assert (i0 == i1).all()
        assert np.allclose(w0, w1, atol=1e-12, rtol=0), np.abs(w0 - w1).max()
        assert np.allclose(w0.sum(1), 1.0, atol=1e-12)


def pin_tie_break_lower_index(o):
    """Equal keys go to the lower expert index; slots are ordered best first."""
    key = np.array([1.0, 3.0, 3.0, 2.0, 3.0], np.float32)
    assert o.topk(key, 2).tolist() == [1, 2]
    assert o.topk(key, 4).tolist() == [1, 2, 4, 3]
    assert o.topk(np.zeros(6, np.float32), 3).tolist() == [0, 1, 2]
    # -0.0 and +0.0 compare equal, so they tie as well
    assert o.topk(np.array([-0.0, 0.0], np.float32), 1).tolist() == [0]


def pin_selection_bias_chooses_but_does_not_weigh(o):
    """A selection bias changes which experts are chosen, not their weights:
    scores [2.0, 0.5, 1.5, -1.0] with +1.2 on expert 1 keep experts {0, 1},
    weighted by the softmax of the unbiased scores [2.0, 0.5]."""
    r = np.array([[2.0, 0.5, 1.5, -1.0]], np.float32)
    sb = np.array([0.0, 1.2, 0.0, 0.0], np.float32)
    e = math.exp(1.5)
    for mode in (0, 1):
        idx, w, _, ps = o.route(r, 2, gate_mode=mode, sel_bias=sb)
        assert idx[0].tolist() == [0, 1], idx
        assert np.allclose(w[0], [e / (1 + e), 1 / (1 + e)], atol=1e-7), w
        # P_i uses the unbiased scores too
        assert np.allclose(ps, o.softmax(r[0].astype(np.float64)), atol=1e-15)


def pin_router_logits_small(o):
    """r = x W_r^T + logit_bias, worked by hand: x = [1, 2], rows of W_r
    [1, 0], [0, 1], [1, 1], [-2, 0.5] -> [1, 2, 3, -1], plus the bias."""
    x = np.array([[1.0, 2.0]], np.float32)
    W = np.array([[1, 0], [0, 1], [1, 1], [-2, 0.5]], np.float32)
    lb = np.array([0.5, -0.25, 0.0, 4.0])
    r64, r32 = o.router_logits(x, W, lb)
    assert r64[0].tolist() == [1.5, 1.75, 3.0, 3.0]
    assert r32.dtype == np.float32 and r32[0].tolist() == [1.5, 1.75, 3.0, 3.0]
    # bf16 inputs are read from their bit patterns: 0x3F80 = 1.0,
    # 0xC000 = -2.0, 0x3E20 = 0.15625, 0xBF40 = -0.75
    xb = np.array([[0x3F80, 0xC000]], np.uint16)
    Wb = np.array([[0x3E20, 0xBF40]], np.uint16)
    r64, _ = o.router_logits(xb, Wb)
    assert r64[0, 0] == 1.0 * 0.15625 + (-2.0) * (-0.75)


def pin_permute_small(o):
    """Pairs grouped by expert, ascending pair id inside an expert, worked
    by hand for topk_idx [[1,0],[1,2],[0,2]] (pair ids 0..5)."""
    off, sp, inv = o.permute(np.array([[1, 0], [1, 2], [0, 2]]), 3)
    assert off.tolist() == [0, 2, 4, 6]
    assert sp.tolist() == [1, 4, 0, 2, 3, 5]
    assert inv.tolist() == [2, 0, 3, 4, 1, 5]
    off, sp, inv = o.permute(np.zeros((0, 2), np.int32), 3)
    assert off.tolist() == [0, 0, 0, 0] and sp.size == 0


# ---------------------------------------------------- library reductions ------
def _torch_swiglu(x, wg, wu, wd):
    x, wg, wu, wd = (torch.from_numpy(np.asarray(a, np.float64)) for a in (x, wg, wu, wd))
    return (torch.nn.functional.silu(x @ wg.T) * (x @ wu.T)) @ wd.T


def pin_router_logits_match_matmul(o):
    rng = _rng(2)
    x = rng.normal(0, 1, (20, 24)).astype(np.float32)
    W = rng.normal(0, 0.5, (7, 24)).astype(np.float32)
    lb = rng.normal(0, 1, 7)
    r64, r32 = o.router_logits(x, W, lb)
    ref = x.astype(np.float64) @ W.astype(np.float64).T + lb
    assert np.allclose(r64, ref, atol=1e-12, rtol=0)
    assert (r32 == ref.astype(np.float32)).all()


def pin_route_matches_library(o):
    """Distinct keys: top-k equals torch.topk (sorted, descending); counts
    equal bincount; prob_sum equals the summed library softmax."""
    rng = _rng(3)
    r = rng.normal(0, 1, (200, 32)).astype(np.float32)
    for k in (1, 2, 8):
        idx, w, counts, ps = o.route(r, k)
        tv, ti = torch.topk(torch.from_numpy(r), k, dim=1, sorted=True)
        assert (idx == ti.numpy()).all()
        ref_w = torch.softmax(tv.double(), dim=1).numpy()
        assert np.allclose(w, ref_w, atol=1e-13)
        assert (counts == np.bincount(idx.ravel(), minlength=32)).all()
        ref_ps = torch.softmax(torch.from_numpy(r).double(), dim=1).sum(0).numpy()
        assert np.allclose(ps, ref_ps, atol=1e-12)


def pin_expert_swiglu_matches_library(o):
    """One expert = silu(x Wg^T) * (x Wu^T) then Wd^T; d != d_ff so a
    transposed operand cannot pass."""
    rng = _rng(4)
    d, dff = 12, 20
    x = rng.normal(0, 1, d)
    wg, wu = rng.normal(0, 0.5, (2, dff, d)).astype(np.float32)
    wd = rng.normal(0, 0.5, (d, dff)).astype(np.float32)
    out = o.expert_swiglu(x, wg, wu, wd)
    ref = _torch_swiglu(x[None], wg, wu, wd)[0].numpy()
    assert np.allclose(out, ref, atol=1e-12, rtol=0), np.abs(out - ref).max()


def pin_single_expert_layer_is_plain_ffn(o):
    """N = 1, k = 1: the layer is one SwiGLU FFN with weight 1."""
    rng = _rng(5)
    T, d, dff = 6, 8, 16
    x = rng.normal(0, 1, (T, d)).astype(np.float32)
    Wr = rng.normal(0, 1, (1, d)).astype(np.float32)
    wg, wu = rng.normal(0, 0.5, (2, 1, dff, d)).astype(np.float32)
    wd = rng.normal(0, 0.5, (1, d, dff)).astype(np.float32)
    out = o.layer(x, Wr, wg, wu, wd, k=1)
    ref = _torch_swiglu(x, wg[0], wu[0], wd[0]).numpy()
    assert np.allclose(out["y"], ref, atol=1e-12, rtol=0)
    assert np.allclose(out["topk_w"], 1.0)


def pin_k_equals_n_is_dense_softmax_moe(o):
    """k = N with the top-k softmax is the dense MoE: every expert runs,
    weighted by the softmax over all scores."""
    rng = _rng(6)
    T, d, dff, N = 5, 8, 12, 4
    x = rng.normal(0, 1, (T, d)).astype(np.float32)
    Wr = rng.normal(0, 1, (N, d)).astype(np.float32)
    wg, wu = rng.normal(0, 0.5, (2, N, dff, d)).astype(np.float32)
    wd = rng.normal(0, 0.5, (N, d, dff)).astype(np.float32)
    out = o.layer(x, Wr, wg, wu, wd, k=N)
    r = torch.from_numpy(x).double() @ torch.from_numpy(Wr).double().T
    G = torch.softmax(r.float().double(), dim=1)
    ref = sum(G[:, e:e + 1] * _torch_swiglu(x, wg[e], wu[e], wd[e]) for e in range(N))
    assert np.allclose(out["y"], ref.numpy(), atol=1e-12, rtol=0)


# ------------------------------------------------------------- brute force ----
def _brute_force_layer(x, Wr, wg, wu, wd, k, N, n_shared, mode, lb=None, sb=None):
    """Dense evaluation: every expert on every token; the routed ones
    weighted by a length-N gate vector that is zero off the top-k."""
    xt = torch.from_numpy(np.asarray(x, np.float64))
    r = xt @ torch.from_numpy(np.asarray(Wr, np.float64)).T
    if lb is not None:
        r = r + torch.from_numpy(np.asarray(lb, np.float64))
    r32 = r.float()
    key = r32 + (torch.from_numpy(np.asarray(sb, np.float32)) if sb is not None else 0)
    T = xt.shape[0]
    y = torch.zeros(T, xt.shape[1], dtype=torch.float64)
    for t in range(T):
        # rank experts by (key desc, index asc) without a sort routine
        order = sorted(range(N), key=lambda e: (-float(key[t, e]), e))[:k]
        rt = r32[t].double()
        G = torch.zeros(N, dtype=torch.float64)
        if mode == 0:
            z = sum(math.exp(float(rt[e]) - float(rt[order].max())) for e in order)
            for e in order:
                G[e] = math.exp(float(rt[e]) - float(rt[order].max())) / z
        else:
            p = torch.softmax(rt, 0)
            for e in order:
                G[e] = p[e] / p[order].sum()
        for e in range(N):
            y[t] += G[e] * _torch_swiglu(xt[t:t + 1].numpy(), wg[e], wu[e], wd[e])[0]
        for s in range(n_shared):
            y[t] += _torch_swiglu(xt[t:t + 1].numpy(), wg[N + s], wu[N + s], wd[N + s])[0]
    return y.numpy()


def pin_brute_force_dense_with_zeroed_gates(o):
    rng = _rng(7)
    T, d, dff, N, k, s = 7, 10, 6, 6, 2, 1
    for mode in (0, 1):
        x = rng.normal(0, 1, (T, d)).astype(np.float32)
        Wr = rng.normal(0, 1, (N, d)).astype(np.float32)
        lb = rng.normal(0, 0.5, N)
        sb = rng.uniform(-0.3, 0.3, N).astype(np.float32)
        wg, wu = rng.normal(0, 0.5, (2, N + s, dff, d)).astype(np.float32)
        wd = rng.normal(0, 0.5, (N + s, d, dff)).astype(np.float32)
        out = o.layer(x, Wr, wg, wu, wd, k=k, gate_mode=mode, logit_bias=lb,
                      sel_bias=sb, n_shared=s)
        ref = _brute_force_layer(x, Wr, wg, wu, wd, k, N, s, mode, lb, sb)
        assert np.allclose(out["y"], ref, atol=1e-12, rtol=0), np.abs(out["y"] - ref).max()


# -------------------------------------------------------------- invariants ---
def pin_permute_invariants(o):
    rng = _rng(8)
    T, N, k = 300, 9, 3
    idx = np.stack([rng.permutation(N)[:k] for _ in range(T)]).astype(np.int32)
    off, sp, inv = o.permute(idx, N)
    P = T * k
    assert off[0] == 0 and off[-1] == P and (np.diff(off) >= 0).all()
    assert (np.diff(off) == np.bincount(idx.ravel(), minlength=N)).all()
    assert sorted(sp.tolist()) == list(range(P))
    assert (inv[sp] == np.arange(P)).all()
    flat = idx.ravel()
    for e in range(N):
        seg = sp[off[e]:off[e + 1]]
        assert (flat[seg] == e).all() and (np.diff(seg) > 0).all()


def pin_expert_relabelling_is_equivariant(o):
    """Relabelling the experts (router rows, biases and weights together)
    relabels topk_idx and counts the same way and leaves y unchanged."""
    rng = _rng(9)
    T, d, dff, N, k = 9, 8, 6, 5, 2
    x = rng.normal(0, 1, (T, d)).astype(np.float32)
    Wr = rng.normal(0, 1, (N, d)).astype(np.float32)
    lb = rng.normal(0, 0.5, N)
    sb = rng.uniform(-0.2, 0.2, N).astype(np.float32)
    wg, wu = rng.normal(0, 0.5, (2, N, dff, d)).astype(np.float32)
    wd = rng.normal(0, 0.5, (N, d, dff)).astype(np.float32)
    a = o.layer(x, Wr, wg, wu, wd, k, 1, lb, sb)
    perm = rng.permutation(N)            # new expert j is old expert perm[j]
    b = o.layer(x, Wr[perm], wg[perm], wu[perm], wd[perm], k, 1, lb[perm], sb[perm])
    assert (perm[b["topk_idx"]] == a["topk_idx"]).all()
    assert (b["counts"] == a["counts"][perm]).all()
    assert np.allclose(a["y"], b["y"], atol=1e-12)


def pin_shared_expert_always_runs_with_weight_one(o):
    """Adding a shared expert adds exactly its plain FFN output."""
    rng = _rng(10)
    T, d, dff, N, k = 4, 8, 6, 3, 1
    x = rng.normal(0, 1, (T, d)).astype(np.float32)
    Wr = rng.normal(0, 1, (N, d)).astype(np.float32)
    wg, wu = rng.normal(0, 0.5, (2, N + 1, dff, d)).astype(np.float32)
    wd = rng.normal(0, 0.5, (N + 1, d, dff)).astype(np.float32)
    a = o.layer(x, Wr, wg[:N], wu[:N], wd[:N], k)
    b = o.layer(x, Wr, wg, wu, wd, k, n_shared=1)
    ref = _torch_swiglu(x, wg[N], wu[N], wd[N]).numpy()
    assert np.allclose(b["y"] - a["y"], ref, atol=1e-12)
    assert (b["counts"] == a["counts"]).all()


def pin_selection_margin_small(o):
    """Worked by hand: keys [3, 1, 2.5, 0] (+ bias [0, 2, 0, 0] -> [3, 3, 2.5,
    0]); the gap after the k-th largest."""
    r = np.array([[3.0, 1.0, 2.5, 0.0]])
    assert np.allclose(o.selection_margin(r, 1), [0.5])
    assert np.allclose(o.selection_margin(r, 2), [1.5])
    assert np.allclose(o.selection_margin(r, 3), [1.0])
    assert np.isinf(o.selection_margin(r, 4)).all()
    sb = np.array([0.0, 2.0, 0.0, 0.0], np.float32)
    assert np.allclose(o.selection_margin(r, 1, sb), [0.0])
    assert np.allclose(o.selection_margin(r, 2, sb), [0.5])


def pin_order_margin_small(o):
    """Worked by hand: keys [10, 0, 7, 6.9, 3] sort to 10, 7, 6.9, 3, 0 with
    neighbour gaps 3, 0.1, 3.9, 3. The selection margin at k = 3 is 3.9, but
    the kept experts 7 and 6.9 are only 0.1 apart."""
    r = np.array([[10.0, 0.0, 7.0, 6.9, 3.0]])
    assert np.allclose(o.order_margin(r, 1), [3.0])
    for k in (2, 3, 4, 5):
        assert np.allclose(o.order_margin(r, k), [0.1])
    assert np.allclose(o.selection_margin(r, 3), [3.9])
    sb = np.array([0.0, 0.0, 0.0, 0.0, 7.0], np.float32)   # 3 + 7 ties with 10
    assert np.allclose(o.order_margin(r, 1, sb), [0.0])
    assert np.isinf(o.order_margin(np.array([[1.5]]), 1)).all()


def pin_order_margin_is_min_pairwise_distance(o):
    """Brute force: the smallest neighbour gap of a sorted set is the
    smallest distance over all pairs of the set; the set is the k+1 largest
    keys (all N when k = N), found here with numpy's argsort."""
    rng = _rng(12)
    for T, N in ((40, 6), (30, 9)):
        r = rng.normal(0, 1, (T, N))
        sb = rng.uniform(-0.3, 0.3, N).astype(np.float32)
        for k in range(1, N + 1):
            got = o.order_margin(r, k, sb)
            key = r + sb.astype(np.float64)
            m = min(k + 1, N)
            for t in range(T):
                top = key[t][np.argsort(-key[t], kind="stable")[:m]]
                best = min(abs(a - b) for i, a in enumerate(top) for b in top[i + 1:])
                assert abs(got[t] - best) <= 1e-15, (T, N, k, t)


def pin_capacity_hand_worked(o):
    """Worked by hand, capacity 1 ("Keeping the experts busy": the extras
    are dropped; the earlier tokens are kept). Pairs in order: p0 (token 0,
    expert 0), p1 (0, 1), p2 (1, 1), p3 (1, 0), p4 (2, 0), p5 (2, 2). Expert
    0 keeps p0 and drops p3, p4; expert 1 keeps p1 and drops p2; expert 2
    keeps p5."""
    idx = np.array([[0, 1], [1, 0], [0, 2]])
    assert o.capacity_keep(idx, 3, 1).tolist() == [1, 1, 0, 0, 0, 1]
    off, sp, inv = o.permute(idx, 3, capacity=1)
    assert off.tolist() == [0, 1, 2, 3]
    assert sp.tolist() == [0, 1, 5]
    assert inv.tolist() == [0, 1, -1, -1, -1, 2]
    # capacity 2: expert 0 keeps p0, p3 and drops p4
    assert o.capacity_keep(idx, 3, 2).tolist() == [1, 1, 1, 1, 0, 1]
    off, sp, inv = o.permute(idx, 3, capacity=2)
    assert off.tolist() == [0, 2, 4, 5] and sp.tolist() == [0, 3, 1, 2, 5]
    # 0 means no cap; a cap at the largest count drops nothing either
    for cap in (0, 3):
        assert o.capacity_keep(idx, 3, cap).all()


def pin_capacity_layer_is_dense_with_dropped_gates_zeroed(o):
    """Brute force: with a capacity, the layer equals the dense evaluation
    of every expert on every token with the gate of each unselected or
    dropped pair set to zero; with no capacity (or one no expert exceeds)
    it equals the uncapped layer."""
    rng = _rng(13)
    T, d, dff, N, k = 9, 8, 6, 3, 2
    x = rng.normal(0, 1, (T, d))
    Wr = rng.normal(0, 1, (N, d))
    wg = rng.normal(0, 0.5, (N, dff, d))
    wu = rng.normal(0, 0.5, (N, dff, d))
    wd = rng.normal(0, 0.5, (N, d, dff))
    base = o.layer(x, Wr, wg, wu, wd, k)
    for cap in (1, 2, 4):
        out = o.layer(x, Wr, wg, wu, wd, k, capacity=cap)
        keep = out["keep"].reshape(T, k)
        for t in range(T):
            ref = np.zeros(d)
            for s in range(k):
                if keep[t, s]:
                    e = out["topk_idx"][t, s]
                    ref += out["topk_w"][t, s] * _torch_swiglu(x[t:t + 1], wg[e], wu[e], wd[e]).numpy()[0]
            assert np.allclose(out["y"][t], ref, atol=1e-12)
        counts = np.bincount(out["topk_idx"].ravel(), minlength=N)
        assert int(keep.sum()) == int(np.minimum(counts, cap).sum())
    full = o.layer(x, Wr, wg, wu, wd, k, capacity=T)
    assert np.array_equal(full["y"], base["y"])


# ------------------------------------------------------- capacity reroute ---
# Reading of "Keeping the experts busy" (the extras are dropped or rerouted):
# after the capacity cut, overflowing pairs re-propose in rounds to their
# token's best expert (selection key, ties to the lower index) that has room
# and that the token does not hold; each expert takes proposals in ascending
# pair id up to its room; a pair with no candidate is dropped.

def _loads(assign, N):
    a = assign.ravel()
    return np.bincount(a[a >= 0], minlength=N)


def pin_reroute_hand_worked(o):
    """Worked by hand.

    Case 1 (N=5, k=2, C=1). Scores: t0 [5,4,3,2,1] -> experts 0,1;
    t1 [5,4,3,3,2] -> 0,1; t2 [4,5,1,3,1] -> 1,0; t3 [5,1,2,0,3] -> 0,4.
    Pairs p0..p7 = (t0:0,1) (t1:0,1) (t2:1,0) (t3:0,4). The cut: expert 0
    keeps p0 (p2, p5, p6 pend), expert 1 keeps p1 (p3, p4 pend), expert 4
    keeps p7. Rooms: e2 = e3 = 1, the rest 0. Round 1: t1's keys for e2 and
    e3 tie at 3, so p2 proposes e2 (lower index) and p3 e3; t2 prefers e3
    (3 > 1): p4 -> e3, p5 -> e2; t3 (holds 0 and 4): p6 -> e2 (2 > 0). e2
    takes p2 (before p5, p6), e3 takes p3 (before p4). Now every expert is
    full, so p4, p5, p6 are dropped in round 2: one round with proposals.

    Case 2 (N=4, k=1, C=1, all scores 0, selection bias [.1, .4, .3, .2]):
    every token ranks 1, 2, 3, 0. t0 keeps 1; round 1 gives 2 to t1, round
    2 gives 3 to t2, round 3 gives 0 to t3, and t4 finds no room: dropped.

    Case 3 (N=4, k=1, C=1, scores [2, NaN, 1, 0] for all three tokens):
    NaN ranks below every number, so t0 keeps 0, t1 gets 2, t2 gets 3."""
    r = np.array([[5, 4, 3, 2, 1], [5, 4, 3, 3, 2], [4, 5, 1, 3, 1], [5, 1, 2, 0, 3]], np.float32)
    idx, _, _, _ = o.route(r, 2)
    assert idx.tolist() == [[0, 1], [0, 1], [1, 0], [0, 4]]
    assign, rounds = o.reroute(r, idx, 1)
    assert assign.tolist() == [[0, 1], [2, 3], [-1, -1], [-1, 4]]
    assert rounds == 1

    r = np.zeros((5, 4), np.float32)
    sb = np.array([0.1, 0.4, 0.3, 0.2], np.float32)
    idx, _, _, _ = o.route(r, 1, sel_bias=sb)
    assert idx.ravel().tolist() == [1] * 5
    assign, rounds = o.reroute(r, idx, 1, sel_bias=sb)
    assert assign.ravel().tolist() == [1, 2, 3, 0, -1]
    assert rounds == 3

    r = np.array([[2, np.nan, 1, 0]] * 3, np.float32)
    idx = np.zeros((3, 1), np.int32)
    assign, rounds = o.reroute(r, idx, 1)
    assert assign.ravel().tolist() == [0, 2, 3]
    assert rounds == 2


def pin_reroute_identical_rankings_closed_form(o):
    """When every token has the same scores, the experts rank in one order
    o_0, o_1, ... (descending key, ties to the lower index). Then each round
    hands the next k experts of that order to the next C tokens, so token t,
    slot s runs on o_{k*floor(t/C) + s}, and is dropped when that index
    reaches N."""
    rng = _rng(21)
    for N, k, C, T in [(6, 2, 1, 5), (8, 3, 2, 9), (5, 1, 3, 20), (7, 2, 2, 8), (16, 4, 3, 17)]:
        row = rng.integers(0, 4, N).astype(np.float32)  # repeated values: ties
        sb = rng.integers(0, 3, N).astype(np.float32) * 0.5 if N % 2 == 0 else None
        key = row + (sb if sb is not None else 0)
        order = sorted(range(N), key=lambda e: (-key[e], e))
        r = np.tile(row, (T, 1))
        idx, _, _, _ = o.route(r, k, sel_bias=sb)
        assign, rounds = o.reroute(r, idx, C, sel_bias=sb)
        for t in range(T):
            for s in range(k):
                j = k * (t // C) + s
                assert assign[t, s] == (order[j] if j < N else -1), (N, k, C, T, t, s)


def pin_reroute_invariants(o):
    """On random scores (with and without a selection bias, and with ties):
    no expert runs more than C pairs; a token's experts are distinct; a pair
    the cut keeps stays on its expert; a rerouted pair runs on an expert
    outside its token's top k; a pair is dropped only when every expert its
    token does not hold is full; the rounds stop within N + 1; with C at
    least the largest count nothing moves."""
    rng = _rng(22)
    for T, N, k, C, bias, ties in [(40, 8, 2, 6, False, False), (60, 16, 4, 9, True, False),
                                   (33, 6, 3, 10, False, True), (50, 12, 1, 2, True, True),
                                   (80, 32, 8, 15, True, False)]:
        r = rng.normal(0, 1, (T, N)).astype(np.float32)
        r += np.linspace(2, 0, N, dtype=np.float32)  # skew: the low experts overflow
        if ties:
            r = np.round(r * 2) / 2
        sb = rng.uniform(-0.5, 0.5, N).astype(np.float32) if bias else None
        idx, _, counts, _ = o.route(r, k, sel_bias=sb)
        keep = o.capacity_keep(idx, N, C).reshape(T, k)
        assign, rounds = o.reroute(r, idx, C, sel_bias=sb)
        load = _loads(assign, N)
        assert (load <= C).all()
        assert 0 <= rounds <= N + 1
        for t in range(T):
            got = [e for e in assign[t] if e >= 0]
            assert len(got) == len(set(got))
            for s in range(k):
                if keep[t, s]:
                    assert assign[t, s] == idx[t, s]
                elif assign[t, s] >= 0:
                    assert assign[t, s] not in idx[t]
                else:
                    hold = set(idx[t].tolist()) | set(got)
                    assert all(load[e] == C for e in range(N) if e not in hold), (t, s)
        assert int((assign >= 0).sum()) >= int(keep.sum())
        big = int(counts.max())
        a2, rounds2 = o.reroute(r, idx, big, sel_bias=sb)
        assert np.array_equal(a2, idx) and rounds2 == 0
        a0, rounds0 = o.reroute(r, idx, 0, sel_bias=sb)
        assert np.array_equal(a0, idx) and rounds0 == 0


def pin_reroute_without_room_is_dropping(o):
    """If the cut leaves every expert full, rerouting has nowhere to send the
    extras: the result is the cut's (kept pairs stay, the rest are -1)."""
    rng = _rng(23)
    T, N, k = 64, 8, 2
    r = rng.normal(0, 1, (T, N)).astype(np.float32)
    idx, _, counts, _ = o.route(r, k)
    C = int(counts.min())
    assert C > 0
    keep = o.capacity_keep(idx, N, C).reshape(T, k)
    assign, rounds = o.reroute(r, idx, C)
    assert np.array_equal(assign, np.where(keep != 0, idx, -1))
    assert rounds == 0


def pin_reroute_layer_is_dense_with_assigned_experts(o):
    """Brute force: with rerouting, each token's output is the sum over its
    slots of the slot's gate weight times the FFN of the expert the slot runs
    on (nothing for a dropped slot), every expert evaluated densely."""
    rng = _rng(24)
    T, d, dff, N, k, C = 10, 8, 6, 4, 2, 2
    x = rng.normal(0, 1, (T, d))
    Wr = rng.normal(0, 1, (N, d))
    Wr[0] += 1.5 * x.mean(0)  # expert 0 popular: it overflows
    wg = rng.normal(0, 0.5, (N, dff, d))
    wu = rng.normal(0, 0.5, (N, dff, d))
    wd = rng.normal(0, 0.5, (N, d, dff))
    out = o.layer(x, Wr, wg, wu, wd, k, capacity=C, reroute=True)
    assign = out["assign"]
    assert (assign != out["topk_idx"]).any() and (assign >= 0).any()
    dense = [_torch_swiglu(x, wg[e], wu[e], wd[e]).numpy() for e in range(N)]
    for t in range(T):
        ref = np.zeros(d)
        for s in range(k):
            if assign[t, s] >= 0:
                ref += out["topk_w"][t, s] * dense[assign[t, s]][t]
        assert np.allclose(out["y"][t], ref, atol=1e-12)


# ------------------------------------------------------------------- FP8 ---
def pin_e4m3_fixed_points(o):
    """E4M3 from its definition (bias 7, 3 mantissa bits, subnormals m*2^-9,
    largest finite 448, field 15 / mantissa 7 = NaN): known codes."""
    assert o.e4m3_decode(0x00) == 0.0
    assert o.e4m3_decode(0x01) == 2.0 ** -9          # smallest subnormal
    assert o.e4m3_decode(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert o.e4m3_decode(0x08) == 2.0 ** -6          # smallest normal
    assert o.e4m3_decode(0x38) == 1.0
    assert o.e4m3_decode(0x3C) == 1.5
    assert o.e4m3_decode(0x40) == 2.0
    assert o.e4m3_decode(0x7E) == 448.0              # largest finite
    assert np.isnan(o.e4m3_decode(0x7F)) and np.isnan(o.e4m3_decode(0xFF))
    assert o.e4m3_decode(0xFE) == -448.0 and o.e4m3_decode(0xB8) == -1.0
    finite = [o.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(finite, finite[1:]))  # strictly increasing magnitudes
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert o.e4m3_encode(o.e4m3_decode(c)) == (c if c != 0x80 else 0x80)


def pin_e4m3_encoder_matches_definition(o):
    """The direct encoder equals the definition form (nearest finite code,
    ties to the even code, saturation at 448) on every code, every midpoint
    between neighbours (the ties), both signs, and random values."""
    finite = [o.e4m3_decode(c) for c in range(0x7F)]
    probes = list(finite)
    probes += [(a + b) / 2 for a, b in zip(finite, finite[1:])]
    probes += [448.0, 460.0, 464.0, 500.0, 1e6, 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11]
    rng = _rng(14)
    probes += rng.uniform(0, 480, 2000).tolist() + (2.0 ** rng.uniform(-12, 9, 2000)).tolist()
    for v in probes:
        for sv in (v, -v):
            assert o.e4m3_encode(sv) == o.e4m3_encode(sv, scan=True), sv
    # the tie between 1.0 (0x38) and 1.125 (0x39) goes to the even code
    assert o.e4m3_encode(1.0625) == 0x38 and o.e4m3_encode(1.1875) == 0x3A


def pin_quantize_rows_hand_worked(o):
    """Row [3.5, -7, 0, 1]: amax 7, scale 7/448 = 2^-6, 448/amax = 64;
    v * 64 = [224, -448, 0, 64], codes 0x76, 0xFE, 0x00, 0x68. A row of zeros
    has scale 0. Row [1.84375]: 448/1.84375 rounds to fp32 242.98305, and
    1.84375 times that rounds to 448.00000 in fp32: code 0x7E."""
    q, sc = o.quantize_rows_e4m3(np.array([[3.5, -7.0, 0.0, 1.0], [0.0, 0.0, 0.0, 0.0]],
                                          np.float32))
    assert sc.tolist() == [2.0 ** -6, 0.0]
    assert q[0].tolist() == [0x76, 0xFE, 0x00, 0x68] and q[1].tolist() == [0, 0, 0, 0]
    q2, _ = o.quantize_rows_e4m3(np.array([[1.84375]], np.float32))
    assert q2.tolist() == [[0x7E]]


def pin_fp8_layer_hand_worked(o):
    """One expert, d = 1, d_ff = 2, worked by hand. Every weight row and x
    quantize back to themselves except W_u row 1 (1.84375 -> 448 * fp32(
    1.84375/448) = 1.84375006): g = 1.75 * [56, 28] = [98, 49], SiLU leaves
    both unchanged in fp64, u = 1.75 * [1.75, 1.84375006], h = [300.125,
    158.10157] -> bf16 [300, 158]. The H row: scale s = fp32(300/448) =
    0.66964287, 158/s = 235.94 rounds to the E4M3 value 240, so H becomes
    [448 s, 240 s] = [300.0000038, 160.7142878]. W_d = [[1, 1]] quantizes to
    448 * fp32(1/448) = 1.0000000447 each: y = 460.7143122 (458.0000205
    without the H quantization)."""
    x = np.array([[1.75]], np.float32)
    Wr = np.array([[1.0]], np.float32)
    wg = np.array([[[56.0], [28.0]]], np.float32)
    wu = np.array([[[1.75], [1.84375]]], np.float32)
    wd = np.array([[[1.0, 1.0]]], np.float32)
    out = o.layer(x, Wr, wg, wu, wd, 1, fp8=True)
    assert abs(out["y"][0, 0] - 460.714312168105) < 1e-9, out["y"]


def pin_fp8_weight_row_scaling_is_exact(o):
    """Scaling one output row of W_d by 2^j leaves its codes unchanged and
    multiplies its scale (so that output column) by exactly 2^j, and no other
    column changes."""
    rng = _rng(15)
    T, d, dff, N, k = 5, 16, 12, 3, 2
    x = rng.normal(0, 1, (T, d)).astype(np.float32)
    Wr = rng.normal(0, 1, (N, d)).astype(np.float32)
    wg = rng.normal(0, 0.3, (N, dff, d)).astype(np.float32)
    wu = rng.normal(0, 0.3, (N, dff, d)).astype(np.float32)
    wd = rng.normal(0, 0.3, (N, d, dff)).astype(np.float32)
    a = o.layer(x, Wr, wg, wu, wd, k, fp8=True)
    wd2 = wd.copy()
    wd2[:, 5, :] *= 8.0
    b = o.layer(x, Wr, wg, wu, wd2, k, fp8=True)
    assert np.array_equal(b["y"][:, 5], 8.0 * a["y"][:, 5])
    other = [c for c in range(d) if c != 5]
    assert np.array_equal(b["y"][:, other], a["y"][:, other])
    # and FP8 stays within a few E4M3 steps (2^-4 relative) of the exact layer
    ref = o.layer(x, Wr, wg, wu, wd, k)
    assert np.abs(a["y"] - ref["y"]).max() <= 0.1 * np.abs(ref["y"]).max()


# ----------------------------------------------------------------- NVFP4 ---
def pin_e2m1_fixed_points(o):
    """E2M1 from its definition (sign, 2 exponent bits with bias 1, 1
    mantissa bit, exponent field 0 = the subnormal 0.5 * m): every code's
    value as 2^(e-1) * (1 + m/2), and every code encodes back to itself."""
    want = [0.0, 0.5] + [2.0 ** (e - 1) * (1 + m / 2) for e in (1, 2, 3) for m in (0, 1)]
    assert want == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(8):
        assert o.e2m1_decode(c) == want[c]
        assert o.e2m1_decode(8 | c) == -want[c]
        assert o.e2m1_encode(want[c]) == c and o.e2m1_encode(-want[c]) == (8 | c)


def pin_e2m1_encoder_matches_definition(o):
    """The direct encoder equals the definition form (nearest code, ties to
    the even code, saturation at 6) on every value, every midpoint (the
    ties), both signs and random values; a few ties by hand."""
    vals = [o.e2m1_decode(c) for c in range(8)]
    probes = vals + [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    probes += [5.9, 6.0, 6.5, 7.0, 100.0, 1e30, 0.1, 0.26, 0.24]
    probes += _rng(21).uniform(0, 8, 3000).tolist()
    for v in probes:
        for sv in (v, -v):
            assert o.e2m1_encode(sv) == o.e2m1_encode(sv, scan=True), sv
    # ties: 0.25 -> 0 (code 0), 0.75 -> 1 (code 2), 1.25 -> 1 (code 2),
    # 1.75 -> 2 (code 4), 2.5 -> 2 (code 4), 3.5 -> 4 (code 6), 5 -> 4 (code 6)
    assert [o.e2m1_encode(v) for v in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)] == \
        [0, 2, 2, 4, 4, 6, 6]
    assert o.e2m1_encode(-0.1) == 8  # rounds to zero, keeps the sign


def pin_quantize_rows_nvfp4_hand_worked(o):
    """Two blocks of 16. amax = 6: scale = fp32(6/2688) = fp32(1/448),
    448/amax = 74.666664, 2688/amax = 448.
    Block 0 [6, -3, 1.5, 0.75, 0 ...]: 6 * 74.666664 rounds to 448 in fp32,
    block code 0x7E (448); element factor 448/448 = 1; codes 7 (6), 0xD
    (-3), 3 (1.5), 2 (0.75 ties to the even code, 1.0).
    Block 1 [0.5, 0.25, -0.125, -0.01, 0 ...]: 0.5 * 74.666664 = 37.333332,
    nearest E4M3 36 (code 0x61); factor fp32(448/36) = 12.444445; 0.5 ->
    6.22 saturates to 6 (7), 0.25 -> 3.11 -> 3 (5), -0.125 -> -1.56 -> -1.5
    (0xB), -0.01 -> -0.124 -> -0 (8)."""
    row = np.zeros((1, 32), np.float32)
    row[0, :4] = [6, -3, 1.5, 0.75]
    row[0, 16:20] = [0.5, 0.25, -0.125, -0.01]
    q, bs, sc = o.quantize_rows_nvfp4(row)
    assert sc.tolist() == [np.float32(6) / np.float32(2688)]
    assert bs.tolist() == [[0x7E, 0x61]]
    assert q[0, :4].tolist() == [7, 0xD, 3, 2] and q[0, 16:20].tolist() == [7, 5, 0xB, 8]
    assert not q[0, 4:16].any() and not q[0, 20:].any()
    q0, bs0, sc0 = o.quantize_rows_nvfp4(np.zeros((1, 16), np.float32))
    assert sc0.tolist() == [0.0] and not bs0.any() and not q0.any()


def pin_nvfp4_error_bounds(o):
    """On random rows of mixed magnitude, from the format's definition: the
    row scale is amax/2688; each block scale is the nearest E4M3 value to
    bmax / (6 * scale) (so within 2^-4 relative, or half a subnormal step);
    each element is within half an E2M1 spacing of v / (block * scale), or
    saturated at 6 when past it."""
    rng = _rng(22)
    m = rng.normal(0, 1, (40, 128)) * 2.0 ** rng.integers(-12, 12, (40, 1))
    m *= 2.0 ** rng.integers(-6, 1, (40, 8)).repeat(16, axis=1)  # blocks well below amax
    m[3, 16:32] = 0.0
    m = m.astype(np.float32)
    q, bs, sc = o.quantize_rows_nvfp4(m)
    e4 = np.array([o.e4m3_decode(c) for c in range(256)])
    e2 = np.array([o.e2m1_decode(c) for c in range(16)])
    for r in range(m.shape[0]):
        amax = np.abs(m[r]).max().astype(np.float64)
        assert abs(sc[r] - amax / 2688) <= 2.0 ** -23 * amax / 2688
        for b in range(8):
            blk = m[r, 16 * b:16 * b + 16].astype(np.float64)
            bmax = np.abs(blk).max()
            want = bmax / (6 * float(sc[r]))
            bv = e4[bs[r, b]]
            assert abs(bv - want) <= max(2.0 ** -4 * want, 2.0 ** -10) * (1 + 1e-5), (r, b)
            if bv == 0:
                assert not (q[r, 16 * b:16 * b + 16] & 7).any()
                continue
            u = np.abs(blk) / (bv * float(sc[r]))
            got = np.abs(e2[q[r, 16 * b:16 * b + 16]])
            spacing = np.where(u < 2, 0.5, np.where(u < 4, 1.0, 2.0))
            ok = (np.abs(got - u) <= spacing / 2 * (1 + 1e-5)) | ((u > 6) & (got == 6))
            assert ok.all(), (r, b)
            nz = blk != 0
            assert (np.signbit(e2[q[r, 16 * b:16 * b + 16]][nz]) == np.signbit(blk[nz])).all()


def pin_nvfp4_layer_hand_worked(o):
    """One expert, d = d_ff = 16 (one block each), x = [6, 2.5, 0 ...],
    W_g rows [0.5, 0 ...], [0, 1, 0 ...], W_u rows [1, 0 ...], [0, 1.5, 0 ...],
    W_d row 0 = [1, 1, 0 ...], all other entries 0.
    x: amax 6, block code 448, element factor fp32(448/448) = 1, so 6 -> 6
    (code 7) and 2.5 ties to 2 (code 4): x becomes [6, 2] times 448 *
    fp32(6/2688) / 1 = 1 + tiny. A weight row with one nonzero v quantizes to
    6 * 448 * fp32(v/2688) = v (1 + tiny). a = [3, 2], b = [6, 3], H =
    SiLU(a) * b = [17.14634, 5.28478] -> bf16 [17.125, 5.28125]. The H row:
    scale fp32(17.125/2688), block code 448, element factor fp32(fp32(2688 /
    17.125) / 448) = 0.35036495: 17.125 -> 6 (code 7), 5.28125 -> 1.850 -> 2
    (code 4), so H becomes [6, 2] * 448 * fp32(17.125/2688). y0 =
    22.8333334407 (without the H quantization about 22.41; with x unquantized
    a1 = 2.5 and y0 about 25.7); every other output is 0."""
    x = np.zeros((1, 16), np.float32)
    x[0, :2] = [6.0, 2.5]
    Wr = np.ones((1, 16), np.float32)
    wg = np.zeros((1, 16, 16), np.float32)
    wu = np.zeros((1, 16, 16), np.float32)
    wd = np.zeros((1, 16, 16), np.float32)
    wg[0, 0, 0], wg[0, 1, 1] = 0.5, 1.0
    wu[0, 0, 0], wu[0, 1, 1] = 1.0, 1.5
    wd[0, 0, :2] = 1.0
    out = o.layer(x, Wr, wg, wu, wd, 1, nvfp4=True)
    assert abs(out["y"][0, 0] - 22.833333440745864) < 1e-9, out["y"]
    assert not out["y"][0, 1:].any()


def pin_nvfp4_power_of_two_scaling_is_exact(o):
    """Scaling a row by 2^j leaves its codes and block codes unchanged and
    multiplies its scale by exactly 2^j; in the layer, scaling one W_d row
    scales that output column exactly and leaves the others; and NVFP4 stays
    within a loose bound of the exact layer."""
    rng = _rng(23)
    m = rng.normal(0, 1, (6, 64)).astype(np.float32)
    q, bs, sc = o.quantize_rows_nvfp4(m)
    q2, bs2, sc2 = o.quantize_rows_nvfp4(m * np.float32(2.0 ** -7))
    assert np.array_equal(q, q2) and np.array_equal(bs, bs2)
    assert np.array_equal(sc2, sc * np.float32(2.0 ** -7))
    T, d, dff, N, k = 5, 32, 16, 3, 2
    x = rng.normal(0, 1, (T, d)).astype(np.float32)
    Wr = rng.normal(0, 1, (N, d)).astype(np.float32)
    wg = rng.normal(0, 0.3, (N, dff, d)).astype(np.float32)
    wu = rng.normal(0, 0.3, (N, dff, d)).astype(np.float32)
    wd = rng.normal(0, 0.3, (N, d, dff)).astype(np.float32)
    a = o.layer(x, Wr, wg, wu, wd, k, nvfp4=True)
    wd2 = wd.copy()
    wd2[:, 5, :] *= 16.0
    b = o.layer(x, Wr, wg, wu, wd2, k, nvfp4=True)
    assert np.array_equal(b["y"][:, 5], 16.0 * a["y"][:, 5])
    other = [c for c in range(d) if c != 5]
    assert np.array_equal(b["y"][:, other], a["y"][:, other])
    ref = o.layer(x, Wr, wg, wu, wd, k)
    assert np.abs(a["y"] - ref["y"]).max() <= 0.35 * np.abs(ref["y"]).max()
    assert np.abs(a["y"] - ref["y"]).max() > 0  # and it is not the exact layer


# -------------------------------------------------------------- backward ---
def _bwd_case(seed, T=5, d=6, N=4, k=2, dff=7, S=1):
    rng = _rng(seed)
    E = N + S
    return dict(x=rng.normal(0, 1, (T, d)), w_router=rng.normal(0, 1, (N, d)),
                wg=rng.normal(0, 0.5, (E, dff, d)), wu=rng.normal(0, 0.5, (E, dff, d)),
                wd=rng.normal(0, 0.5, (E, d, dff)), dy=rng.normal(0, 1, (T, d)), k=k, n_shared=S)


def _loss(o, c, gate_mode, alpha, aux_grad, capacity=0, reroute=False, **over):
    """sum(dy * y) + aux_grad * aux from the oracle's forward (fp64 inputs),
    and the experts the pairs ran on."""
    a = dict(c, **over)
    out = o.layer(a["x"], a["w_router"], a["wg"], a["wu"], a["wd"], a["k"],
                  gate_mode=gate_mode, n_shared=a["n_shared"], capacity=capacity,
                  reroute=reroute)
    T = a["x"].shape[0]
    _, _, aux = o.balance_stats(out["counts"], out["prob_sum"], T, a["k"], alpha)
    ran = np.concatenate([out["topk_idx"], out["assign"]], axis=1)
    return float((a["dy"] * out["y"]).sum() + aux_grad * aux), ran


def _finite_differences(o, c, name, gate_mode, alpha, aux_grad, h, capacity=0, reroute=False):
    arr = c[name]
    fd = np.zeros_like(arr)
    base = _loss(o, c, gate_mode, alpha, aux_grad, capacity, reroute)[1]
    for i in np.ndindex(arr.shape):
        plus, minus = arr.copy(), arr.copy()
        plus[i] += h
        minus[i] -= h
        lp, ip = _loss(o, c, gate_mode, alpha, aux_grad, capacity, reroute, **{name: plus})
        lm, im = _loss(o, c, gate_mode, alpha, aux_grad, capacity, reroute, **{name: minus})
        assert (ip == base).all() and (im == base).all(), "a step changed the routing"
        fd[i] = (lp - lm) / (2 * h)
    return fd


_GRAD_OF = dict(x="dx", w_router="dw_router", wg="dw_gate", wu="dw_up", wd="dw_down")


def _rel(a, b):
    return float(np.abs(a - b).max() / max(1e-300, np.abs(b).max()))


def pin_backward_matches_finite_differences(o):
    """Every gradient against central differences of the forward's loss
    sum(dy * y) + aux_grad * aux, in both gate modes, with a shared expert.
    The forward rounds scores to fp32 (2^-24 relative) before the softmax,
    so the router-side differences carry ~6e-8 / h of noise; the expert
    weights see none."""
    c = _bwd_case(21)
    for mode in (0, 1):
        g = o.layer_backward(c["x"], c["w_router"], c["wg"], c["wu"], c["wd"], c["k"], c["dy"],
                             gate_mode=mode, n_shared=c["n_shared"], alpha=0.01, aux_grad=3.0)
        for name in ("x", "w_router", "wg", "wu", "wd"):
            fd = _finite_differences(o, c, name, mode, 0.01, 3.0, h=1e-3)
            tol = 1e-3 if name in ("x", "w_router") else 1e-5
            assert _rel(g[_GRAD_OF[name]], fd) < tol, (mode, name, _rel(g[_GRAD_OF[name]], fd))


def pin_backward_rerouted_matches_finite_differences(o):
    """With a capacity whose overflow is rerouted, every gradient against
    central differences of the rerouted forward's loss: a rerouted slot's
    gate weight multiplies its new expert's output, so the gradient reaches
    that expert's weights and, through the slot's gate, the router."""
    c = _bwd_case(26, T=9, N=4, k=2, S=1)
    c["w_router"][0] += 2.0 * c["x"].mean(0)  # expert 0 popular: it overflows
    out = o.layer(c["x"], c["w_router"], c["wg"], c["wu"], c["wd"], c["k"], n_shared=1,
                  capacity=3, reroute=True)
    moved = (out["assign"] != out["topk_idx"]) & (out["assign"] >= 0)
    assert moved.any()
    g = o.layer_backward(c["x"], c["w_router"], c["wg"], c["wu"], c["wd"], c["k"], c["dy"],
                         n_shared=1, capacity=3, alpha=0.01, aux_grad=2.0, reroute=True)
    for name in ("x", "w_router", "wg", "wu", "wd"):
        fd = _finite_differences(o, c, name, 0, 0.01, 2.0, h=1e-3, capacity=3, reroute=True)
        tol = 1e-3 if name in ("x", "w_router") else 1e-5
        assert _rel(g[_GRAD_OF[name]], fd) < tol, (name, _rel(g[_GRAD_OF[name]], fd))


def pin_backward_balance_term_alone(o):
    """With dy = 0 only the balance term moves the loss: dx and dW_r against
    central differences of aux alone, and every expert-weight gradient is
    exactly zero (f is held fixed, so the experts do not enter aux)."""
    c = _bwd_case(22, T=6, N=5, k=2, S=0)
    c["dy"] = np.zeros_like(c["dy"])
    g = o.layer_backward(c["x"], c["w_router"], c["wg"], c["wu"], c["wd"], c["k"], c["dy"],
                         alpha=0.01, aux_grad=50.0)
    for name in ("x", "w_router"):
        fd = _finite_differences(o, c, name, 0, 0.01, 50.0, h=1e-3)
        assert _rel(g[_GRAD_OF[name]], fd) < 1e-3, (name, _rel(g[_GRAD_OF[name]], fd))
    for key in ("dw_gate", "dw_up", "dw_down"):
        assert not g[key].any(), key


def pin_backward_collapsed_example(o):
    """Mixture of Experts and Guided Decoding, the auxiliary-loss example
    (N = 4, collapsed routing f = [1, 0, 0, 0], P = [0.7, 0.1, 0.1, 0.1]), as
    one token with d = 1: x = 1 and router weights [ln 7, 0, 0, 0] give
    p = P, and top-1 picks expert 0. With dy = 0 the score gradient is the
    balance term alone, alpha * N / T * p_i * (f_i - sum_m p_m f_m)
    = alpha * 4 * [0.7 * 0.3, -0.1 * 0.7, -0.1 * 0.7, -0.1 * 0.7]
    = alpha * [0.84, -0.28, -0.28, -0.28], which is dW_r (x = 1) and sums
    into dx = sum_e dr_e * W_r[e] = alpha * 0.84 * ln 7."""
    g0 = golden("balance_loss_n4.json")
    alpha = g0["alpha"]
    P = np.array(g0["collapsed"]["P"])
    wr = np.log(P / P[-1]).reshape(4, 1)       # [ln 7, 0, 0, 0]
    x = np.ones((1, 1))
    z = np.zeros((4, 2, 1))
    g = o.layer_backward(x, wr, z, z, np.zeros((4, 1, 2)), 1, np.zeros((1, 1)), alpha=alpha,
                         aux_grad=1.0)
    want = alpha * np.array([0.84, -0.28, -0.28, -0.28])
    assert np.allclose(g["dw_router"][:, 0], want, rtol=1e-6, atol=0), g["dw_router"]
    assert abs(g["dx"][0, 0] - alpha * 0.84 * math.log(7.0)) < 1e-8, g["dx"]


def pin_backward_gate_modes_agree(o):
    """A softmax over all scores renormalised over the kept experts equals a
    softmax over the kept scores, so the two gate modes have the same
    gradient (with the balance term and a capacity cut too)."""
    c = _bwd_case(23, T=8, N=5, k=3, S=1)
    args = (c["x"], c["w_router"], c["wg"], c["wu"], c["wd"], c["k"], c["dy"])
    a = o.layer_backward(*args, gate_mode=0, n_shared=1, capacity=4, aux_grad=2.0)
    b = o.layer_backward(*args, gate_mode=1, n_shared=1, capacity=4, aux_grad=2.0)
    for key in a:
        assert _rel(a[key], b[key]) < 1e-12, key


def pin_backward_matches_autograd(o):
    """The whole layer written with torch fp64 ops and differentiated by
    autograd, with the oracle's routing (top-k sets and kept pairs) held
    fixed: softmax gates over the kept scores, SwiGLU experts
    (F.silu), a shared expert, a capacity cut, and the balance term with f
    held constant. The oracle's gates use scores rounded to fp32, so the two
    agree to ~1e-7 relative."""
    F = torch.nn.functional
    c = _bwd_case(24, T=7, d=5, N=4, k=2, dff=6, S=1)
    cap, alpha, ag = 3, 0.01, 5.0
    g = o.layer_backward(c["x"], c["w_router"], c["wg"], c["wu"], c["wd"], c["k"], c["dy"],
                         n_shared=1, capacity=cap, alpha=alpha, aux_grad=ag)
    fwd = o.layer(c["x"], c["w_router"], c["wg"], c["wu"], c["wd"], c["k"], n_shared=1,
                  capacity=cap)
    idx, keep = fwd["topk_idx"], fwd["keep"].reshape(-1, c["k"])
    T, N, k = c["x"].shape[0], c["w_router"].shape[0], c["k"]
    f = torch.tensor(np.bincount(idx.ravel(), minlength=N) / (T * k))
    t = {n: torch.tensor(c[n], requires_grad=True)
         for n in ("x", "w_router", "wg", "wu", "wd")}
    r = t["x"] @ t["w_router"].T
    p = torch.softmax(r, dim=1)

    def expert(e, xt):
        return t["wd"][e] @ (F.silu(t["wg"][e] @ xt) * (t["wu"][e] @ xt))

    ys = []
    for tok in range(T):
        kept = torch.tensor(idx[tok].tolist())
        gates = torch.softmax(r[tok, kept], dim=0)
        y = expert(N, t["x"][tok])
        for s in range(k):
            if keep[tok, s]:
                y = y + gates[s] * expert(int(idx[tok, s]), t["x"][tok])
        ys.append(y)
    aux = alpha * N * (f * p.mean(dim=0)).sum()
    loss = (torch.stack(ys) * torch.tensor(c["dy"])).sum() + ag * aux
    loss.backward()
    for n in t:
        assert _rel(g[_GRAD_OF[n]], t[n].grad.numpy()) < 1e-6, (n, _rel(g[_GRAD_OF[n]], t[n].grad.numpy()))


def pin_backward_samples_match_full(o):
    """The sampled gradients (dx rows; rows of dW_g, dW_u and columns of
    dW_d) equal the same entries of the full backward, shared expert and
    capacity cut included."""
    c = _bwd_case(25, T=9, d=6, N=4, k=2, dff=5, S=1)
    args = (c["x"], c["w_router"], c["wg"], c["wu"], c["wd"], c["k"], c["dy"])
    kw = dict(n_shared=1, capacity=4, aux_grad=2.0, gate_mode=1)
    full = o.layer_backward(*args, **kw)
    cols = [(0, 1), (3, 4), (4, 0), (2, 2)]
    experts = {e: (c["wg"][e], c["wu"][e], c["wd"][e]) for e in range(5)}
    smp = o.backward_samples(c["x"], c["w_router"], experts, 4, c["k"], c["dy"], tokens=[0, 4, 8],
                             columns=cols, **kw)
    assert _rel(smp["dx_rows"], full["dx"][[0, 4, 8]]) < 1e-12
    for n, (e, j) in enumerate(cols):
        assert _rel(smp["dw_gate_rows"][n], full["dw_gate"][e, j]) < 1e-12
        assert _rel(smp["dw_up_rows"][n], full["dw_up"][e, j]) < 1e-12
        assert _rel(smp["dw_down_cols"][n], full["dw_down"][e, :, j]) < 1e-12


def pin_backward_balance_entry_matches_full(o):
    """The dy = 0 entry point equals the full backward with dy = 0."""
    c = _bwd_case(26, T=7, N=5, k=2, S=0)
    dy0 = np.zeros_like(c["dy"])
    full = o.layer_backward(c["x"], c["w_router"], c["wg"], c["wu"], c["wd"], c["k"], dy0,
                            gate_mode=1, aux_grad=4.0)
    dx, dwr = o.balance_backward(c["x"], c["w_router"], c["k"], gate_mode=1, aux_grad=4.0)
    assert _rel(dx, full["dx"]) < 1e-12 and _rel(dwr, full["dw_router"]) < 1e-12


def pin_balance_stats_sum_to_one(o):
    rng = _rng(11)
    T, N, k = 64, 8, 2
    r = rng.normal(0, 1, (T, N)).astype(np.float32)
    _, _, counts, ps = o.route(r, k)
    f, P, aux = o.balance_stats(counts, ps, T, k, 0.01)
    assert abs(f.sum() - 1) < 1e-12 and abs(P.sum() - 1) < 1e-12
    assert abs(aux - 0.01 * N * (f * P).sum()) < 1e-15
    assert counts.sum() == T * k


ALL_PINS = [v for k_, v in sorted(globals().items()) if k_.startswith("pin_")]
