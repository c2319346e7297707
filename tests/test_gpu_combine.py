"""K5 parity: moe_combine, the gate-weighted sum back into token order,
through the C ABI.

* The pages' three-expert gated sum (gates [0.5, 0.3, 0.2], expert outputs
  [2, 4, 0] -> 2.2), fed to the kernel as a token with three slots and
  every element of the d = 8 rows equal to the printed scalar.
* Seeded random cases against the oracle's gated sum, token by token: fp32
  within fp32 rounding; bf16 output within one bf16 rounding of the fp64
  value (plus fp32 accumulation). With and without gate weights, with
  shared experts, and with an out-of-range position (contributes zero).
"""
import json
import os

import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_gated_sum_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "gated_sum_3_experts.json")))
    k, d = 3, 8
    cfg = moe.config(T=1, d_model=d, n_experts=3, top_k=k, d_ff=8, dtype=moe.MOE_F32)
    y_perm = torch.tensor([[v] * d for v in g["expert_outputs"]], dtype=torch.float32,
                          device="cuda")
    inv_pos = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    w = torch.tensor([g["gates"]], dtype=torch.float32, device="cuda")
    y = torch.full((1, d), float("nan"), device="cuda")
    moe.moe_combine(cfg, y_perm, inv_pos, w, y)
    torch.cuda.synchronize()
    assert np.abs(y.cpu().numpy() - g["output"]).max() <= 1e-6


CASES = [
    # T, d, k, n_shared, dtype, weighted
    (1, 8, 1, 0, moe.MOE_F32, True),
    (37, 64, 2, 0, moe.MOE_F32, True),
    (200, 4096, 2, 0, moe.MOE_BF16, True),
    (129, 7168, 8, 1, moe.MOE_BF16, False),
    (64, 256, 8, 4, moe.MOE_BF16, True),      # the most terms a token can have
    (50, 520, 3, 2, moe.MOE_F32, True),
]


@pytest.mark.parametrize("T,d,k,s,dtype,weighted", CASES)
def test_combine_matches_oracle(oracle, T, d, k, s, dtype, weighted):
    rng = np.random.default_rng(T * 7 + d)
    P = T * k
    rows = P + s * T
    y_perm64 = rng.normal(0, 1, (rows, d))
    tdt = torch.bfloat16 if dtype == moe.MOE_BF16 else torch.float32
    y_perm = torch.from_numpy(y_perm64).to(tdt)
    stored = y_perm.double().numpy()                   # the values the kernel reads
    inv = rng.permutation(P).astype(np.int32)
    if P > 3:
        inv[3] = P + 5                                  # out of range: contributes zero
    w = rng.uniform(0, 1, (T, k)).astype(np.float32) if weighted else None
    cfg = moe.config(T=T, d_model=d, n_experts=max(k, 8), top_k=k, d_ff=8, n_shared=s,
                     dtype=dtype)
    y = torch.full((T, d), float("nan"), dtype=tdt, device="cuda")
    moe.moe_combine(cfg, y_perm.cuda(), torch.from_numpy(inv).cuda(),
                    None if w is None else torch.from_numpy(w).cuda(), y)
    torch.cuda.synchronize()
    got = y.double().cpu().numpy()
    ref = np.empty((T, d))
    for t in range(T):
        G, E = [], []
        for j in range(k):
            pos = inv[t * k + j]
            if 0 <= pos < P:
                G.append(1.0 if w is None else float(w[t, j]))
                E.append(stored[pos])
        for q in range(s):
            G.append(1.0)
            E.append(stored[P + q * T + t])
        ref[t] = oracle.gated_sum(np.array(G), np.array(E)) if G else 0.0
    err = np.abs(got - ref)
    if dtype == moe.MOE_F32:
        assert (err <= 1e-5 * (1 + np.abs(ref))).all()
    else:  # one bf16 rounding of the output (2^-8 relative) plus fp32 accumulation
        assert (err <= 2.0 ** -8 * np.abs(ref) + 1e-5).all()
