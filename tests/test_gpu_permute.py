"""K2 parity: expert offsets, the pair order, its inverse and the gathered
rows are unique, so they must equal the oracle's bit for bit."""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_router_gb300 as moe

pytestmark = pytest.mark.gpu


def random_idx(T, N, k, seed, skew=0.0):
    """Each token picks k distinct experts; skew > 0 favours low indices."""
    rng = np.random.default_rng(seed)
    p = np.arange(1, N + 1, dtype=np.float64) ** (-skew)
    p /= p.sum()
    return np.stack([rng.choice(N, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32) \
        if T else np.zeros((0, k), np.int32)


def run_permute(cfg, x, idx):  # noqa: D103
    T, k, d = cfg.T, cfg.top_k, cfg.d_model
    P = T * k
    dev = "cuda"
    off = torch.full((cfg.n_experts + 1,), -9, dtype=torch.int32, device=dev)
    sp = torch.full((max(P, 1),), -9, dtype=torch.int32, device=dev)
    inv = torch.full((max(P, 1),), -9, dtype=torch.int32, device=dev)
    xp = torch.zeros((max(P, 1), d), dtype=x.dtype, device=dev)
    ws = moe.workspace(cfg, "permute", dev)
    moe.moe_permute(cfg, x, idx, off, sp, inv, xp, ws)
    return off, sp[:P], inv[:P], xp[:P], moe.moe_stream_status(ws)


CASES = [
    # T, N, k, d, dtype, skew
    (1, 4, 2, 64, moe.MOE_BF16, 0.0),
    (3, 8, 2, 8, moe.MOE_F32, 0.0),
    (1000, 8, 2, 256, moe.MOE_BF16, 0.0),
    (5000, 256, 8, 72, moe.MOE_BF16, 0.0),     # 20 chunks of 2048 pairs
    (3000, 128, 8, 64, moe.MOE_BF16, 1.2),     # Zipf-skewed
    (2048, 4, 4, 16, moe.MOE_F32, 0.0),        # k = N
    (777, 33, 3, 40, moe.MOE_BF16, 2.0),
    (9000, 64, 8, 16, moe.MOE_BF16, 0.5),     # 72000 pairs: the chunked four-launch path
]


@pytest.mark.parametrize("T,N,k,d,dtype,skew", CASES)
def test_permute_is_bit_exact(oracle, T, N, k, d, dtype, skew):
    idx = random_idx(T, N, k, seed=T + N, skew=skew)
    tdt = torch.bfloat16 if dtype == moe.MOE_BF16 else torch.float32
    g = torch.Generator(device="cuda").manual_seed(T)
    x = torch.randn(T, d, generator=g, device="cuda").to(tdt)
    cfg = moe.config(T=T, d_model=d, n_experts=N, top_k=k, d_ff=8, dtype=dtype)
    off, sp, inv, xp, st = run_permute(cfg, x, torch.from_numpy(idx).cuda())
    assert st == 0
    r_off, r_sp, r_inv = oracle.permute(idx, N)
    assert np.array_equal(off.cpu().numpy(), r_off)
    assert np.array_equal(sp.cpu().numpy(), r_sp)
    assert np.array_equal(inv.cpu().numpy(), r_inv)
    # gathered rows, byte for byte
    ref_rows = x[torch.from_numpy(r_sp // k).long().cuda()]
    assert torch.equal(xp.view(torch.int16) if tdt == torch.bfloat16 else xp.view(torch.int32),
                       ref_rows.view(torch.int16) if tdt == torch.bfloat16 else ref_rows.view(torch.int32))


CAPACITY_CASES = [
    # T, N, k, capacity, skew: one case per launch shape (one block, expert
    # groups, chunks); the skew makes hot experts overflow
    (100, 8, 2, 10, 1.5),
    (3000, 128, 8, 150, 1.2),
    (9000, 64, 8, 900, 0.8),
    (500, 4, 2, 1, 0.0),       # one row per expert
]


@pytest.mark.parametrize("T,N,k,cap,skew", CAPACITY_CASES)
def test_permute_with_capacity_is_bit_exact(oracle, T, N, k, cap, skew):
    """Each expert keeps its first `cap` pairs in ascending token order; the
    rest get inv_pos = -1 and no row."""
    idx = random_idx(T, N, k, seed=T + N + cap, skew=skew)
    x = torch.randn(T, 32, device="cuda").to(torch.bfloat16)
    cfg = moe.config(T=T, d_model=32, n_experts=N, top_k=k, d_ff=8, capacity=cap)
    off, sp, inv, xp, st = run_permute(cfg, x, torch.from_numpy(idx).cuda())
    assert st == 0
    r_off, r_sp, r_inv = oracle.permute(idx, N, capacity=cap)
    assert np.array_equal(off.cpu().numpy(), r_off)
    rows = int(r_off[-1])
    assert rows < T * k  # something was dropped
    assert np.array_equal(sp.cpu().numpy()[:rows], r_sp)
    assert np.array_equal(inv.cpu().numpy(), r_inv)
    assert torch.equal(xp[:rows].view(torch.int16),
                       x[torch.from_numpy(r_sp // k).long().cuda()].view(torch.int16))


def test_all_tokens_to_one_expert(oracle):
    T, N, k, d = 4096, 8, 1, 64
    idx = np.full((T, 1), 3, np.int32)
    x = torch.randn(T, d, device="cuda").to(torch.bfloat16)
    cfg = moe.config(T=T, d_model=d, n_experts=N, top_k=k, d_ff=8)
    off, sp, inv, xp, st = run_permute(cfg, x, torch.from_numpy(idx).cuda())
    assert st == 0
    assert off.cpu().tolist() == [0, 0, 0, 0, T, T, T, T, T]
    assert np.array_equal(sp.cpu().numpy(), np.arange(T))
    assert torch.equal(xp, x)


def test_empty_batch():
    cfg = moe.config(T=0, d_model=64, n_experts=5, top_k=2, d_ff=8)
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    off, sp, inv, xp, st = run_permute(cfg, x, torch.empty(0, 2, dtype=torch.int32, device="cuda"))
    assert st == 0 and off.cpu().tolist() == [0] * 6


@pytest.mark.parametrize("T,k", [(100, 2), (1500, 2), (9000, 8)])
def test_out_of_range_expert_is_reported(T, k):
    """An index outside [0, N) is caught by the kernel's own bounds check
    (single-block, expert-group and chunked paths): the status word reports
    it and nothing is written out of bounds."""
    N, d = 8, 32
    idx = random_idx(T, N, k, seed=1)
    idx[17, 1] = N + 3
    idx[40, 0] = -2
    x = torch.randn(T, d, device="cuda").to(torch.bfloat16)
    cfg = moe.config(T=T, d_model=d, n_experts=N, top_k=k, d_ff=8)
    off, sp, inv, xp, st = run_permute(cfg, x, torch.from_numpy(idx).cuda())
    assert st == moe.MOE_ERR_DEVICE_CHECK
    assert off.cpu()[-1].item() == T * k - 2
