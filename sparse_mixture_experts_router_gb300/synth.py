"""Seeded synthetic inputs of the MoE layer workloads.

Random draws only: this module holds none of the layer's arithmetic. The
same tensors feed both the CUDA library and the CPU oracle in the tests and
the benchmark. Distributions: tokens x ~ N(0, 1); router and expert weights
~ N(0, 0.02^2) (standard deviation 0.02); a selection bias ~ U(-0.1, 0.1)
where the workload has one; all rounded to the workload's storage type.

The Zipf workload's per-expert score offset, -s * ln(e + 1) with s = 1.2,
is the log of a Zipf(s) weight ~ (e + 1)^-s: added to a score it multiplies
that expert's odds by its Zipf weight, making the low-numbered experts hot.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    n_shared: int = 0
    dtype: str = "bf16"            # "bf16" or "f32"
    gate_mode: int = 0             # 0: softmax over kept, 1: all-softmax + renorm
    sel_bias: bool = False         # per-expert selection bias ~ U(-0.1, 0.1)
    zipf_s: float = 0.0            # > 0: per-expert Zipf score offset
    seed: int = 0
    capacity_factor: float = 0.0   # > 0: expert capacity ceil(factor * T * k / N)
    tiles: int = 0                 # grouped-GEMM tiling (moe_config.tiles); 0 = the library's
    gather: int = 0                # where the row gather runs (moe_config.gather); 0 = the library's
    overflow: int = 0              # pairs over the capacity (moe_config.overflow): 0 dropped, 1 rerouted

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def pairs(self) -> int:
        return self.T * self.top_k


# The layer shapes the library is measured and checked on.
TINY = Workload("tiny_fp32", T=64, d_model=64, n_experts=4, top_k=2, d_ff=128, dtype="f32", seed=0)
MIXTRAL_PREFILL = Workload("mixtral_8x7b_prefill", T=4096, d_model=4096, n_experts=8, top_k=2,
                           d_ff=14336, seed=1)
MIXTRAL_DECODE = [MIXTRAL_PREFILL.replace(name=f"mixtral_8x7b_decode_T{t}", T=t, seed=2)
                  for t in (1, 8, 32, 64)]
DEEPSEEK_V3 = Workload("deepseek_v3_moe", T=8192, d_model=7168, n_experts=256, top_k=8, d_ff=2048,
                       n_shared=1, gate_mode=1, sel_bias=True, seed=3)
ZIPF = Workload("zipf_imbalanced", T=16384, d_model=4096, n_experts=128, top_k=8, d_ff=1536,
                zipf_s=1.2, seed=4)
# The imbalanced layer with an expert capacity of 1.25x the even share: the
# hot experts keep their first 1280 pairs and drop the rest.
ZIPF_CAPACITY = ZIPF.replace(name="zipf_imbalanced_capacity_1.25", capacity_factor=1.25)
# The same cap with the overflow rerouted to each token's next-best expert
# with room instead of dropped.
ZIPF_REROUTE = ZIPF_CAPACITY.replace(name="zipf_imbalanced_capacity_1.25_reroute", overflow=1)
ALL = [TINY, MIXTRAL_PREFILL, *MIXTRAL_DECODE, DEEPSEEK_V3, ZIPF, ZIPF_CAPACITY, ZIPF_REROUTE]


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_into(out: torch.Tensor, std: float, g: torch.Generator):
    """Fill `out` with N(0, std^2) draws, one leading slice at a time (so
    that a multi-GB bf16 weight never needs an fp32 copy of itself)."""
    if out.numel() == 0:
        return out
    flat = out.view(out.shape[0], -1) if out.dim() > 1 else out.view(1, -1)
    for i in range(flat.shape[0]):
        v = torch.randn(flat.shape[1], generator=g, device=out.device, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        flat[i].copy_(v)
    return out


def make_inputs(w: Workload, device="cuda", seed: int | None = None) -> dict:
    """Tensors of one workload: x [T, d], w_router [N, d], w_gate / w_up
    [N+s, d_ff, d], w_down [N+s, d, d_ff] in the workload dtype, and the fp32
    biases sel_bias [N] / logit_bias [N] (None when the workload has none)."""
    seed = w.seed if seed is None else seed
    g = _gen(device, seed)
    dt = w.torch_dtype
    E = w.n_experts + w.n_shared
    x = _normal_into(torch.empty(w.T, w.d_model, dtype=dt, device=device), 1.0, g)
    w_router = _normal_into(torch.empty(w.n_experts, w.d_model, dtype=dt, device=device), 0.02, g)
    w_gate = _normal_into(torch.empty(E, w.d_ff, w.d_model, dtype=dt, device=device), 0.02, g)
    w_up = _normal_into(torch.empty(E, w.d_ff, w.d_model, dtype=dt, device=device), 0.02, g)
    w_down = _normal_into(torch.empty(E, w.d_model, w.d_ff, dtype=dt, device=device), 0.02, g)
    sel_bias = None
    if w.sel_bias:
        sel_bias = (torch.rand(w.n_experts, generator=g, device=device, dtype=torch.float32) * 0.2 - 0.1)
    logit_bias = None
    if w.zipf_s > 0:
        logit_bias = torch.tensor([-w.zipf_s * math.log(e + 1) for e in range(w.n_experts)],
                                  dtype=torch.float32, device=device)
    return dict(x=x, w_router=w_router, w_gate=w_gate, w_up=w_up, w_down=w_down,
                sel_bias=sel_bias, logit_bias=logit_bias)


def make_grad_output(w: Workload, device="cuda", seed: int | None = None) -> torch.Tensor:
    """dL/dy [T, d] for the backward: N(0, 1) in the workload dtype, drawn
    from a generator of its own (the workload seed + 1000), so the forward
    inputs are the same with or without it."""
    g = _gen(device, (w.seed if seed is None else seed) + 1000)
    return _normal_into(torch.empty(w.T, w.d_model, dtype=w.torch_dtype, device=device), 1.0, g)


def redraw_rows(x: torch.Tensor, rows, seed: int, round_: int):
    """Replace the listed token rows with fresh N(0, 1) draws (a separate
    stream per round), in place."""
    if len(rows) == 0:
        return x
    g = _gen(x.device, 1_000_003 * (seed + 1) + round_)
    idx = torch.as_tensor(list(rows), dtype=torch.long, device=x.device)
    fresh = torch.randn(len(rows), x.shape[1], generator=g, device=x.device, dtype=torch.float32)
    x[idx] = fresh.to(x.dtype)
    return x


def random_logits(T: int, N: int, seed: int, ties: bool = True, device="cpu") -> torch.Tensor:
    """fp32 router scores for routing-only checks. With ties=True about a
    quarter of the scores are snapped to a coarse grid of 0.25 so equal
    scores (and equal selection keys) occur often."""
    g = _gen(device, seed)
    r = torch.randn(T, N, generator=g, device=device, dtype=torch.float32) * 1.5
    if ties:
        snap = torch.rand(T, N, generator=g, device=device) < 0.25
        r = torch.where(snap, torch.round(r * 4) / 4, r)
    return r


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a bf16 tensor as a numpy array (what the
    oracle reads), or the numpy array itself for fp32."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
