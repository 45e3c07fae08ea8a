"""Seeded synthetic inputs for the attention forward.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  The CUDA path and the fp64 oracle both take their
inputs from here, so the same stored bits reach both sides.

Recipe (every config): ``numpy.random.default_rng(seed)`` (PCG64), seed 0
unless stated.  Draw order: q ~ N(0,1) [B,h,Tq,dk], k ~ N(0,1) [B,hkv,Tk,dk],
v ~ N(0,1) [B,hkv,Tk,dv] as float32, then q and k are multiplied by the
config's norm factor, then the per-head parameters are drawn in the order
b, eps, tau.  bf16 configs are rounded to bf16 (round-to-nearest-even) by
torch.  The per-head scalars follow the parametrisations on the pages:
b and eps pass through a softplus (raw 0 gives log 2, "Softmax-Free Attention
in JAX/Flax NNX", section "One module, two compatibility functions");
tau = softplus(raw) + 1 ("s^tau" page, core formula).

The five workloads mirror the shapes and norm regimes of the pages'
experiments (char-level GPT attention, a mid-size causal layer, a GQA
long-context layer, a long cross-attention); the pages' datasets and trained
weights are not used.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

LN2 = math.log(2.0)


def _softplus64(x):
    x = np.asarray(x, dtype=np.float64)
    return np.logaddexp(0.0, x)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    h: int
    hkv: int
    Tq: int
    Tk: int
    dk: int
    dv: int
    dtype: str  # "bf16" | "f32"
    causal: bool
    qk_factor: float = 1.0
    # per-head parameter recipes
    yat_param: str = "ln2"          # "ln2" | "softplus_uniform" | "softplus_normal_0.5"
    stau_eps: float = 1e-6
    tau_param: str = "softplus_normal_plus1"  # or a constant given by tau_const
    tau_const: float | None = None
    seed: int = 0
    description: str = ""

    @property
    def scale(self) -> float:
        """Score scale for softmax and s^tau (Yat uses the raw q.k)."""
        return 1.0 / math.sqrt(self.dk)

    def flops(self) -> float:
        """2*B*h*Tq*Tk*(dk+dv), halved when causal (the metric's own count)."""
        f = 2.0 * self.B * self.h * self.Tq * self.Tk * (self.dk + self.dv)
        return f / 2.0 if self.causal else f

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "cfg1_f32": Workload(
        "cfg1_f32", B=1, h=4, hkv=4, Tq=256, Tk=256, dk=32, dv=32, dtype="f32", causal=True,
        yat_param="ln2",
        description="Yat/softmax causal fp32, B=1 h=4 T=256 d=32, b=eps=ln2"),
    "cfg2_s1": Workload(
        "cfg2_s1", B=32, h=4, hkv=4, Tq=256, Tk=256, dk=64, dv=64, dtype="bf16", causal=True,
        qk_factor=1.0, yat_param="softplus_uniform",
        description="char-level GPT shapes, q/k x1, b,eps=softplus(U(-1,1))"),
    "cfg2_s4": Workload(
        "cfg2_s4", B=32, h=4, hkv=4, Tq=256, Tk=256, dk=64, dv=64, dtype="bf16", causal=True,
        qk_factor=4.0, yat_param="softplus_uniform",
        description="char-level GPT shapes, q/k x4"),
    "cfg2_s16": Workload(
        "cfg2_s16", B=32, h=4, hkv=4, Tq=256, Tk=256, dk=64, dv=64, dtype="bf16", causal=True,
        qk_factor=16.0, yat_param="softplus_uniform",
        description="char-level GPT shapes, q/k x16 (large kappa)"),
    "cfg3": Workload(
        "cfg3", B=16, h=16, hkv=16, Tq=4096, Tk=4096, dk=128, dv=128, dtype="bf16", causal=True,
        yat_param="softplus_normal_0.5",
        description="mid-size causal B=16 h=16 T=4096 d=128, b,eps=softplus(N(0,0.5))"),
    "cfg4_gqa": Workload(
        "cfg4_gqa", B=4, h=16, hkv=8, Tq=8192, Tk=8192, dk=128, dv=128, dtype="bf16", causal=True,
        yat_param="softplus_normal_0.5", stau_eps=1e-6,
        description="s^tau causal GQA 16/8, T=8192, d=128, tau=softplus(N(0,1))+1, eps=1e-6"),
    "cfg5_cross": Workload(
        "cfg5_cross", B=1, h=32, hkv=32, Tq=2048, Tk=32768, dk=128, dv=64, dtype="bf16", causal=False,
        qk_factor=8.0, yat_param="ln2", stau_eps=1e-6, tau_param="const", tau_const=6.0,
        description="non-causal cross-attention Tq=2048 Tk=32768 dk=128 dv=64, q/k x8"),
}


def generate(w: Workload, device=None):
    """Draw the inputs of workload ``w``.

    Returns a dict with torch tensors q, k, v (dtype bf16 or float32, on
    ``device`` or the CPU) and float32 numpy arrays ``yat_b``, ``yat_eps``,
    ``stau_eps``, ``tau`` (one value per query head), plus ``scale`` and
    ``causal``.
    """
    import torch

    rng = np.random.default_rng(w.seed)
    q = rng.standard_normal((w.B, w.h, w.Tq, w.dk), dtype=np.float32)
    k = rng.standard_normal((w.B, w.hkv, w.Tk, w.dk), dtype=np.float32)
    v = rng.standard_normal((w.B, w.hkv, w.Tk, w.dv), dtype=np.float32)
    if w.qk_factor != 1.0:
        q *= np.float32(w.qk_factor)
        k *= np.float32(w.qk_factor)

    if w.yat_param == "ln2":
        yb = np.full(w.h, LN2)
        ye = np.full(w.h, LN2)
    elif w.yat_param == "softplus_uniform":
        yb = _softplus64(rng.uniform(-1.0, 1.0, w.h))
        ye = _softplus64(rng.uniform(-1.0, 1.0, w.h))
    elif w.yat_param == "softplus_normal_0.5":
        yb = _softplus64(rng.normal(0.0, 0.5, w.h))
        ye = _softplus64(rng.normal(0.0, 0.5, w.h))
    else:
        raise ValueError(w.yat_param)
    if w.tau_param == "const":
        tau = np.full(w.h, w.tau_const)
    else:
        tau = _softplus64(rng.normal(0.0, 1.0, w.h)) + 1.0

    tdtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    out = {
        "q": torch.from_numpy(q).to(tdtype),
        "k": torch.from_numpy(k).to(tdtype),
        "v": torch.from_numpy(v).to(tdtype),
        "yat_b": yb.astype(np.float32),
        "yat_eps": ye.astype(np.float32),
        "stau_eps": np.full(w.h, w.stau_eps, dtype=np.float32),
        "tau": tau.astype(np.float32),
        "scale": w.scale,
        "causal": w.causal,
    }
    if device is not None:
        for key in ("q", "k", "v"):
            out[key] = out[key].to(device)
    return out


def grad_output(w: Workload, device=None):
    """dL/d out for the backward: standard normal [B, h, Tq, dv] in the
    workload's dtype, from a generator of its own (seed + 7919) so that the
    forward inputs stay those of ``generate``."""
    import torch

    rng = np.random.default_rng(w.seed + 7919)
    d = rng.standard_normal((w.B, w.h, w.Tq, w.dv), dtype=np.float32)
    t = torch.from_numpy(d).to(torch.bfloat16 if w.dtype == "bf16" else torch.float32)
    return t if device is None else t.to(device)


def sample_rows(w: Workload, n_random: int = 64, seed: int = 1):
    """Deterministic subset of flat query-row indices into [B, h, Tq].

    Every (batch, head) pair contributes rows {0, 1, 127, 128, Tq/2, Tq-1}
    (those that exist), and ``n_random`` further rows are drawn uniformly over
    the whole problem with a separate seeded generator.
    """
    fixed = sorted({r for r in (0, 1, 127, 128, w.Tq // 2, w.Tq - 1) if 0 <= r < w.Tq})
    rows = []
    for bh in range(w.B * w.h):
        rows.extend(bh * w.Tq + r for r in fixed)
    rng = np.random.default_rng(seed)
    rows.extend(rng.integers(0, w.B * w.h * w.Tq, n_random).tolist())
    return np.unique(np.asarray(rows, dtype=np.int64))
