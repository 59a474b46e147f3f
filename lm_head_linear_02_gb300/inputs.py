"""Seeded synthetic inputs for fused linear cross-entropy (FLCE).

This module holds input preparation only: random draws, the fp32 -> bf16 rounding of those
draws, and target sampling. It contains none of the method's arithmetic, so that the float64
oracle and the CUDA path can be fed the same bytes without sharing any code that computes the
loss or its gradients.

Workloads are the LM-head shapes of the pages' benchmarks:

* "Fused linear + cross-entropy" (KernelIndex operation page), "Current records": vocab 128256,
  hidden 4096, tokens in {4096, 8192, 16384, 32768}, bf16.
* "feat(FLCE): add helion version of fused linear cross entropy" (Liger-Kernel PR #928), the
  failing-test list: (B, T, H, V) = (2, 1024, 4096, 32000) and (3, 423, 1000, 10000); and its
  benchmark tables for a Qwen3 head (H=4096, V=151936, BT=32768), a Gemma3 head (H=2304,
  V=262208, BT=8192) and an fp32 head (H=4096, V=32000, BT=32768).

The pages ship no datasets; these synthetic draws stand in for the benchmark scripts' random
activations and weights: x ~ N(0, 1), weight ~ N(0, 0.02^2), and targets either uniform over the
vocabulary or Zipf-distributed with exponent 1.1 (rank 1 = id 0).

Two further recipes put the softmax where a trained LM head has it, which the near-uniform
softmax of weight ~ N(0, 0.02^2) never reaches (the Helion PR #1268 discussion upcasts bf16
logits to fp32 for this regime):

* a wide logit spread: weight ~ N(0, w_std^2) with a larger w_std (0.3 at hidden 1024 gives
  logits of standard deviation ~10, so a few columns of each row carry most of the softmax);
* confident predictions: after the draws, weight[target[t]] += margin * x[t] / |x[t]|^2 for
  every token (x already rounded to the input dtype), so that the target logit of each token
  stands `margin` above its drawn value and its probability approaches 1 (loss near 0).

Every array comes from ``numpy.random.Generator(PCG64)`` seeded with ``1000 + index`` of the
workload, one spawned child stream per tensor (x, weight, target). PCG64 is platform independent,
so x86-64 and aarch64 hosts produce identical bytes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "FlceInputs",
    "make_inputs",
    "bf16_round_bits",
    "bf16_bits_to_f32",
    "zipf_targets",
]


@dataclass(frozen=True)
class Workload:
    """One synthetic LM-head workload: tokens T, hidden H, vocab V and its draw recipe."""

    name: str
    index: int               # seed = 1000 + index
    T: int
    H: int
    V: int
    dtype: str               # "f32" or "bf16": the type the inputs are stored and computed in
    target_dist: str         # "uniform" or "zipf"
    reductions: tuple = ("mean",)
    x_std: float = 1.0
    w_std: float = 0.02
    zipf_s: float = 1.1
    confident_margin: float = 0.0  # > 0: raise each token's target logit by this much
    note: str = field(default="", compare=False)

    @property
    def seed(self) -> int:
        return 1000 + self.index


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 1, 128, 256, 2048, "f32", "uniform", ("mean",),
                 note="tiny CPU-checkable case"),
        Workload("ragged", 2, 1269, 1000, 10000, "f32", "uniform", ("sum", "mean"),
                 note="3x423 tokens, ragged against every tile size"),
        Workload("llama2_head", 3, 4096, 4096, 32000, "bf16", "uniform", ("mean",),
                 note="2x2048 tokens through a Llama-2-sized head"),
        Workload("llama3_head_t4096", 4, 4096, 4096, 128256, "bf16", "zipf", ("mean",)),
        Workload("llama3_head_t8192", 4, 8192, 4096, 128256, "bf16", "zipf", ("mean",)),
        Workload("llama3_head_t16384", 4, 16384, 4096, 128256, "bf16", "zipf", ("mean",),
                 note="headline workload"),
        Workload("llama3_head_t32768", 5, 32768, 4096, 128256, "bf16", "uniform", ("mean",),
                 note="large batch; peak memory must stay below the bf16 logits size"),
        Workload("qwen3_head_t32768", 6, 32768, 4096, 151936, "bf16", "uniform", ("mean",),
                 note="Qwen3-sized head"),
        Workload("gemma3_head_t8192", 7, 8192, 2304, 262208, "bf16", "uniform", ("mean",),
                 note="Gemma3-sized head: narrow hidden, very wide vocabulary"),
        Workload("fp32_head_t32768", 11, 32768, 4096, 32000, "f32", "uniform", ("mean",),
                 note="fp32 head of the Liger-Kernel PR's fp32 tables (T=32768, V=32000)"),
        Workload("spread", 8, 1100, 1024, 8000, "bf16", "uniform", ("sum", "mean", "none"),
                 w_std=0.3, note="logits of standard deviation ~10: a peaked softmax"),
        Workload("confident", 9, 1100, 1024, 8000, "bf16", "uniform", ("sum", "mean", "none"),
                 confident_margin=14.0,
                 note="target probability ~0.99, loss ~1e-2"),
        Workload("spread_confident", 10, 1100, 1024, 8000, "bf16", "uniform",
                 ("sum", "mean", "none"), w_std=0.3, confident_margin=60.0,
                 note="logits spread over tens of units and a dominant target"),
    ]
}


def bf16_round_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return the uint16 bits.

    Inputs are finite normal draws, so no NaN/Inf handling is needed; an infinite or NaN input
    raises instead of being rounded silently.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    if not np.all(np.isfinite(a)):
        raise ValueError("bf16_round_bits expects finite values")
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to the float32 values they represent (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def zipf_targets(rng: np.random.Generator, n: int, V: int, s: float) -> np.ndarray:
    """Draw n ids in [0, V) with P(id = k) proportional to (k + 1)^-s, by inverse CDF."""
    weights = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(weights)
    u = rng.random(n) * cdf[-1]
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, V - 1).astype(np.int64)


@dataclass
class FlceInputs:
    """Host arrays for one workload.

    ``x`` and ``weight`` are float32 arrays holding exactly the values both paths see (for bf16
    workloads every element is bf16-representable). ``x_bits``/``weight_bits`` hold the uint16
    bf16 patterns for bf16 workloads (None for f32).
    """

    workload: Workload
    x: np.ndarray
    weight: np.ndarray
    target: np.ndarray
    x_bits: np.ndarray | None
    weight_bits: np.ndarray | None


def _draw_normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def make_inputs(workload: Workload | str, T: int | None = None, H: int | None = None,
                V: int | None = None, dtype: str | None = None,
                target_dist: str | None = None, seed: int | None = None,
                w_std: float | None = None, confident_margin: float | None = None) -> FlceInputs:
    """Generate the seeded inputs of a workload; the keyword arguments override its fields."""
    if isinstance(workload, str):
        workload = WORKLOADS[workload]
    T = workload.T if T is None else int(T)
    H = workload.H if H is None else int(H)
    V = workload.V if V is None else int(V)
    dtype = workload.dtype if dtype is None else dtype
    target_dist = workload.target_dist if target_dist is None else target_dist
    seed = workload.seed if seed is None else int(seed)
    w_std = workload.w_std if w_std is None else float(w_std)
    margin = workload.confident_margin if confident_margin is None else float(confident_margin)
    wl = Workload(workload.name, workload.index, T, H, V, dtype, target_dist,
                  workload.reductions, workload.x_std, w_std, workload.zipf_s, margin,
                  workload.note)

    child = np.random.SeedSequence(seed).spawn(3)
    rx, rw, ry = (np.random.Generator(np.random.PCG64(c)) for c in child)
    x = _draw_normal(rx, (T, H), wl.x_std)
    w = _draw_normal(rw, (V, H), wl.w_std)
    if target_dist == "uniform":
        y = ry.integers(0, V, size=T, dtype=np.int64)
    elif target_dist == "zipf":
        y = zipf_targets(ry, T, V, wl.zipf_s)
    else:
        raise ValueError(f"unknown target distribution {target_dist!r}")

    if dtype not in ("bf16", "f32"):
        raise ValueError(f"unknown dtype {dtype!r}")
    xb = wb = None
    if dtype == "bf16":
        xb = bf16_round_bits(x)
        x = bf16_bits_to_f32(xb)
    if margin > 0.0:
        # raise each target logit by `margin` (relative to the x both paths see); tokens that
        # share a target add their shifts to the same weight row
        x64 = x.astype(np.float64)
        shift = margin * x64 / np.einsum("th,th->t", x64, x64)[:, None]
        w64 = w.astype(np.float64)
        np.add.at(w64, y, shift)
        w = w64.astype(np.float32)
    if dtype == "bf16":
        wb = bf16_round_bits(w)
        w = bf16_bits_to_f32(wb)
    return FlceInputs(wl, x, w, y, xb, wb)
