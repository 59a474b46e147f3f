"""Float64 CPU oracle for fused linear cross-entropy (FLCE).

TEST INFRASTRUCTURE ONLY. This is the plain, slow, obviously correct statement of what the GPU
path computes. Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference arm may import it. The product path (the C-ABI library and its Python binding) never
imports, calls or links anything here, and nothing here imports the product path.

What is computed, by page and section:

* "Fused linear + cross-entropy" (KernelIndex operation page), summary and "Semantics" table:
  x float[tokens, hidden], weight float[vocab, hidden], target int64[tokens], loss float[1].
  The logits z = x . weight^T are the LM-head projection and are scored by cross-entropy
  against the integer targets.
* "[example] fused_linear_cross_entropy kernel" (Helion PR #1268), description: the forward
  yields the per-token log-sum-exp (kept for the backward) and the target logits; the backward
  recomputes the logits and produces grad_input and grad_weight.
* "feat(FLCE): add helion version of fused linear cross entropy" (Liger-Kernel PR #928), the
  failing-test list: the two reductions 'sum' and 'mean'.

The fused method reaches the textbook definition exactly (up to rounding order): the pages say
only that the logits are never materialised, never that they are approximated. So this oracle is
the definition written out in float64:

    z[t, v]   = sum_h x[t, h] * weight[v, h]
    lse[t]    = m_t + ln sum_v exp(z[t, v] - m_t),      m_t = max_v z[t, v]
    l[t]      = lse[t] - z[t, target[t]]
    loss      = sum_t l[t]            (sum)   or   (1/T) sum_t l[t]   (mean)   or   l   (none)
    g         = grad_loss             (sum)   or   grad_loss / T      (mean)   or   grad_loss[t]
    dz[t, v]  = (exp(z[t, v] - lse[t]) - [v == target[t]]) * g
    grad_x    = dz . weight          grad_weight = dz^T . x

Token chunking below bounds memory only (no T x V float64 array is ever held); each chunk uses
the same formulas, and grad_weight is summed over chunks in increasing token order.

Readings where the pages are silent: no bias term; natural logarithm; the 'mean' denominator is
the token count T (the pages define no ignore_index, so every target counts and a target outside
[0, V) is an error); loss is a scalar for 'sum' and 'mean'. The 'none' reduction (an extension:
the pages list only 'sum' and 'mean') returns the per-token losses l[t] that the two reductions
aggregate, and its backward takes one upstream gradient per token.

Pins (tests/test_oracle_pins.py): closed forms for weight = 0, x = 0 and identical weight rows,
a hand-derived 2x2x3 example (tests/golden/), brute-force pure-Python loops, torch's float64
cross_entropy as a library special case, central finite differences, the two-class logistic
special case, row sums of dz, shift invariance, sum = T * mean, and chunk-size independence.
The per-row helpers (sampled_rows, grad_weight_rows) are pinned against the full oracle, and
grad_weight_rows also against the weight = 0 closed form with lse given in closed form, torch's
float64 autograd with torch's own logsumexp, and finite differences.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "REDUCTIONS",
    "logits",
    "log_sum_exp",
    "grad_scale",
    "dlogits",
    "forward",
    "backward",
    "flce",
    "sampled_rows",
    "grad_weight_rows",
]

REDUCTIONS = ("sum", "mean", "none")


def _check(x, weight, target):
    x = np.asarray(x, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    target = np.asarray(target, dtype=np.int64)
    if x.ndim != 2 or weight.ndim != 2 or target.ndim != 1:
        raise ValueError("expected x[T,H], weight[V,H], target[T]")
    if x.shape[1] != weight.shape[1] or x.shape[0] != target.shape[0]:
        raise ValueError("shape mismatch between x, weight and target")
    V = weight.shape[0]
    if target.size and (target.min() < 0 or target.max() >= V):
        raise ValueError("target outside [0, vocab)")
    return x, weight, target


def logits(x_rows: np.ndarray, weight: np.ndarray) -> np.ndarray:
    """z = x . weight^T: the LM-head projection ("Fused linear + cross-entropy", summary)."""
    return x_rows @ weight.T


def log_sum_exp(z: np.ndarray) -> np.ndarray:
    """Per-row log-sum-exp with the row maximum taken out first (Helion PR #1268, forward)."""
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def grad_scale(grad_loss, reduction: str, T: int):
    """g: d loss / d l[t] times the incoming grad_loss ('sum' -> 1, 'mean' -> 1/T, 'none' -> the
    per-token upstream gradients themselves, an array of T values)."""
    if reduction == "sum":
        return float(grad_loss)
    if reduction == "mean":
        return float(grad_loss) / T
    if reduction == "none":
        g = np.asarray(grad_loss, dtype=np.float64).reshape(-1)
        if g.shape != (T,):
            raise ValueError("reduction 'none' needs one upstream gradient per token")
        return g
    raise ValueError(f"reduction must be one of {REDUCTIONS}")


def dlogits(z: np.ndarray, lse: np.ndarray, target: np.ndarray, g) -> np.ndarray:
    """dz = (softmax(z) - onehot(target)) * g for a block of rows (Helion PR #1268, backward);
    g is a scalar or one value per row."""
    p = np.exp(z - lse[:, None])
    p[np.arange(z.shape[0]), target] -= 1.0
    g = np.asarray(g, dtype=np.float64)
    return p * (g[:, None] if g.ndim == 1 else g)


def forward(x, weight, target, reduction: str = "mean", chunk: int = 256):
    """Loss and saved per-token lse (Helion PR #1268, forward; KernelIndex "Semantics")."""
    x, weight, target = _check(x, weight, target)
    if reduction not in REDUCTIONS:
        raise ValueError(f"reduction must be one of {REDUCTIONS}")
    T = x.shape[0]
    lse = np.empty(T, dtype=np.float64)
    per_token = np.empty(T, dtype=np.float64)
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        z = logits(x[t0:t1], weight)
        lse[t0:t1] = log_sum_exp(z)
        per_token[t0:t1] = lse[t0:t1] - z[np.arange(t1 - t0), target[t0:t1]]
    if reduction == "none":
        return per_token, lse
    total = per_token.sum()
    loss = total if reduction == "sum" else total / T
    return float(loss), lse


def backward(x, weight, target, lse, reduction: str = "mean", grad_loss=1.0,
             chunk: int = 256):
    """grad_x and grad_weight from recomputed logits (Helion PR #1268, backward)."""
    x, weight, target = _check(x, weight, target)
    lse = np.asarray(lse, dtype=np.float64)
    T = x.shape[0]
    g = grad_scale(grad_loss, reduction, T)
    grad_x = np.empty_like(x)
    grad_w = np.zeros_like(weight)
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        z = logits(x[t0:t1], weight)
        gc = g[t0:t1] if isinstance(g, np.ndarray) else g
        dz = dlogits(z, lse[t0:t1], target[t0:t1], gc)
        grad_x[t0:t1] = dz @ weight
        grad_w += dz.T @ x[t0:t1]
    return grad_x, grad_w


def flce(x, weight, target, reduction: str = "mean", grad_loss=1.0, chunk: int = 256):
    """Forward and backward in one call: dict with loss, lse, grad_x, grad_weight (float64).
    For 'none' the loss is the per-token array and grad_loss holds one value per token."""
    loss, lse = forward(x, weight, target, reduction, chunk)
    grad_x, grad_w = backward(x, weight, target, lse, reduction, grad_loss, chunk)
    return {"loss": loss, "lse": lse, "grad_x": grad_x, "grad_weight": grad_w}


def sampled_rows(x, weight, target, rows, reduction: str = "mean", grad_loss=1.0):
    """lse, per-token loss and grad_x for selected token rows only.

    Each token row depends on its own logits row alone, so these values are exact for any total
    token count T = x.shape[0]; they let a full-size run be checked one row at a time.
    """
    rows = np.asarray(rows, dtype=np.int64)
    T = np.asarray(x).shape[0]
    x_rows, weight, target_rows = _check(np.asarray(x)[rows], weight, np.asarray(target)[rows])
    g = grad_scale(grad_loss, reduction, T)
    if isinstance(g, np.ndarray):
        g = g[rows]
    z = logits(x_rows, weight)
    lse = log_sum_exp(z)
    per_token = lse - z[np.arange(rows.size), target_rows]
    dz = dlogits(z, lse, target_rows, g)
    return {"lse": lse, "per_token_loss": per_token, "grad_x": dz @ weight}



def grad_weight_rows(x, weight, target, lse, vocab_rows, reduction: str = "mean",
                     grad_loss=1.0, chunk: int = 4096):
    """grad_weight[v, :] for selected vocabulary rows v only, given the forward's lse.

    Written out from the definition (Helion PR #1268, backward): for one vocabulary row v,
    column v of the logits is z[:, v] = x . weight[v], column v of dz is
    (exp(z[:, v] - lse) - [target == v]) * g, and grad_weight[v] = sum_t dz[t, v] * x[t].
    Each row needs only its own logits column and the per-token lse, so a full-size problem can
    be checked one vocabulary row at a time. Tokens are taken in chunks (memory only), summed in
    increasing token order.
    """
    x, weight, target = _check(x, weight, target)
    lse = np.asarray(lse, dtype=np.float64).reshape(-1)
    rows = np.asarray(vocab_rows, dtype=np.int64).reshape(-1)
    T = x.shape[0]
    if lse.shape != (T,):
        raise ValueError("lse needs one value per token")
    if rows.size and (rows.min() < 0 or rows.max() >= weight.shape[0]):
        raise ValueError("vocab row outside [0, vocab)")
    g = grad_scale(grad_loss, reduction, T)
    out = np.zeros((rows.size, x.shape[1]), dtype=np.float64)
    for t0 in range(0, T, chunk):
        t1 = min(T, t0 + chunk)
        zc = logits(x[t0:t1], weight[rows])                   # [chunk, rows]: logit columns
        dzc = np.exp(zc - lse[t0:t1, None])
        dzc -= (target[t0:t1, None] == rows[None, :])         # one-hot of the target column
        gc = g[t0:t1] if isinstance(g, np.ndarray) else g
        dzc *= (gc[:, None] if isinstance(gc, np.ndarray) else gc)
        out += dzc.T @ x[t0:t1]
    return out
