"""Write the float64 oracle's results for the full-size Llama-3-head workloads.

The workloads are the "Current records" shapes of the KernelIndex "Fused linear +
cross-entropy" page: hidden 4096, vocab 128256, tokens 4096, 8192, 16384 (Zipf targets) and
32768 (uniform targets), bf16 inputs, reduction 'mean'. For each one this script stores what the
oracle computes, so that the GPU tests can compare against the oracle itself at full size:

* the loss and all T per-token log-sum-exp values (the oracle's forward over every token);
* grad_x for a set of token rows (``oracle.sampled_rows``: each row needs only its own logits);
* grad_weight for a set of vocabulary rows (``oracle.grad_weight_rows``, given the forward's
  lse: each row needs only its own logits column), including id 0, the most frequent Zipf
  target, the last id, and the rows on both sides of tile, slab and chunk boundaries.

Only ``oracle`` and the seeded input generators are imported: no value here comes from the GPU
path. The loss and lse are stored in float64; the sampled gradient rows in float32 (a relative
rounding of 6e-8, against a comparison tolerance of 2e-2). Each workload also records a SHA-256
digest of the input bytes it was computed from, which the tests check before comparing.

    python tests/golden/make_llama3_oracle.py            # writes llama3_head_oracle.npz here
"""
from __future__ import annotations

import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from lm_head_linear_02_gb300.inputs import make_inputs  # noqa: E402

OUT = os.path.join(HERE, "llama3_head_oracle.npz")
WORKLOADS = ("llama3_head_t4096", "llama3_head_t8192", "llama3_head_t16384",
             "llama3_head_t32768")


def inputs_digest(inp) -> str:
    """SHA-256 over the bf16 bit patterns of x and weight and the int64 targets."""
    h = hashlib.sha256()
    for a in (inp.x_bits, inp.weight_bits, inp.target):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def token_rows(T: int) -> np.ndarray:
    """Rows at tile and chunk edges (128, 256, 512 token tiles; halves and quarters of T) and
    the last rows, plus seeded random rows."""
    fixed = [0, 1, 127, 128, 255, 256, 511, 512, T // 4 - 1, T // 4, T // 2 - 1, T // 2,
             3 * T // 4 - 1, 3 * T // 4, T - 2, T - 1]
    rnd = np.random.default_rng(7000 + T).integers(0, T, 10)
    return np.unique(np.concatenate([fixed, rnd])).astype(np.int64)


def vocab_rows(V: int) -> np.ndarray:
    """The most frequent Zipf ids, rows on both sides of 256-row tiles, 512-row pair tiles and
    the backward's vocabulary slabs at these token counts, the last ids, and seeded random
    rows."""
    fixed = [0, 1, 2, 3, 255, 256, 511, 512, 16127, 16128, 32255, 32256, 64255, 64256,
             V - 257, V - 256, V - 2, V - 1]
    rnd = np.random.default_rng(8000 + V).integers(0, V, 8)
    return np.unique(np.concatenate([fixed, rnd])).astype(np.int64)


def main() -> None:
    out = {}
    for name in WORKLOADS:
        t0 = time.time()
        inp = make_inputs(name)
        T, V = inp.workload.T, inp.workload.V
        loss, lse = oracle.forward(inp.x, inp.weight, inp.target, "mean")
        rows = token_rows(T)
        sr = oracle.sampled_rows(inp.x, inp.weight, inp.target, rows, "mean", 1.0)
        vrows = vocab_rows(V)
        gw = oracle.grad_weight_rows(inp.x, inp.weight, inp.target, lse, vrows, "mean", 1.0)
        out[f"{name}__inputs_sha256"] = np.array(inputs_digest(inp))
        out[f"{name}__loss"] = np.array(loss, dtype=np.float64)
        out[f"{name}__lse"] = lse.astype(np.float64)
        out[f"{name}__token_rows"] = rows
        out[f"{name}__grad_x_rows"] = sr["grad_x"].astype(np.float32)
        out[f"{name}__vocab_rows"] = vrows
        out[f"{name}__grad_weight_rows"] = gw.astype(np.float32)
        print(f"{name}: loss {loss:.9f}  ({time.time() - t0:.0f} s)", flush=True)
        del inp
    np.savez_compressed(OUT, **out)
    print(f"wrote {OUT} ({os.path.getsize(OUT) / 1e6:.2f} MB)")


if __name__ == "__main__":
    main()
