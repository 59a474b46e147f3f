"""The stored oracle results for the full-size Llama-3-head workloads (CPU).

tests/golden/llama3_head_oracle.npz is written by tests/golden/make_llama3_oracle.py, which
calls only the oracle and the seeded input generators. This test regenerates the inputs of the
smallest of those workloads and checks, against the oracle recomputed here, that the file still
matches: the input digest, the loss against the stored lse and the target logits, and one of
each kind of stored row (lse, grad_x row, grad_weight row).
"""
import hashlib
import os

import numpy as np

import oracle
from lm_head_linear_02_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "llama3_head_oracle.npz")


def test_stored_llama3_oracle_results_reproduce():
    name = "llama3_head_t4096"
    with np.load(GOLDEN) as z:
        g = {k.split("__", 1)[1]: z[k] for k in z.files if k.startswith(name + "__")}
        names = {k.split("__", 1)[0] for k in z.files}
    assert names == {"llama3_head_t4096", "llama3_head_t8192", "llama3_head_t16384",
                     "llama3_head_t32768"}
    inp = make_inputs(name)
    h = hashlib.sha256()
    for a in (inp.x_bits, inp.weight_bits, inp.target):
        h.update(np.ascontiguousarray(a).tobytes())
    assert h.hexdigest() == str(g["inputs_sha256"])
    T = inp.workload.T
    assert g["lse"].shape == (T,)
    # the mean loss is the mean of lse[t] - z[t, target[t]]
    x = inp.x.astype(np.float64)
    zy = np.einsum("th,th->t", x, inp.weight[inp.target].astype(np.float64))
    assert abs(np.mean(g["lse"] - zy) - float(g["loss"])) < 1e-9
    t = int(g["token_rows"][3])
    s = oracle.sampled_rows(inp.x, inp.weight, inp.target, [t], "mean", 1.0)
    assert abs(s["lse"][0] - g["lse"][t]) < 1e-10
    assert np.allclose(s["grad_x"][0], g["grad_x_rows"][3], rtol=1e-6, atol=1e-12)
    v = int(g["vocab_rows"][0])  # id 0, the most frequent Zipf target
    assert v == 0
    gw = oracle.grad_weight_rows(inp.x, inp.weight, inp.target, g["lse"], [v], "mean", 1.0)
    assert np.allclose(gw[0], g["grad_weight_rows"][0], rtol=1e-6, atol=1e-12)
