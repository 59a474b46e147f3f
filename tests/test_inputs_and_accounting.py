"""Host-side checks of the seeded input generators and of the byte/FLOP accounting."""
import json
import os

import numpy as np
import pytest

from lm_head_linear_02_gb300 import inputs, roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_generator_is_deterministic_and_seeded():
    a = inputs.make_inputs("tiny")
    b = inputs.make_inputs("tiny")
    assert np.array_equal(a.x, b.x) and np.array_equal(a.weight, b.weight)
    assert np.array_equal(a.target, b.target)
    c = inputs.make_inputs("tiny", seed=999)
    assert not np.array_equal(a.x, c.x)
    assert a.x.shape == (128, 256) and a.weight.shape == (2048, 256)
    assert a.target.dtype == np.int64 and a.target.min() >= 0 and a.target.max() < 2048
    assert abs(a.x.std() - 1.0) < 0.02 and abs(a.weight.std() - 0.02) < 0.001


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(0)
    v = np.concatenate([r.standard_normal(100000).astype(np.float32),
                        np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -1.0 - 2**-8, 0.0, -0.0],
                                 dtype=np.float32)])
    bits = inputs.bf16_round_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
    back = inputs.bf16_bits_to_f32(bits)
    assert np.array_equal(back, torch.from_numpy(v).to(torch.bfloat16).float().numpy())


def test_bf16_workload_values_are_representable():
    a = inputs.make_inputs("llama2_head", T=64, V=300)
    assert a.x_bits is not None
    assert np.array_equal(inputs.bf16_bits_to_f32(inputs.bf16_round_bits(a.x)), a.x)


def test_zipf_targets_follow_power_law():
    r = np.random.Generator(np.random.PCG64(7))
    V = 128256
    y = inputs.zipf_targets(r, 200000, V, 1.1)
    assert y.min() >= 0 and y.max() < V
    w = np.arange(1, V + 1, dtype=np.float64) ** -1.1
    p0 = w[0] / w.sum()
    assert abs((y == 0).mean() - p0) < 0.005
    assert abs((y == 1).mean() / (y == 0).mean() - 2.0 ** -1.1) < 0.03


def test_kernelindex_dram_floor_reproduced():
    g = json.load(open(os.path.join(GOLDEN, "kernelindex_dram_floor.json")))
    w = g["workload"]
    nbytes = roofline.declared_tensor_bytes(w["T"], w["H"], w["V"], w["elem_bytes"])
    us = nbytes / g["bandwidth_bytes_per_s"] * 1e6
    assert abs(us - g["printed_floor_us"]) <= g["printed_precision_us"]


def test_flop_counts():
    assert roofline.flops(16384, 4096, 128256) == 8 * 16384 * 4096 * 128256
    assert roofline.flops(1, 1, 1, "fwd") == 2 and roofline.flops(1, 1, 1, "bwd") == 6


def test_traffic_digest_ignores_comments_but_not_code():
    """bench.py keys the recorded ncu DRAM traffic by a digest of the kernel sources without
    comments and whitespace: editing a comment keeps the record, editing code voids it."""
    import bench
    code = 'int a = 1; // note\n/* block\n comment */ const char* s = "//x/*y*/"; char c = \'"\';\n'
    assert bench.strip_comments(code) == 'inta=1;constchar*s="//x/*y*/";charc=\'"\';'
    strip = bench.strip_comments
    assert strip(code.replace("// note", "// another note")) == strip(code)
    assert strip(code.replace("a = 1", "a = 2")) != strip(code)
    assert strip(code.replace('"//x/*y*/"', '"//x/*z*/"')) != strip(code)  # inside a literal
    # the digest reads the kernel sources through the same stripping
    sources = {}

    def read(name):
        import os
        with open(os.path.join(bench.CSRC, name), encoding="utf-8") as f:
            sources[name] = f.read()
        return sources[name] + "\n// an added comment\n"

    assert bench.sources_digest(read) == bench.sources_digest()
    assert sources and len(bench.sources_digest()) == 64
