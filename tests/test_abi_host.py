"""Host-side checks of the C ABI: the library builds, loads, exports every declared symbol, and
rejects bad arguments with the documented codes before touching the GPU.

Pointers passed here are fake addresses; every call below must fail validation before any
CUDA call, so nothing is dereferenced.
"""
import os
import re
import subprocess

import numpy as np
import pytest

from lm_head_linear_02_gb300 import binding as B
from lm_head_linear_02_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "flce_forward" in names and "flce_backward" in names
    out = subprocess.run(["nm", "-D", "--defined-only", B.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (flce_[a-z_0-9]+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)


def test_version_and_strerror(lib):
    assert B.flce_version() == 10000
    for code in (0, -1, -2, -3, -4, -5):
        assert B.flce_strerror(code)
    assert "unknown" in B.flce_strerror(-99)


def test_workspace_sizes():
    T, H, V = 16384, 4096, 128256
    fwd = B.flce_forward_workspace_size(T, H, V, B.FLCE_DTYPE_BF16)
    n_tiles = (V + 255) // 256
    assert fwd >= 2 * 4 * n_tiles * T + 4 * T
    bwd = B.flce_backward_workspace_size(T, H, V, B.FLCE_DTYPE_BF16)
    vc = B.flce_backward_slab_width(T, H, V, B.FLCE_DTYPE_BF16)
    assert vc % 256 == 0 and 256 <= vc <= V + 255
    # as few slabs of at most 1 GiB as possible (4), of nearly equal width
    assert vc == 32256 and 2 * T * vc <= 1 << 30 and -(-V // vc) == 4
    # Gemma-3-sized head: 5 balanced slabs, not 4 wide ones and a 64-column sliver
    assert B.flce_backward_slab_width(8192, 2304, 262208, B.FLCE_DTYPE_BF16) == 52480
    assert bwd >= 2 * T * vc
    # never anything close to the tokens x vocab logits
    assert fwd + bwd < 2 * T * V
    for bad in [(0, H, V, 0), (T, 0, V, 0), (T, H, -1, 0), (T, H, V, 7)]:
        assert B.flce_forward_workspace_size(*bad) == 0
        assert B.flce_backward_workspace_size(*bad) == 0


def test_workspace_stays_below_logits_size_at_32k_tokens():
    T, H, V = 32768, 4096, 128256
    logits_bf16 = 2 * T * V
    fwd = B.flce_forward_workspace_size(T, H, V, B.FLCE_DTYPE_BF16)
    bwd = B.flce_backward_workspace_size(T, H, V, B.FLCE_DTYPE_BF16)
    inputs_outputs = 2 * (2 * T * H + 2 * V * H) + 8 * T + 4 * T
    assert inputs_outputs + max(fwd, bwd) < logits_bf16


def test_slab_override(lib):
    try:
        B.flce_set_backward_slab_width(512)
        assert B.flce_backward_slab_width(1000, 64, 10000, 0) == 512
        assert B.flce_backward_slab_width(1000, 64, 300, 0) == 512  # clamped to round_up(V)
        with pytest.raises(B.FlceError):
            B.flce_set_backward_slab_width(100)
    finally:
        B.flce_set_backward_slab_width(0)
    assert B.flce_backward_slab_width(1000, 64, 300, 0) == 512


FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


def _fwd(**kw):
    a = dict(x=FAKE, weight=FAKE + 0x10000000, target=FAKE + 0x20000000, T=64, H=64, V=512,
             dtype=0, reduction=1, loss=FAKE + 0x30000000, lse=FAKE + 0x30001000,
             workspace=FAKE + 0x40000000, workspace_bytes=1 << 30, status=FAKE + 0x30000100,
             stream=0)
    a.update(kw)
    return B.flce_forward(a["x"], a["weight"], a["target"], a["T"], a["H"], a["V"], a["dtype"],
                          a["reduction"], a["loss"], a["lse"], a["workspace"],
                          a["workspace_bytes"], a["status"], a["stream"], check=False)


def _bwd(**kw):
    a = dict(x=FAKE, weight=FAKE + 0x10000000, target=FAKE + 0x20000000,
             lse=FAKE + 0x21000000, T=64, H=64, V=512, dtype=0, reduction=1,
             grad_loss=FAKE + 0x22000000, grad_x=FAKE + 0x30000000,
             grad_weight=FAKE + 0x31000000, workspace=FAKE + 0x40000000,
             workspace_bytes=1 << 30, status=FAKE + 0x32000000, stream=0)
    a.update(kw)
    return B.flce_backward(a["x"], a["weight"], a["target"], a["lse"], a["T"], a["H"], a["V"],
                           a["dtype"], a["reduction"], a["grad_loss"], a["grad_x"],
                           a["grad_weight"], a["workspace"], a["workspace_bytes"], a["status"],
                           a["stream"], check=False)


@pytest.mark.parametrize("kw,code", [
    (dict(x=0), B.FLCE_ERR_ARG),
    (dict(target=0), B.FLCE_ERR_ARG),
    (dict(loss=0), B.FLCE_ERR_ARG),
    (dict(status=0), B.FLCE_ERR_ARG),
    (dict(T=0), B.FLCE_ERR_ARG),
    (dict(V=-3), B.FLCE_ERR_ARG),
    (dict(T=1 << 30), B.FLCE_ERR_ARG),
    (dict(dtype=2), B.FLCE_ERR_ARG),
    (dict(reduction=3), B.FLCE_ERR_ARG),
    (dict(H=60), B.FLCE_ERR_UNSUPPORTED),          # 120-byte rows for bf16
    (dict(H=6, dtype=1), B.FLCE_ERR_UNSUPPORTED),  # 24-byte rows for f32
    (dict(x=FAKE + 8), B.FLCE_ERR_UNSUPPORTED),
    (dict(workspace=0), B.FLCE_ERR_WORKSPACE),
    (dict(workspace_bytes=16), B.FLCE_ERR_WORKSPACE),
    (dict(workspace=FAKE + 0x40000010), B.FLCE_ERR_UNSUPPORTED),
    (dict(lse=FAKE + 0x100), B.FLCE_ERR_ALIAS),     # lse overlaps x
    (dict(loss=FAKE + 0x30001004), B.FLCE_ERR_ALIAS),  # loss inside lse
    (dict(workspace=FAKE + 0x10000000), B.FLCE_ERR_ALIAS),  # workspace over weight
])
def test_forward_validation(lib, kw, code):
    assert _fwd(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(lse=0), B.FLCE_ERR_ARG),
    (dict(grad_loss=0), B.FLCE_ERR_ARG),
    (dict(grad_weight=0), B.FLCE_ERR_ARG),
    (dict(H=4), B.FLCE_ERR_UNSUPPORTED),
    (dict(grad_x=FAKE + 0x30000004), B.FLCE_ERR_UNSUPPORTED),
    (dict(workspace_bytes=0), B.FLCE_ERR_WORKSPACE),
    (dict(grad_x=FAKE + 0x10), B.FLCE_ERR_ALIAS),           # grad_x over x
    (dict(grad_weight=FAKE + 0x30000000), B.FLCE_ERR_ALIAS),  # the two outputs overlap
    (dict(status=FAKE + 0x21000000), B.FLCE_ERR_ALIAS),      # status inside lse
])
def test_backward_validation(lib, kw, code):
    assert _bwd(**kw) == code


def test_binding_raises_on_error(lib):
    with pytest.raises(B.FlceError) as e:
        B.flce_forward(0, 0, 0, 1, 8, 8, 0, 0, 0, 0, 0, 0, 0, 0)
    assert e.value.code == B.FLCE_ERR_ARG


def test_wrapper_refuses_what_the_c_entry_points_cannot_check():
    """The saved lse's length and device, and the reduction name, are checked in the PyTorch
    wrapper before any buffer is allocated or the library is called."""
    torch = pytest.importorskip("torch")
    from lm_head_linear_02_gb300 import autograd as A

    cpu = torch.device("cpu")
    ok = A._saved_lse(torch.zeros(6, dtype=torch.float64), 6, cpu)
    assert ok.dtype == torch.float32 and ok.shape == (6,)
    for bad in (torch.zeros(5), torch.zeros(7), torch.zeros(6, 1), torch.zeros(())):
        with pytest.raises(ValueError):
            A._saved_lse(bad, 6, cpu)
    with pytest.raises(ValueError):
        A._saved_lse(torch.zeros(6), 6, torch.device("cuda", 0))
    assert A._reduction("sum") == B.FLCE_REDUCTION_SUM
    assert A._reduction("mean") == B.FLCE_REDUCTION_MEAN
    assert A._reduction("none") == B.FLCE_REDUCTION_NONE
    for bad in ("avg", "Mean", ""):
        with pytest.raises(ValueError):
            A._reduction(bad)
    # tensors that are not on a CUDA device are refused before anything else happens
    x, w, y = torch.zeros(4, 8), torch.zeros(16, 8), torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError):
        A.flce_forward(x, w, y, "mean")


def test_tuning_knobs_validate(lib):
    assert B.flce_get_tuning(B.FLCE_TUNE_RASTER_ROWS) == 2048
    for key, bad in [(B.FLCE_TUNE_RASTER_ROWS, 100), (B.FLCE_TUNE_RASTER_ROWS, 0),
                     (B.FLCE_TUNE_SM_PAIRS, 8), (B.FLCE_TUNE_SM_PAIRS, -2),
                     (B.FLCE_TUNE_WIDE_TILES, 8), (B.FLCE_TUNE_WIDE_TILES, -2),
                     (B.FLCE_TUNE_RASTER_VOCAB, 100), (B.FLCE_TUNE_RASTER_VOCAB, -256),
                     (B.FLCE_TUNE_SPLIT_EPILOGUE, 8), (B.FLCE_TUNE_SPLIT_EPILOGUE, -2),
                     (B.FLCE_TUNE_CHUNK_BYTES, -1), (B.FLCE_TUNE_ORDERED_DRAIN, 8),
                     (B.FLCE_TUNE_ORDERED_DRAIN, -2), (99, 1)]:
        with pytest.raises(B.FlceError):
            B.flce_set_tuning(key, bad)
    B.flce_set_tuning(B.FLCE_TUNE_RASTER_ROWS, 4096)
    try:
        assert B.flce_get_tuning(B.FLCE_TUNE_RASTER_ROWS) == 4096
    finally:
        B.flce_set_tuning(B.FLCE_TUNE_RASTER_ROWS, 2048)
    # the wide-tile mask needs no device to report: default (all roles) or the value set
    assert B.flce_get_tuning(B.FLCE_TUNE_WIDE_TILES) == 7
    B.flce_set_tuning(B.FLCE_TUNE_WIDE_TILES, 5)
    try:
        assert B.flce_get_tuning(B.FLCE_TUNE_WIDE_TILES) == 5
    finally:
        B.flce_set_tuning(B.FLCE_TUNE_WIDE_TILES, -1)
    assert B.flce_get_tuning(B.FLCE_TUNE_WIDE_TILES) == 7
    # vocabulary raster groups: 4096 rows by default, multiples of 256 (0: token raster)
    assert B.flce_get_tuning(B.FLCE_TUNE_RASTER_VOCAB) == 4096
    B.flce_set_tuning(B.FLCE_TUNE_RASTER_VOCAB, 0)
    try:
        assert B.flce_get_tuning(B.FLCE_TUNE_RASTER_VOCAB) == 0
    finally:
        B.flce_set_tuning(B.FLCE_TUNE_RASTER_VOCAB, 4096)
    # two epilogue warps per row block: off by default; -1 restores the default
    assert B.flce_get_tuning(B.FLCE_TUNE_SPLIT_EPILOGUE) == 0
    B.flce_set_tuning(B.FLCE_TUNE_SPLIT_EPILOGUE, B.FLCE_ROLE_FORWARD | B.FLCE_ROLE_DZ)
    try:
        assert B.flce_get_tuning(B.FLCE_TUNE_SPLIT_EPILOGUE) == 3
    finally:
        B.flce_set_tuning(B.FLCE_TUNE_SPLIT_EPILOGUE, -1)
    assert B.flce_get_tuning(B.FLCE_TUNE_SPLIT_EPILOGUE) == 0
    # row halves drained one after the other: a role mask; -1 restores the default
    default = B.flce_get_tuning(B.FLCE_TUNE_ORDERED_DRAIN)
    assert default == B.FLCE_ROLE_FORWARD | B.FLCE_ROLE_DZ
    B.flce_set_tuning(B.FLCE_TUNE_ORDERED_DRAIN, B.FLCE_ROLE_DZ)
    try:
        assert B.flce_get_tuning(B.FLCE_TUNE_ORDERED_DRAIN) == B.FLCE_ROLE_DZ
    finally:
        B.flce_set_tuning(B.FLCE_TUNE_ORDERED_DRAIN, -1)
    assert B.flce_get_tuning(B.FLCE_TUNE_ORDERED_DRAIN) == default


def test_single_call_chunk_rule(lib):
    """Tokens per chunk of the single-call schedule: a multiple of 256, at most half of T (so no
    chunk ever holds all tokens' logits) and at most FLCE_TUNE_CHUNK_BYTES (1.5 GiB by default)
    of bf16 logits; bf16 only, T >= 512. The workspace holds the chunk buffer and the per-half-
    tile partials, no V x H accumulator, so at the headline size the whole call (inputs and
    gradients included) stays below the bf16 logits it avoids."""
    bf16 = B.FLCE_DTYPE_BF16
    assert B.flce_get_tuning(B.FLCE_TUNE_CHUNK_BYTES) == 3 << 29
    assert B.flce_forward_backward_chunk_tokens(16384, 4096, 128256, bf16) == 5632  # 3 chunks
    assert B.flce_forward_backward_chunk_tokens(32768, 4096, 128256, bf16) == 5632  # 6 chunks
    assert B.flce_forward_backward_chunk_tokens(4096, 4096, 32000, bf16) == 2048
    assert B.flce_forward_backward_chunk_tokens(1269, 1000, 10000, bf16) == 768
    assert B.flce_forward_backward_chunk_tokens(300, 256, 1500, bf16) == 300  # below 512: T
    assert B.flce_forward_backward_chunk_tokens(16384, 4096, 128256, B.FLCE_DTYPE_F32) == 16384
    # Gemma-3-sized head: 3 chunks of nearly equal size (2816 + 2816 + 2560), not 3840 + 3840 + 512
    assert B.flce_forward_backward_chunk_tokens(8192, 2304, 262208, bf16) == 2816
    T, H, V = 16384, 4096, 128256
    ws = B.flce_forward_backward_workspace_size(T, H, V, bf16)
    assert ws + 2 * 2 * H * (T + V) < 2 * T * V  # x, weight, grad_x, grad_weight + workspace
    for T, V in [(16384, 128256), (32768, 151936), (8192, 262208), (600, 513), (100000, 50000)]:
        c = B.flce_forward_backward_chunk_tokens(T, 4096, V, bf16)
        ldz = -(-V // 256) * 256
        assert c % 256 == 0 and c >= 256
        assert c <= -(-T // 2 // 256) * 256 + 256 and c < T
        assert c == 256 or 2 * c * ldz <= 3 << 29
    # the budget is a knob: 2 GiB gives 2 chunks of 8192 at the headline size; 0 restores it
    B.flce_set_tuning(B.FLCE_TUNE_CHUNK_BYTES, 1 << 31)
    try:
        assert B.flce_forward_backward_chunk_tokens(16384, 4096, 128256, bf16) == 8192
    finally:
        B.flce_set_tuning(B.FLCE_TUNE_CHUNK_BYTES, 0)
    assert B.flce_forward_backward_chunk_tokens(16384, 4096, 128256, bf16) == 5632


def _fb(**kw):
    a = dict(x=FAKE, weight=FAKE + 0x10000000, target=FAKE + 0x20000000, T=64, H=64, V=512,
             dtype=0, reduction=1, grad_loss=FAKE + 0x22000000, loss=FAKE + 0x23000000,
             lse=FAKE + 0x23001000, grad_x=FAKE + 0x30000000, grad_weight=FAKE + 0x31000000,
             workspace=FAKE + 0x40000000, workspace_bytes=1 << 30, status=FAKE + 0x32000000,
             stream=0)
    a.update(kw)
    return B.flce_forward_backward(a["x"], a["weight"], a["target"], a["T"], a["H"], a["V"],
                                   a["dtype"], a["reduction"], a["grad_loss"], a["loss"],
                                   a["lse"], a["grad_x"], a["grad_weight"], a["workspace"],
                                   a["workspace_bytes"], a["status"], a["stream"], check=False)


@pytest.mark.parametrize("kw,code", [
    (dict(x=0), B.FLCE_ERR_ARG),
    (dict(grad_loss=0), B.FLCE_ERR_ARG),
    (dict(grad_weight=0), B.FLCE_ERR_ARG),
    (dict(status=0), B.FLCE_ERR_ARG),
    (dict(T=0), B.FLCE_ERR_ARG),
    (dict(dtype=2), B.FLCE_ERR_ARG),
    (dict(reduction=3), B.FLCE_ERR_ARG),
    (dict(H=60), B.FLCE_ERR_UNSUPPORTED),                     # 120-byte bf16 rows
    (dict(grad_x=FAKE + 0x30000008), B.FLCE_ERR_UNSUPPORTED),  # misaligned output
    (dict(workspace=0), B.FLCE_ERR_WORKSPACE),
    (dict(workspace_bytes=64), B.FLCE_ERR_WORKSPACE),
    (dict(workspace=FAKE + 0x40000010), B.FLCE_ERR_UNSUPPORTED),  # not 256-byte aligned
    (dict(loss=FAKE + 0x23001004), B.FLCE_ERR_ALIAS),          # loss inside lse
    (dict(grad_x=FAKE + 0x10), B.FLCE_ERR_ALIAS),              # grad_x over x
    (dict(workspace=FAKE + 0x31000000), B.FLCE_ERR_ALIAS),     # workspace over grad_weight
    # 'none': the loss is [T] = 256 bytes, so at 0xF80 it reaches lse (a scalar would not)
    (dict(reduction=2, loss=FAKE + 0x23000F80), B.FLCE_ERR_ALIAS),
    (dict(status=FAKE + 0x22000000), B.FLCE_ERR_ALIAS),        # status over grad_loss (input)
])
def test_single_call_validation(lib, kw, code):
    """flce_forward_backward checks every argument before it touches the device (every case
    here fails validation, so no device work is ever enqueued on the fake addresses)."""
    assert _fb(**kw) == code



def test_static_scratch_size_checks_on_host(lib):
    """flce_forward_static_scratch checks the problem against its fixed scratch size first."""
    rc = B.flce_forward_static_scratch(FAKE, FAKE + 0x10000000, FAKE + 0x20000000, 0, 64, 512,
                                       B.FLCE_DTYPE_BF16, B.FLCE_REDUCTION_MEAN, FAKE + 0x30000000,
                                       FAKE + 0x30001000, FAKE + 0x30000100, 0, check=False)
    assert rc == B.FLCE_ERR_ARG
    rc = B.flce_forward_static_scratch(FAKE, FAKE + 0x10000000, FAKE + 0x20000000, 32768, 4096,
                                       128256, B.FLCE_DTYPE_BF16, B.FLCE_REDUCTION_MEAN,
                                       FAKE + 0x30000000, FAKE + 0x30001000, FAKE + 0x30000100, 0,
                                       check=False)
    assert rc == B.FLCE_ERR_WORKSPACE
    assert B.flce_forward_workspace_size(16384, 4096, 128256, B.FLCE_DTYPE_BF16) <= 64 << 20
    # fp32 problems keep their TF32 hi/lo copies of x and weight in the scratch too, 8 (T + V) H
    # bytes: the ragged fp32 workload (1269 x 1000 x 10000) needs about 90 MB and is rejected
    need = B.flce_forward_workspace_size(1269, 1000, 10000, B.FLCE_DTYPE_F32)
    assert need >= 8 * (1269 + 10000) * 1000 > 64 << 20
    rc = B.flce_forward_static_scratch(FAKE, FAKE + 0x10000000, FAKE + 0x20000000, 1269, 1000,
                                       10000, B.FLCE_DTYPE_F32, B.FLCE_REDUCTION_MEAN,
                                       FAKE + 0x30000000, FAKE + 0x30001000, FAKE + 0x30000100, 0,
                                       check=False)
    assert rc == B.FLCE_ERR_WORKSPACE
    assert B.flce_forward_workspace_size(128, 256, 2048, B.FLCE_DTYPE_F32) <= 64 << 20
    # a null output is refused before the size check or any CUDA call
    rc = B.flce_forward_static_scratch(FAKE, FAKE + 0x10000000, FAKE + 0x20000000, 128, 256, 2048,
                                       B.FLCE_DTYPE_BF16, B.FLCE_REDUCTION_MEAN, 0,
                                       FAKE + 0x30001000, FAKE + 0x30000100, 0, check=False)
    assert rc == B.FLCE_ERR_ARG


def test_plain_c_caller(lib, tmp_path):
    """include/flce.h compiles as strict C99 and a C program linked against libflce.so gets the
    documented answers from the size queries and the argument checks (no GPU involved)."""
    import shutil

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    pkg = os.path.dirname(B.lib_path())
    exe = str(tmp_path / "c_abi_host_check")
    src = os.path.join(ROOT, "tests", "c_abi_host_check.c")
    build = subprocess.run([cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                            "-I", os.path.join(ROOT, "include"), src, "-o", exe, "-L", pkg,
                            "-lflce", "-Wl,-rpath," + pkg], capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "ok", run.stdout + run.stderr


def test_sizing_rules_hold_on_random_shapes(lib):
    """The slab, chunk and workspace sizes for 300 random shapes (log-uniform T and V, both
    dtypes): 256-column granularity, no empty slab or chunk, the 1 GiB slab and 1.5 GiB chunk
    budgets, as few slabs as the budget allows, slabs and chunks of nearly equal size, and
    workspaces that hold what the kernels write (for bf16, nothing more than that)."""
    r = np.random.default_rng(2024)
    budget_slab, budget_chunk = 1 << 30, 3 << 29
    up = lambda a, b: -(-a // b) * b  # noqa: E731
    for _ in range(300):
        T = int(np.exp(r.uniform(0, np.log(1 << 18))))
        V = int(np.exp(r.uniform(0, np.log(1 << 19))))
        H = 8 * int(r.integers(1, 2049))
        for dt in (B.FLCE_DTYPE_BF16, B.FLCE_DTYPE_F32):
            label = f"T={T} H={H} V={V} dtype={dt}"
            vc = B.flce_backward_slab_width(T, H, V, dt)
            n = -(-V // vc)
            per_col = 2 * T if dt == B.FLCE_DTYPE_BF16 else 16 * up(T, 4) + 16 * H
            vc_max = max(256, budget_slab // per_col // 256 * 256)
            assert vc % 256 == 0 and 256 <= vc <= up(V, 256), label
            assert (n - 1) * vc < V <= n * vc, label
            assert vc <= vc_max, label
            assert n == 1 or up(-(-V // (n - 1)), 256) > vc_max, label  # no fewer slabs fit
            assert vc - (V - (n - 1) * vc) <= 256 * n, label             # nearly equal widths
            bws = B.flce_backward_workspace_size(T, H, V, dt)
            if dt == B.FLCE_DTYPE_BF16:
                need = 2 * T * vc + (4 * T * H if n > 1 else 0)
                assert need <= bws <= need + 4096, label
            else:
                # dz hi/lo in both orientations, x hi/lo in both, one weight slab's hi/lo in
                # both: O((T + Vc) H), never O(V H)
                need = 8 * T * vc + 8 * vc * up(T, 4) + 8 * T * H + 8 * H * up(T, 4) \
                    + 8 * vc * H + 8 * H * up(vc, 4)
                assert need <= bws <= need + 8192, label
            fws = B.flce_forward_workspace_size(T, H, V, dt)
            nt = -(-V // 256)
            assert 8 * nt * T + 4 * T <= fws, label
            if dt == B.FLCE_DTYPE_F32:  # x hi/lo and one weight slab of at most 256 MB of copies
                vf_max = max(256, (1 << 28) // (8 * H) // 256 * 256)
                assert fws <= 8 * nt * T + 8 * T + 8 * T * H + 8 * min(vf_max, up(V, 256)) * H \
                    + 4 * (T // 32 + 1) + 8192, label
            c = B.flce_forward_backward_chunk_tokens(T, H, V, dt)
            if dt != B.FLCE_DTYPE_BF16 or T < 512:
                assert c == T, label
                continue
            k = -(-T // c)
            ldz = up(V, 256)
            assert c % 256 == 0 and 256 <= c < T, label
            assert (k - 1) * c < T <= k * c, label
            assert c <= up(-(-T // 2), 256), label
            assert c == 256 or 2 * c * ldz <= budget_chunk, label
            assert c - (T - (k - 1) * c) <= 256 * k, label
            fbs = B.flce_forward_backward_workspace_size(T, H, V, dt)
            need = 2 * c * ldz + 2 * 4 * (ldz // 128) * c  # chunk logits + half-tile partials
            # plus per-row target logit and target-excluded sum, block sums, tile counter
            assert need <= fbs <= need + 8 * c + 4 * (T // 32 + 1) + 6 * 256, label


def test_missing_library_fails_loudly(lib, monkeypatch, tmp_path):
    """Without libflce.so every call raises FlceNotBuilt: there is no fallback path."""
    monkeypatch.setattr(B, "_LIB", None)
    monkeypatch.setattr(B, "lib_path", lambda: str(tmp_path / "libflce.so"))
    with pytest.raises(B.FlceNotBuilt):
        B.flce_version()
    with pytest.raises(B.FlceNotBuilt):
        B.flce_forward_workspace_size(16, 64, 512, B.FLCE_DTYPE_BF16)


def test_build_is_current_and_covers_every_source(lib):
    """build() leaves a library newer than every source, header and the public header, and the
    build inputs include every .cu and .cuh/.h file of the source directory."""
    assert build_mod.up_to_date()
    names = {os.path.basename(f) for f in build_mod._inputs()}
    on_disk = {f for f in os.listdir(build_mod.CSRC) if f.endswith((".cu", ".cuh", ".h"))}
    assert on_disk <= names
    assert "flce.h" in names
