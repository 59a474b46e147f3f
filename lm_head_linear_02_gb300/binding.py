"""ctypes binding of libflce (argument marshalling only).

Every name here mirrors a C entry point of ``include/flce.h``; each function converts Python ints
and device/host addresses to C types, calls the library and turns a negative return code into a
``FlceError``. No step of the computation happens in Python. If ``libflce.so`` has not been built
the first call raises ``FlceNotBuilt``: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "FlceError", "FlceNotBuilt", "lib", "lib_path",
    "FLCE_OK", "FLCE_ERR_ARG", "FLCE_ERR_UNSUPPORTED", "FLCE_ERR_WORKSPACE", "FLCE_ERR_ALIAS",
    "FLCE_ERR_CUDA", "FLCE_STATUS_TARGET_RANGE", "FLCE_STATUS_TIMEOUT",
    "FLCE_DTYPE_BF16", "FLCE_DTYPE_F32", "FLCE_REDUCTION_SUM", "FLCE_REDUCTION_MEAN",
    "FLCE_REDUCTION_NONE",
    "flce_forward_workspace_size", "flce_backward_workspace_size", "flce_backward_slab_width",
    "flce_set_backward_slab_width", "flce_forward", "flce_backward", "flce_strerror",
    "flce_forward_backward", "flce_forward_backward_workspace_size",
    "flce_forward_backward_chunk_tokens", "flce_test_withhold_signal",
    "flce_version", "flce_timing_enable", "flce_timing_read", "TIMING_ROLES",
    "flce_set_tuning", "flce_get_tuning", "FLCE_TUNE_RASTER_ROWS", "FLCE_TUNE_SM_PAIRS", "FLCE_TUNE_WIDE_TILES", "FLCE_TUNE_RASTER_VOCAB", "FLCE_TUNE_SPLIT_EPILOGUE", "FLCE_TUNE_CHUNK_BYTES", "FLCE_TUNE_ORDERED_DRAIN", "FLCE_ROLE_FORWARD", "FLCE_ROLE_DZ", "FLCE_ROLE_GRADS",
    "dtype_code", "reduction_code",
]

FLCE_OK = 0
FLCE_ERR_ARG = -1
FLCE_ERR_UNSUPPORTED = -2
FLCE_ERR_WORKSPACE = -3
FLCE_ERR_ALIAS = -4
FLCE_ERR_CUDA = -5
FLCE_STATUS_TARGET_RANGE = 1
FLCE_STATUS_TIMEOUT = 2
FLCE_DTYPE_BF16 = 0
FLCE_DTYPE_F32 = 1
FLCE_REDUCTION_SUM = 0
FLCE_REDUCTION_MEAN = 1
FLCE_REDUCTION_NONE = 2

_HERE = os.path.dirname(os.path.abspath(__file__))


class FlceError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {flce_strerror(code)} (code {code})")


class FlceNotBuilt(RuntimeError):
    pass


_LIB = None


def lib_path() -> str:
    return os.path.join(_HERE, "libflce.so")


def lib() -> ctypes.CDLL:
    """Load libflce.so (once). Raises FlceNotBuilt when it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise FlceNotBuilt(f"{path} is missing: build it with __graft_entry__.build() "
                           "or python -m lm_head_linear_02_gb300.build")
    L = ctypes.CDLL(path)
    i64, sz, vp, ci = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
    L.flce_forward_workspace_size.argtypes = [i64, i64, i64, ci]
    L.flce_forward_workspace_size.restype = sz
    L.flce_backward_workspace_size.argtypes = [i64, i64, i64, ci]
    L.flce_backward_workspace_size.restype = sz
    L.flce_backward_slab_width.argtypes = [i64, i64, i64, ci]
    L.flce_backward_slab_width.restype = i64
    L.flce_set_backward_slab_width.argtypes = [i64]
    L.flce_set_backward_slab_width.restype = ci
    L.flce_forward.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, vp, vp, vp, sz, vp, vp]
    L.flce_forward.restype = ci
    L.flce_backward.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci, vp, vp, vp, vp, sz, vp, vp]
    L.flce_backward.restype = ci
    L.flce_forward_backward_workspace_size.argtypes = [i64, i64, i64, ci]
    L.flce_forward_backward_workspace_size.restype = sz
    L.flce_forward_backward_chunk_tokens.argtypes = [i64, i64, i64, ci]
    L.flce_forward_backward_chunk_tokens.restype = i64
    L.flce_forward_backward.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, vp, vp, vp, vp, vp, vp,
                                        sz, vp, vp]
    L.flce_forward_backward.restype = ci
    L.flce_timing_enable.argtypes = [ci]
    L.flce_timing_enable.restype = ci
    L.flce_timing_read.argtypes = [ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)]
    L.flce_timing_read.restype = ci
    L.flce_get_tuning.argtypes = [ci, ctypes.POINTER(i64)]
    L.flce_get_tuning.restype = ci
    L.flce_set_tuning.argtypes = [ci, i64]
    L.flce_set_tuning.restype = ci
    L.flce_test_withhold_signal.argtypes = []
    L.flce_test_withhold_signal.restype = ci
    L.flce_strerror.argtypes = [ci]
    L.flce_strerror.restype = ctypes.c_char_p
    L.flce_version.argtypes = []
    L.flce_version.restype = ci
    _LIB = L
    return L


def dtype_code(name: str) -> int:
    return {"bf16": FLCE_DTYPE_BF16, "f32": FLCE_DTYPE_F32}[name]


def reduction_code(name: str) -> int:
    return {"sum": FLCE_REDUCTION_SUM, "mean": FLCE_REDUCTION_MEAN,
            "none": FLCE_REDUCTION_NONE}[name]


def _check(rc: int, where: str) -> int:
    if rc != FLCE_OK:
        raise FlceError(rc, where)
    return rc


def flce_test_withhold_signal() -> None:
    """Testing aid: the next single-SM contraction launch ends with FLCE_STATUS_TIMEOUT."""
    _check(int(lib().flce_test_withhold_signal()), "flce_test_withhold_signal")


def flce_strerror(code: int) -> str:
    return lib().flce_strerror(int(code)).decode()


def flce_version() -> int:
    return int(lib().flce_version())


def flce_forward_workspace_size(T: int, H: int, V: int, dtype: int) -> int:
    return int(lib().flce_forward_workspace_size(T, H, V, dtype))


def flce_backward_workspace_size(T: int, H: int, V: int, dtype: int) -> int:
    return int(lib().flce_backward_workspace_size(T, H, V, dtype))


def flce_backward_slab_width(T: int, H: int, V: int, dtype: int) -> int:
    return int(lib().flce_backward_slab_width(T, H, V, dtype))


def flce_set_backward_slab_width(vc: int) -> None:
    """Force the backward vocab slab width (multiple of 256); 0 restores the automatic choice."""
    _check(int(lib().flce_set_backward_slab_width(int(vc))), "flce_set_backward_slab_width")


TIMING_ROLES = ("forward", "backward_dz", "backward_grad_weight", "backward_grad_x",
                "backward_grads")
FLCE_TUNE_RASTER_ROWS = 1
FLCE_TUNE_SM_PAIRS = 2
FLCE_TUNE_WIDE_TILES = 3
FLCE_TUNE_RASTER_VOCAB = 4
FLCE_TUNE_SPLIT_EPILOGUE = 5
FLCE_TUNE_CHUNK_BYTES = 6
FLCE_TUNE_ORDERED_DRAIN = 7
FLCE_ROLE_FORWARD = 1
FLCE_ROLE_DZ = 2
FLCE_ROLE_GRADS = 4


def flce_get_tuning(key: int) -> int:
    """Effective value of a tuning key on the current device (automatic choices resolved)."""
    v = ctypes.c_int64()
    _check(int(lib().flce_get_tuning(int(key), ctypes.byref(v))), "flce_get_tuning")
    return int(v.value)


def flce_set_tuning(key: int, value: int) -> None:
    """Set a process-wide tuning value (FLCE_TUNE_*); affects speed only, never results."""
    _check(int(lib().flce_set_tuning(int(key), int(value))), "flce_set_tuning")


def flce_timing_enable(on: bool) -> None:
    """Bracket every tensor-core kernel launch with CUDA events (benchmarking aid)."""
    _check(int(lib().flce_timing_enable(1 if on else 0)), "flce_timing_enable")


def flce_timing_read() -> dict:
    """Launch counts and summed milliseconds per kernel role since the previous read."""
    counts = (ctypes.c_int64 * len(TIMING_ROLES))()
    ms = (ctypes.c_double * len(TIMING_ROLES))()
    _check(int(lib().flce_timing_read(counts, ms)), "flce_timing_read")
    return {r: (int(counts[i]), float(ms[i])) for i, r in enumerate(TIMING_ROLES)}


def flce_forward(x: int, weight: int, target: int, T: int, H: int, V: int, dtype: int,
                 reduction: int, loss: int, lse: int, workspace: int, workspace_bytes: int,
                 status: int, stream: int, check: bool = True) -> int:
    """Enqueue the forward. Pointer arguments are integer device addresses."""
    rc = lib().flce_forward(x, weight, target, T, H, V, dtype, reduction, loss, lse, workspace,
                            workspace_bytes, status, stream)
    return _check(rc, "flce_forward") if check else rc


def flce_backward(x: int, weight: int, target: int, lse: int, T: int, H: int, V: int,
                  dtype: int, reduction: int, grad_loss: int, grad_x: int, grad_weight: int,
                  workspace: int, workspace_bytes: int, status: int, stream: int,
                  check: bool = True) -> int:
    """Enqueue the backward. Pointer arguments are integer device addresses."""
    rc = lib().flce_backward(x, weight, target, lse, T, H, V, dtype, reduction, grad_loss,
                             grad_x, grad_weight, workspace, workspace_bytes, status, stream)
    return _check(rc, "flce_backward") if check else rc


def flce_forward_backward_workspace_size(T: int, H: int, V: int, dtype: int) -> int:
    return int(lib().flce_forward_backward_workspace_size(T, H, V, dtype))


def flce_forward_backward_chunk_tokens(T: int, H: int, V: int, dtype: int) -> int:
    return int(lib().flce_forward_backward_chunk_tokens(T, H, V, dtype))


def flce_forward_backward(x: int, weight: int, target: int, T: int, H: int, V: int, dtype: int,
                          reduction: int, grad_loss: int, loss: int, lse: int, grad_x: int,
                          grad_weight: int, workspace: int, workspace_bytes: int, status: int,
                          stream: int, check: bool = True) -> int:
    """Enqueue forward and backward in one call (upstream gradient known in advance)."""
    rc = lib().flce_forward_backward(x, weight, target, T, H, V, dtype, reduction, grad_loss,
                                     loss, lse, grad_x, grad_weight, workspace, workspace_bytes,
                                     status, stream)
    return _check(rc, "flce_forward_backward") if check else rc


def flce_forward_static_scratch(x: int, weight: int, target: int, T: int, H: int, V: int,
                                dtype: int, reduction: int, loss: int, lse: int, status: int,
                                stream: int, check: bool = True) -> int:
    """Enqueue the forward with the library's static device scratch (no workspace argument).

    For callers that cannot allocate device memory; see include/flce.h for its size limit and
    the sharing rules of the static scratch array.
    """
    L = lib()
    fn = L.flce_forward_static_scratch
    if fn.argtypes is None:
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        fn.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, vp, vp, vp, vp]
        fn.restype = ci
    rc = fn(x, weight, target, T, H, V, dtype, reduction, loss, lse, status, stream)
    return _check(rc, "flce_forward_static_scratch") if check else rc
