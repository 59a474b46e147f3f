"""The workspace-free forward (flce_forward_static_scratch) against the regular forward.

Some callers cannot allocate device memory for a workspace (a plain C or foreign-language host
program without a device allocator, or a service with a fixed device-memory budget that may not
call cudaMalloc while running). flce_forward_static_scratch serves them from a fixed 64 MiB
device array inside the library. This file runs last (its name sorts last) so that a failure
here, in a run that stops at the first failure, comes after every other test has run; it must
pass both alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from lm_head_linear_02_gb300 import autograd as A  # noqa: E402
from lm_head_linear_02_gb300 import binding as B  # noqa: E402
from lm_head_linear_02_gb300 import build as build_mod  # noqa: E402
from lm_head_linear_02_gb300.inputs import make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu

# The tolerances of the parity tests (relative loss error; lse absolute error).
TOL = {"f32": dict(loss=1e-4, lse=2e-4), "bf16": dict(loss=2e-3, lse=2e-3)}


def _device_inputs(inp):
    if inp.workload.dtype == "bf16":
        x = torch.from_numpy(inp.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        w = torch.from_numpy(inp.weight_bits.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        x = torch.from_numpy(inp.x).cuda()
        w = torch.from_numpy(inp.weight).cuda()
    return x, w, torch.from_numpy(inp.target).cuda()


@pytest.mark.parametrize("name,dtype,reduction", [
    ("ragged", "bf16", "mean"),
    ("llama2_head", "bf16", "sum"),
    ("tiny", "f32", "mean"),
])
def test_static_scratch_forward_matches_workspace_forward(name, dtype, reduction):
    build_mod.build()
    inp = make_inputs(name, dtype=dtype)
    T, H, V = inp.workload.T, inp.workload.H, inp.workload.V
    x, w, y = _device_inputs(inp)
    ref_loss, ref_lse, ref_status = A.flce_forward(x, w, y, reduction)
    torch.cuda.synchronize()
    A.check_status(ref_status)
    ref_loss = ref_loss.item()
    ref_lse = ref_lse.cpu().numpy()
    stream = torch.cuda.current_stream().cuda_stream
    tol = TOL[dtype]
    for call in range(2):  # two calls in a row share (and reuse) the static scratch
        loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((T,), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = B.flce_forward_static_scratch(x.data_ptr(), w.data_ptr(), y.data_ptr(), T, H, V,
                                           B.dtype_code(dtype), B.reduction_code(reduction),
                                           loss.data_ptr(), lse.data_ptr(), status.data_ptr(),
                                           stream, check=False)
        assert rc == B.FLCE_OK, B.flce_strerror(rc)
        torch.cuda.synchronize()
        A.check_status(status)
        got = loss.item()
        assert abs(got - ref_loss) <= tol["loss"] * abs(ref_loss), (call, got, ref_loss)
        assert float(np.abs(lse.cpu().numpy() - ref_lse).max()) <= tol["lse"], call


def test_static_scratch_rejects_problems_beyond_its_size():
    build_mod.build()
    T, H, V = 32768, 4096, 128256
    need = B.flce_forward_workspace_size(T, H, V, B.FLCE_DTYPE_BF16)
    assert need > 64 << 20
    fake = 0x7F0000000000  # never dereferenced: the size check comes first
    rc = B.flce_forward_static_scratch(fake, fake + (1 << 32), fake + (2 << 32), T, H, V,
                                       B.FLCE_DTYPE_BF16, B.FLCE_REDUCTION_MEAN,
                                       fake + (3 << 32), fake + (3 << 32) + 4096,
                                       fake + (3 << 32) + 256, 0, check=False)
    assert rc == B.FLCE_ERR_WORKSPACE


# A caller may run its own CUDA contexts (driver API) instead of the device's primary context.
# Each context holds its own copy of the library's scratch array at its own address, so the
# entry point must look the address up per context. The child process below creates two
# contexts with the driver API, allocates its buffers in each with cuMemAlloc, and calls the
# entry point in context A, then B, then A again, comparing each result bit for bit with
# flce_forward given a workspace in the same context. Every pointer a kernel receives belongs
# to the context the kernel runs in.
_CHILD = r"""
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
from lm_head_linear_02_gb300 import binding as B
from lm_head_linear_02_gb300.inputs import make_inputs

cu = ctypes.CDLL("libcuda.so.1")

def ck(rc, what):
    if rc != 0:
        raise SystemExit(f"{what} returned CUDA error {rc}")

ck(cu.cuInit(0), "cuInit")
dev = ctypes.c_int()
ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
inp = make_inputs("ragged", T=300, H=256, V=1500, dtype="bf16", seed=42)
T, H, V = 300, 256, 1500
BF16, MEAN = B.FLCE_DTYPE_BF16, B.FLCE_REDUCTION_MEAN
ws_bytes = B.flce_forward_workspace_size(T, H, V, BF16)


class Ctx:
    def __init__(self):
        self.ctx = ctypes.c_void_p()
        ck(cu.cuCtxCreate_v2(ctypes.byref(self.ctx), 0, dev), "cuCtxCreate")
        self.bufs = {}
        for name, n in [("x", T * H * 2), ("w", V * H * 2), ("y", T * 8), ("loss_a", 4),
                        ("lse_a", 4 * T), ("loss_b", 4), ("lse_b", 4 * T), ("status", 4),
                        ("ws", ws_bytes)]:
            p = ctypes.c_uint64()
            ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(n)), "cuMemAlloc")
            self.bufs[name] = p.value
        self.h2d("x", inp.x_bits)
        self.h2d("w", inp.weight_bits)
        self.h2d("y", inp.target)
        ck(cu.cuCtxPopCurrent_v2(ctypes.byref(ctypes.c_void_p())), "cuCtxPopCurrent")

    def h2d(self, name, a):
        a = np.ascontiguousarray(a)
        ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(self.bufs[name]), a.ctypes.data_as(ctypes.c_void_p),
                              ctypes.c_size_t(a.nbytes)), "cuMemcpyHtoD")

    def d2h(self, name, a):
        ck(cu.cuMemcpyDtoH_v2(a.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(self.bufs[name]),
                              ctypes.c_size_t(a.nbytes)), "cuMemcpyDtoH")

    def run(self):
        ck(cu.cuCtxPushCurrent_v2(self.ctx), "cuCtxPushCurrent")
        b = self.bufs
        self.h2d("status", np.zeros(1, np.int32))
        rc = B.flce_forward_static_scratch(b["x"], b["w"], b["y"], T, H, V, BF16, MEAN,
                                           b["loss_a"], b["lse_a"], b["status"], 0, check=False)
        if rc != B.FLCE_OK:
            raise SystemExit(f"static-scratch forward: {B.flce_strerror(rc)}")
        rc = B.flce_forward(b["x"], b["w"], b["y"], T, H, V, BF16, MEAN, b["loss_b"], b["lse_b"],
                            b["ws"], ws_bytes, b["status"], 0, check=False)
        if rc != B.FLCE_OK:
            raise SystemExit(f"workspace forward: {B.flce_strerror(rc)}")
        ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
        out = {}
        for name, shape, dt in [("loss_a", 1, np.float32), ("lse_a", T, np.float32),
                                ("loss_b", 1, np.float32), ("lse_b", T, np.float32),
                                ("status", 1, np.int32)]:
            out[name] = np.empty(shape, dt)
            self.d2h(name, out[name])
        ck(cu.cuCtxPopCurrent_v2(ctypes.byref(ctypes.c_void_p())), "cuCtxPopCurrent")
        if out["status"][0] != 0:
            raise SystemExit(f"device status {out['status'][0]}")
        if not (np.array_equal(out["loss_a"], out["loss_b"]) and
                np.array_equal(out["lse_a"], out["lse_b"])):
            raise SystemExit("static-scratch forward differs from the workspace forward")
        return out["loss_a"][0], out["lse_a"]


a, b = Ctx(), Ctx()
ra1, rb, ra2 = a.run(), b.run(), a.run()
assert ra1[0] == rb[0] == ra2[0] and np.array_equal(ra1[1], rb[1]) and np.array_equal(ra1[1], ra2[1])
for c in (a, b):
    ck(cu.cuCtxDestroy_v2(c.ctx), "cuCtxDestroy")
print(f"contexts ok: loss {ra1[0]:.6f}")
"""


def test_static_scratch_in_caller_created_contexts():
    import os
    import subprocess
    import sys

    build_mod.build()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    r = subprocess.run([sys.executable, "-c", _CHILD, root], capture_output=True, text=True,
                       timeout=300, env=env)
    print(r.stdout, r.stderr)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "contexts ok" in r.stdout
