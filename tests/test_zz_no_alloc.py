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
