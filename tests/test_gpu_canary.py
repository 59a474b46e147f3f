"""Nothing is written outside the caller's buffers, and inputs are never written.

compute-sanitizer is not available here, so out-of-bounds writes are caught with canaries:
every output buffer and the workspace are carved out of a larger allocation whose margins hold
a byte pattern, the calls run on shapes ragged against every tile size (token rows not a
multiple of the 32-row store blocks, hidden and vocabulary sizes not multiples of the 256-wide
tiles), and afterwards the margins must be intact and the inputs bit-identical
(KernelIndex "Semantics": inputs are neither modified nor aliased).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from lm_head_linear_02_gb300 import binding as B  # noqa: E402
from lm_head_linear_02_gb300.inputs import make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu

PAD = 4096  # bytes of canary on each side (a multiple of 256 keeps the interior aligned)
CANARY = 0xA5


class Guarded:
    """A device buffer of `nbytes` with canary margins on both sides."""

    def __init__(self, nbytes):
        self.nbytes = int(nbytes)
        self.raw = torch.full((self.nbytes + 2 * PAD,), CANARY, dtype=torch.uint8, device="cuda")

    @property
    def ptr(self):
        return self.raw.data_ptr() + PAD

    def margins_intact(self):
        head = self.raw[:PAD]
        tail = self.raw[PAD + self.nbytes:]
        return bool((head == CANARY).all()) and bool((tail == CANARY).all())


def _inputs(T, H, V, seed):
    inp = make_inputs("tiny", T=T, H=H, V=V, dtype="bf16", seed=seed)
    x = torch.from_numpy(inp.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    w = torch.from_numpy(inp.weight_bits.view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.from_numpy(inp.target).cuda()
    return x, w, y


@pytest.mark.parametrize("T,H,V", [
    (1269, 1000, 10000),  # the ragged Liger shape: 1269 = 39 x 32 + 21 rows
    (600, 264, 513),      # single call with a ragged second chunk; V just past 2 tiles
    (33, 72, 300),        # rows in one partial 32-row block; H not a multiple of 64
])
@pytest.mark.parametrize("schedule", ["two_calls", "single_call"])
def test_no_writes_outside_outputs_and_inputs_unchanged(T, H, V, schedule):
    x, w, y = _inputs(T, H, V, seed=T + H)
    x0, w0, y0 = x.clone(), w.clone(), y.clone()
    dt, red = B.FLCE_DTYPE_BF16, B.FLCE_REDUCTION_MEAN
    loss, lse = Guarded(4), Guarded(4 * T)
    gx, gw = Guarded(2 * T * H), Guarded(2 * V * H)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gl = torch.ones(1, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    if schedule == "two_calls":
        fws = B.flce_forward_workspace_size(T, H, V, dt)
        bws = B.flce_backward_workspace_size(T, H, V, dt)
        ws_f, ws_b = Guarded(fws), Guarded(bws)
        B.flce_forward(x.data_ptr(), w.data_ptr(), y.data_ptr(), T, H, V, dt, red, loss.ptr,
                       lse.ptr, ws_f.ptr, fws, status.data_ptr(), stream)
        B.flce_backward(x.data_ptr(), w.data_ptr(), y.data_ptr(), lse.ptr, T, H, V, dt, red,
                        gl.data_ptr(), gx.ptr, gw.ptr, ws_b.ptr, bws, status.data_ptr(), stream)
        workspaces = [ws_f, ws_b]
    else:
        fbs = B.flce_forward_backward_workspace_size(T, H, V, dt)
        ws = Guarded(fbs)
        B.flce_forward_backward(x.data_ptr(), w.data_ptr(), y.data_ptr(), T, H, V, dt, red,
                                gl.data_ptr(), loss.ptr, lse.ptr, gx.ptr, gw.ptr, ws.ptr, fbs,
                                status.data_ptr(), stream)
        workspaces = [ws]
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for name, buf in [("loss", loss), ("lse", lse), ("grad_x", gx), ("grad_weight", gw)]:
        assert buf.margins_intact(), f"write outside {name}"
    for i, buf in enumerate(workspaces):
        assert buf.margins_intact(), f"write outside workspace {i}"
    assert torch.equal(x, x0) and torch.equal(w, w0) and torch.equal(y, y0), "an input changed"
    # the outputs were written (no canary byte pattern left in them)
    loss_v = loss.raw[PAD:PAD + 4].view(torch.float32).item()
    assert np.isfinite(loss_v) and loss_v > 0
