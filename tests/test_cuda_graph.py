"""The library's calls inside a captured CUDA graph.

Every call only enqueues work on the caller's stream and allocates no device memory, so a whole
training-step loss (forward and backward, or the single call) can be captured once with
torch.cuda.graph and replayed: no host work per step. Replays must reproduce the eager results
bit for bit (the kernels are deterministic and take their tiles from counters that the captured
memsets reset on every replay).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from lm_head_linear_02_gb300 import autograd as A  # noqa: E402
from lm_head_linear_02_gb300.inputs import make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


def _device_inputs(inp):
    x = torch.from_numpy(inp.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
    w = torch.from_numpy(inp.weight_bits.view(np.int16)).cuda().view(torch.bfloat16)
    return x, w, torch.from_numpy(inp.target).cuda()


def _two_calls(x, w, y, g):
    loss, lse, status = A.flce_forward(x, w, y, "mean")
    gx, gw, status = A.flce_backward(x, w, y, lse, g, "mean", status=status)
    return loss, lse, gx, gw, status


def _single_call(x, w, y, g):
    return A.flce_forward_backward(x, w, y, g, "mean")


@pytest.mark.parametrize("step", [_two_calls, _single_call], ids=["two_calls", "single_call"])
def test_graph_replay_matches_eager(step):
    inp = make_inputs("ragged", dtype="bf16", T=2048, seed=41)  # 2 token chunks, several tiles
    x, w, y = _device_inputs(inp)
    g = torch.full((1,), 1.0, dtype=torch.float32, device="cuda")
    eager = [t.clone() for t in step(x, w, y, g)]
    torch.cuda.synchronize()
    A.check_status(eager[-1])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on a side stream, as graph capture requires
        step(x, w, y, g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = step(x, w, y, g)
    for replay in range(3):
        for t in captured[:-1]:
            t.fill_(float("nan") if t.is_floating_point() else 0)  # replays must rewrite them
        graph.replay()
        torch.cuda.synchronize()
        A.check_status(captured[-1])
        for a, b in zip(eager[:-1], captured[:-1]):
            assert torch.equal(a, b), f"replay {replay} differs from the eager call"
