"""The forward pass captured in a CUDA graph: the three kernels of mha_forward
(and its error-word reset) recorded once on static buffers and replayed,
which removes the host's launch work from every call of a serving loop.
Replays must give exactly the eager result."""

import pytest
import torch

from head_scaled_dot_gb300 import mha, workloads
from helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return mha.load()


@pytest.mark.parametrize("idx", [1, 2])
def test_forward_replayed_from_a_cuda_graph_matches_eager(idx):
    w = workloads.WORKLOADS[idx]
    inp = workloads.make_inputs(w)
    t = to_dev(inp)
    dev = t["X_q"].device
    X = t["X_q"].clone()  # static input buffer of the graph
    Y = torch.empty((w.B, w.n_q, w.d_o), dtype=X.dtype, device=dev)
    ws = torch.empty(mha.workspace_size(w.B, w.n_q, w.n_k, w.d_model, w.h, w.d_h, w.d_vh, w.d_o,
                                        w.dtype), dtype=torch.uint8, device=dev)

    def call():
        mha.forward(X, None, t["W_Q"], t["W_K"], t["W_V"], t["W_O"], w.h, w.d_h, w.d_vh, w.c,
                    w.mask, inp["valid_len"], out=Y, workspace=ws, check=False)

    # eager reference (also sets the kernels' launch attributes before capture)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = Y.clone()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    # 1. a replay on the same input gives the eager bits
    Y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Y, eager)
    # 2. new input in the graph's buffer: the replay computes on it, and
    # matches an eager call on the same input
    X.copy_(torch.flip(t["X_q"], dims=[0]))
    g.replay()
    torch.cuda.synchronize()
    replayed = Y.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(replayed, Y)
    assert not torch.equal(replayed, eager)
    assert mha.get_device_error(ws) == 0
