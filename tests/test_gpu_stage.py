"""dq_stage: the library's copy kernel between page-locked host memory and
device memory (-m gpu).  The bytes must arrive unchanged in both directions,
inside a CUDA graph after a GEMV (the copy waits for the kernel before it),
and bad arguments are refused before anything is launched."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import TOL, dev_bytes, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dq():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import dequant_gemv_moe_gb300 as dq
    return dq


@pytest.mark.parametrize("nbytes", [16, 4096, 53248, 172032, 3 << 20])
def test_stage_round_trip(dq, nbytes):
    rng = np.random.default_rng(nbytes)
    h = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    dq.stage(d, h)
    dq.stage(back, d)
    torch.cuda.synchronize()
    assert torch.equal(back, h)
    d2 = torch.empty_like(d)
    dq.stage(d2, d)                                       # device to device
    torch.cuda.synchronize()
    assert torch.equal(d2.cpu(), h)


def test_stage_in_a_decode_graph(dq, orc):
    # upload x, one GEMV, read y back, all in one graph replayed with new host x
    N, K = 4096, 4096
    g = synth.streams(7600, 3)
    W = synth.quant_matrix(g[0], 1, N, K)
    dW = dev_bytes(W)
    hx = torch.empty(1, K, dtype=torch.float16).pin_memory()
    hy = torch.empty(1, N, dtype=torch.float32).pin_memory()
    x = torch.empty(1, K, dtype=torch.float16, device="cuda")
    y = torch.empty(1, N, dtype=torch.float32, device="cuda")

    def step():
        dq.stage(x, hx)
        dq.qgemv(1, dW, N, K, x, y=y, weights_early=True)
        dq.stage(hy, y)

    hx.copy_(torch.from_numpy(synth.activations(g[1], (1, K), 1)))
    step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(gr, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for r in range(3):
        xh = synth.activations(synth.streams(7700 + r, 1)[0], (1, K), 1)
        hx.copy_(torch.from_numpy(xh))
        gr.replay()
        torch.cuda.synchronize()
        assert rel_err(hy.numpy(), orc.qgemv(1, W, N, K, xh, 1, 1)) <= TOL[1]


def test_stage_argument_errors(dq):
    f = dq.lib.dq_stage
    d = torch.empty(64, dtype=torch.uint8, device="cuda")
    P = ctypes.c_void_p
    assert f(None, P(d.data_ptr()), 16, None) == -1
    assert f(P(d.data_ptr()), P(d.data_ptr() + 32), 0, None) == -1
    assert f(P(d.data_ptr()), P(d.data_ptr() + 32), 24, None) == -2        # size
    assert f(P(d.data_ptr() + 8), P(d.data_ptr() + 32), 16, None) == -2    # dst alignment
    assert f(P(d.data_ptr()), P(d.data_ptr() + 16), 32, None) == -1        # overlap
