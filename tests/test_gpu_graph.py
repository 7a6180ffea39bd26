"""CUDA-graph capture of the decode hot path (-m gpu).

A decode loop replays one graph per step: the MoE layer (router, top-k,
permute, grouped expert kernels, combine) and chains of qGEMV calls are
captured once, then replayed with new activations copied into the captured
input buffers.  Every kernel of the library takes its inputs, outputs and
workspace from the caller and makes no allocation or host synchronisation, so
the replay must give the same bits as the eager calls (the kernels sum in a
fixed order).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import dev_act, dev_bytes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dq():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import dequant_gemv_moe_gb300 as dq
    return dq


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    return g


@pytest.mark.parametrize("E,k,H,F,ns,T,xdt", [
    (16, 4, 1024, 512, 1, 1, 2),     # decode, one token, shared expert
    (16, 4, 1024, 512, 1, 8, 1),
    (4, 2, 512, 512, 0, 80, 1),      # ~40 tokens per expert: tcgen05 path inside
])
def test_moe_layer_graph_replay(dq, E, k, H, F, ns, T, xdt):
    w = synth.moe_weights(7700 + E + T, E, H, F, ns, 1)
    dev = {kk: (dev_bytes(v) if v is not None and v.dtype == np.uint8 else
                (torch.from_numpy(v).cuda() if v is not None else None)) for kk, v in w.items()}
    desc = dq.ops.make_desc(E, k, H, F, ns, 1, dev["router_W"], dev["w_gate"], dev["w_up"],
                            dev["w_down"], dev["sh_gate"], dev["sh_up"], dev["sh_down"])
    g = synth.streams(7800 + T, 3)
    xs = [dev_act(synth.activations(g[i], (T, H), xdt), xdt) for i in range(3)]
    refs = [dq.moe_forward(desc, x).clone() for x in xs]        # eager
    xbuf = xs[0].clone()
    ybuf = torch.empty(T, H, dtype=torch.float32, device="cuda")
    ws = torch.empty(dq.moe_workspace_size(desc, T), dtype=torch.uint8, device="cuda")
    graph = _capture(lambda: dq.moe_forward(desc, xbuf, y=ybuf, ws=ws))
    for i in (1, 2, 0, 1):
        xbuf.copy_(xs[i])
        graph.replay()
        torch.cuda.synchronize()
        assert dq.device_status() == 0
        np.testing.assert_array_equal(ybuf.cpu().numpy(), refs[i].cpu().numpy())


def test_qgemv_chain_graph_replay(dq):
    # a decode layer's dependent GEMVs: the second reads the first's fp32 output
    g = synth.streams(7900, 4)
    N1, K1, N2 = 6144, 4096, 1024
    W1 = dev_bytes(synth.quant_matrix(g[0], 1, N1, K1))
    W2 = dev_bytes(synth.quant_matrix(g[1], 3, N2, N1))
    xs = [dev_act(synth.activations(g[2 + i], (1, K1), 1), 1) for i in range(2)]

    def chain(x, y1, y2):
        dq.qgemv(1, W1, N1, K1, x, y=y1, weights_early=True)
        dq.qgemv(3, W2, N2, N1, y1, y=y2, weights_early=True)   # fp32 activations

    refs = []
    for x in xs:
        y1 = torch.empty(1, N1, device="cuda")
        y2 = torch.empty(1, N2, device="cuda")
        chain(x, y1, y2)
        refs.append((y1.clone(), y2.clone()))
    xbuf = xs[0].clone()
    y1b = torch.empty(1, N1, device="cuda")
    y2b = torch.empty(1, N2, device="cuda")
    graph = _capture(lambda: chain(xbuf, y1b, y2b))
    for i in (1, 0, 1):
        xbuf.copy_(xs[i])
        graph.replay()
        torch.cuda.synchronize()
        assert dq.device_status() == 0
        np.testing.assert_array_equal(y1b.cpu().numpy(), refs[i][0].cpu().numpy())
        np.testing.assert_array_equal(y2b.cpu().numpy(), refs[i][1].cpu().numpy())
