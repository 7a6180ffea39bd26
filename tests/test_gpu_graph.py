"""CUDA-graph capture of the decode hot path (-m gpu).

A decode loop replays one graph per step: the MoE layer (router, top-k,
permute, grouped expert kernels, combine) and chains of qGEMV calls are
captured once, then replayed with new activations copied into the captured
input buffers.  Every kernel of the library takes its inputs, outputs and
workspace from the caller and makes no allocation or host synchronisation, so
the replay must give the same bits as the eager calls (the kernels sum in a
fixed order), and every replayed output is also compared with the CPU oracle.
The last test captures a whole decode step of the DeepSeek-V3-shaped layer
(T = 1) between two GEMVs in one graph, as [KTransformers, §技术原理] runs one
graph launch per decode step, and checks each stage of every replay against
the oracle on the exact inputs that stage saw.
"""
import numpy as np
import pytest
import torch

import moe_layers
import synth
from gpu_util import TOL, dev_act, dev_bytes, rel_err
from moe_layers import ref_under_selection

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dq():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import dequant_gemv_moe_gb300 as dq
    return dq


def _capture(fn, warm=False):
    """fn captured on a new stream; warm: fn runs once on that stream first,
    outside capture (a layer with one-token experts beside the general kernels
    then also captures its side stream's branch)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        if warm:
            fn()
            torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    return g


@pytest.mark.parametrize("E,k,H,F,ns,T,xdt", [
    (16, 4, 1024, 512, 1, 1, 2),     # decode, one token, shared expert
    (16, 4, 1024, 512, 1, 8, 1),
    (4, 2, 512, 512, 0, 80, 1),      # ~40 tokens per expert: tcgen05 path inside
    # one-token experts (side stream) beside the general kernels (shared
    # expert, experts with two tokens), forked and joined inside the graph
    (64, 2, 1024, 512, 1, 4, 2),
])
def test_moe_layer_graph_replay(dq, orc, E, k, H, F, ns, T, xdt):
    w = synth.moe_weights(7700 + E + T, E, H, F, ns, 1)
    dev = {kk: (dev_bytes(v) if v is not None and v.dtype == np.uint8 else
                (torch.from_numpy(v).cuda() if v is not None else None)) for kk, v in w.items()}
    desc = dq.ops.make_desc(E, k, H, F, ns, 1, dev["router_W"], dev["w_gate"], dev["w_up"],
                            dev["w_down"], dev["sh_gate"], dev["sh_up"], dev["sh_down"])
    g = synth.streams(7800 + T, 3)
    xh = [synth.activations(g[i], (T, H), xdt) for i in range(3)]
    xs = [dev_act(a, xdt) for a in xh]
    refs = [dq.moe_forward(desc, x).clone() for x in xs]        # eager
    oref = [orc.moe_forward(1, E, k, H, F, ns, w["router_W"], w["w_gate"], w["w_up"],
                            w["w_down"], w["sh_gate"], w["sh_up"], w["sh_down"], a, xdt, T)
            for a in xh]
    xbuf = xs[0].clone()
    ybuf = torch.empty(T, H, dtype=torch.float32, device="cuda")
    ws = torch.empty(dq.moe_workspace_size(desc, T), dtype=torch.uint8, device="cuda")
    graph = _capture(lambda: dq.moe_forward(desc, xbuf, y=ybuf, ws=ws), warm=True)
    for i in (1, 2, 0, 1):
        xbuf.copy_(xs[i])
        graph.replay()
        torch.cuda.synchronize()
        assert dq.device_status() == 0
        np.testing.assert_array_equal(ybuf.cpu().numpy(), refs[i].cpu().numpy())
        assert _moe_err(orc, w, 1, E, k, H, F, ns, xh[i], xdt, ybuf.cpu().numpy(),
                        oref[i]) <= MOE_TOL


MOE_TOL = 2e-3


def _moe_err(orc, w, fmt, E, k, H, F, ns, x, xdt, y, oref, idx=None):
    """Relative error of a GPU layer output y against the oracle's (y, idx,
    gate, logits) = oref; tokens the GPU routed differently at a near-tie of
    the logits (idx given) are compared under the GPU's selection."""
    y_ref, idx_ref, _, L_ref = oref
    ref = y_ref.copy()
    if idx is not None:
        for t in range(x.shape[0]):
            if not np.array_equal(idx[t], idx_ref[t]):
                ref[t] = ref_under_selection(orc, fmt, w, E, k, H, F, ns, x, xdt, t, idx[t], L_ref)
    return rel_err(y, ref)


def test_qgemv_chain_graph_replay(dq, orc):
    # a decode layer's dependent GEMVs: the second reads the first's fp32 output
    g = synth.streams(7900, 4)
    N1, K1, N2 = 6144, 4096, 1024
    W1h = synth.quant_matrix(g[0], 1, N1, K1)
    W2h = synth.quant_matrix(g[1], 3, N2, N1)
    W1, W2 = dev_bytes(W1h), dev_bytes(W2h)
    xh = [synth.activations(g[2 + i], (1, K1), 1) for i in range(2)]
    xs = [dev_act(a, 1) for a in xh]

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
        y1 = y1b.cpu().numpy()
        np.testing.assert_array_equal(y1, refs[i][0].cpu().numpy())
        np.testing.assert_array_equal(y2b.cpu().numpy(), refs[i][1].cpu().numpy())
        # the oracle: the first GEMV on the fp16 input, the second on the
        # first's fp32 output as the GPU produced it
        assert rel_err(y1, orc.qgemv(1, W1h, N1, K1, xh[i], 1, 1)) <= TOL[1]
        assert rel_err(y2b.cpu().numpy(), orc.qgemv(3, W2h, N2, N1, y1, 0, 1)) <= TOL[0]


def test_decode_step_graph_deepseek(dq, orc):
    # one decode step of the DeepSeek-V3-shaped layer in one graph: an input
    # projection (Q4_K 7168 x 7168, bf16 x) -> bf16 -> the MoE layer (256
    # experts top-8 + 1 shared, T = 1) -> bf16 -> an output GEMV (Q8_0
    # 2048 x 7168), replayed with new activations; each stage is compared with
    # the oracle on the inputs it read, as the GPU produced them
    c = synth.MOE_DEEPSEEK
    E, k, H, F, ns, fmt = c["E"], c["top_k"], c["H"], c["F"], c["n_shared"], c["fmt"]
    w, dev, desc = moe_layers.deepseek()
    g = synth.streams(7950, 5)
    Wi = synth.quant_matrix(g[0], 1, H, H)
    Wo = synth.quant_matrix(g[1], 3, 2048, H)
    dWi, dWo = dev_bytes(Wi), dev_bytes(Wo)
    xbuf = torch.empty(1, H, dtype=torch.bfloat16, device="cuda")
    a = torch.empty(1, H, dtype=torch.float32, device="cuda")
    a16 = torch.empty(1, H, dtype=torch.bfloat16, device="cuda")
    m = torch.empty(1, H, dtype=torch.float32, device="cuda")
    m16 = torch.empty(1, H, dtype=torch.bfloat16, device="cuda")
    z = torch.empty(1, 2048, dtype=torch.float32, device="cuda")
    idx = torch.empty(1, k, dtype=torch.int32, device="cuda")
    gate = torch.empty(1, k, dtype=torch.float32, device="cuda")
    logits = torch.empty(1, E, dtype=torch.float32, device="cuda")
    ws = torch.empty(dq.moe_workspace_size(desc, 1), dtype=torch.uint8, device="cuda")
    import ctypes

    def step():
        dq.qgemv(1, dWi, H, H, xbuf, y=a, weights_early=True)
        a16.copy_(a)
        rc = dq.lib.dq_moe_forward(ctypes.byref(desc), ctypes.c_void_p(a16.data_ptr()), 2, 1,
                                   ctypes.c_void_p(m.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                   ws.numel(), ctypes.c_void_p(idx.data_ptr()),
                                   ctypes.c_void_p(gate.data_ptr()),
                                   ctypes.c_void_p(logits.data_ptr()),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, rc
        m16.copy_(m)
        dq.qgemv(3, dWo, 2048, H, m16, y=z, weights_early=True)

    xbuf.copy_(dev_act(synth.activations(g[2], (1, H), 2), 2))
    step()                                   # eager once (kernel attributes)
    torch.cuda.synchronize()
    graph = _capture(step)
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)
    for r in range(3):
        xh = synth.activations(g[2 + r], (1, H), 2)
        xbuf.copy_(dev_act(xh, 2))
        graph.replay()
        torch.cuda.synchronize()
        assert dq.device_status() == 0
        ah, a16h, mh, m16h, zh = (a.cpu().numpy(), bits(a16), m.cpu().numpy(), bits(m16),
                                  z.cpu().numpy())
        assert np.isfinite(zh).all()
        assert rel_err(ah, orc.qgemv(1, Wi, H, H, xh, 2, 1)) <= TOL[2]
        oref = orc.moe_forward(fmt, E, k, H, F, ns, w["router_W"], w["w_gate"], w["w_up"],
                               w["w_down"], w["sh_gate"], w["sh_up"], w["sh_down"], a16h, 2, 1)
        assert _moe_err(orc, w, fmt, E, k, H, F, ns, a16h, 2, mh, oref,
                        idx=idx.cpu().numpy()) <= MOE_TOL
        assert rel_err(zh, orc.qgemv(3, Wo, 2048, H, m16h, 2, 1)) <= TOL[2]
