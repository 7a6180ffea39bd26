"""dq_moe_forward_noalloc against dq_moe_forward (-m gpu).

The allocation-free entry point serves callers that cannot allocate device
memory (a host framework that owns all of it and gives no workspace hook, or
a decode loop that must not allocate on its hot path).  Its scratch is a
fixed array inside the library.  This test calls both entry points through the
C ABI on the same inputs, twice in a row for the allocation-free one (the
array keeps the previous call's contents), and checks that the outputs agree
within the MoE-layer tolerance.  It also checks that a token count whose scratch
would not fit in the array is refused before anything is launched.  The file
is collected last, so a run that stops at its first failure has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import dev_act, dev_bytes, rel_err

pytestmark = pytest.mark.gpu

MOE_TOL = 2e-3


def _layer(dq, fmt, E, k, H, F, ns, seed):
    w = synth.moe_weights(seed, E, H, F, ns, fmt)
    dev = {kk: (dev_bytes(v) if v is not None and v.dtype == np.uint8 else
                (torch.from_numpy(v).cuda() if v is not None else None)) for kk, v in w.items()}
    desc = dq.ops.make_desc(E, k, H, F, ns, fmt, dev["router_W"], dev["w_gate"], dev["w_up"],
                            dev["w_down"], dev["sh_gate"], dev["sh_up"], dev["sh_down"])
    return desc, dev


def _noalloc(dq, desc, x, xdt, T, y, idx):
    P = ctypes.c_void_p
    return dq.lib.dq_moe_forward_noalloc(ctypes.byref(desc), P(x.data_ptr()), xdt, T,
                                         P(y.data_ptr()), P(idx.data_ptr()), None, None,
                                         P(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("fmt,E,k,H,F,ns,T,xdt", [
    (1, 8, 2, 512, 1024, 1, 5, 1),
    (3, 16, 4, 1024, 512, 0, 16, 2),
    # one-token experts beside the shared expert's group: dq_moe_forward may
    # fork a second stream here, the allocation-free entry stays on one
    (1, 64, 2, 1024, 512, 1, 4, 2),
])
def test_noalloc_matches_workspace_entry(fmt, E, k, H, F, ns, T, xdt):
    assert torch.cuda.is_available(), "GPU test"
    import dequant_gemv_moe_gb300 as dq
    desc, dev = _layer(dq, fmt, E, k, H, F, ns, seed=8800 + E + T)
    g = synth.streams(8900 + T, 2)
    xa = dev_act(synth.activations(g[0], (T, H), xdt), xdt)
    xb = dev_act(synth.activations(g[1], (T, H), xdt), xdt)
    # reference: the entry point with a caller-provided workspace
    ref_a, idx_ref, _, _ = dq.moe_forward(desc, xa, want_routing=True)
    ref_b = dq.moe_forward(desc, xb)
    # two calls in a row on the shared array, different inputs
    y = torch.empty(T, H, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    assert _noalloc(dq, desc, xa, xdt, T, y, idx) == 0
    ya = y.cpu().numpy()
    assert np.array_equal(idx.cpu().numpy(), idx_ref.cpu().numpy())
    assert _noalloc(dq, desc, xb, xdt, T, y, idx) == 0
    yb = y.cpu().numpy()
    assert dq.device_status() == 0
    assert rel_err(ya, ref_a.cpu().numpy()) <= MOE_TOL
    assert rel_err(yb, ref_b.cpu().numpy()) <= MOE_TOL


def test_noalloc_rejects_oversized_scratch():
    import dequant_gemv_moe_gb300 as dq
    desc, dev = _layer(dq, 1, 8, 2, 512, 1024, 1, seed=8700)
    T = 4096                               # needs far more than the fixed array
    assert dq.moe_workspace_size(desc, T) > (32 << 20)
    x = torch.zeros(T, 512, dtype=torch.float16, device="cuda")
    y = torch.full((T, 512), 7.0, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, 2, dtype=torch.int32, device="cuda")
    assert _noalloc(dq, desc, x, 1, T, y, idx) == -4          # DQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())                             # nothing was launched
