"""Expert streaming (-m gpu): routed experts in page-locked host memory, a
device cache of expert slots, copies in chunks overlapped with the grouped
kernels.  Every streamed output is compared with the oracle, and with
dq_moe_forward's within the layer's tolerance (the streamed layer keeps every
expert on the grouped mma.sync kernel; the resident one runs one-token experts
on the block-diagonal kernel and experts above 32 tokens on the tensor-core
GEMM).  The cache counters must
account for every expert of every call."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import dev_act, dev_bytes, rel_err
from moe_layers import ref_under_selection
from test_gpu_moe import MOE_TOL, NVFP4, Q4_K, Q8_0, dq  # noqa: F401

pytestmark = pytest.mark.gpu


def _layer(seed, fmt, E, H, F, ns):
    w = synth.moe_weights(seed, E, H, F, ns, fmt)
    dev = {k: (dev_bytes(v) if v is not None and v.dtype == np.uint8 else
               (torch.from_numpy(v).cuda() if v is not None else None)) for k, v in w.items()}
    host = {k: torch.from_numpy(w[k]).pin_memory() for k in ("w_gate", "w_up", "w_down")}
    return w, dev, host


@pytest.mark.parametrize("fmt,E,k,H,F,ns,phases,Ts", [
    (Q4_K, 16, 2, 1024, 512, 1, 2, [1, 2, 1, 2, 2, 1]),
    (Q4_K, 16, 4, 512, 512, 0, 1, [2, 1, 2]),          # all copies before the compute
    (Q4_K, 32, 2, 1024, 1024, 1, 4, [4, 4, 3, 4]),      # several chunks per call
    (Q8_0, 8, 2, 768, 512, 1, 3, [3, 2, 3]),
    (NVFP4, 16, 2, 512, 512, 0, 2, [2, 2, 1]),
])
def test_streamed_equals_resident(dq, orc, fmt, E, k, H, F, ns, phases, Ts):
    w, dev, host = _layer(9100 + E + F, fmt, E, H, F, ns)
    maxT = max(Ts)
    cache = dq.ExpertCache(E, k, H, F, ns, fmt, dev["router_W"], host["w_gate"], host["w_up"],
                           host["w_down"], dev["sh_gate"], dev["sh_up"], dev["sh_down"],
                           max_tokens=maxT, phases=phases)
    desc = dq.ops.make_desc(E, k, H, F, ns, fmt, dev["router_W"], dev["w_gate"], dev["w_up"],
                            dev["w_down"], dev["sh_gate"], dev["sh_up"], dev["sh_down"])
    qk, nb = synth.BLOCK[fmt]
    expert_bytes = 2 * F * (H // qk) * nb + H * (F // qk) * nb
    g = synth.streams(9200 + E, len(Ts))
    distinct = 0
    for i, T in enumerate(Ts):
        xh = synth.activations(g[i], (T, H), 1)
        x = dev_act(xh, 1)
        y_s = cache.forward(x)
        y_r, idx, _, _ = dq.moe_forward(desc, x, want_routing=True)
        torch.cuda.synchronize()
        assert dq.device_status() == 0
        ys, yr = y_s.cpu().numpy(), y_r.cpu().numpy()
        # the streamed layer keeps every expert on the grouped mma.sync kernel,
        # the resident one runs one-token experts on the block-diagonal kernel:
        # both match the oracle, and each other within the layer's tolerance
        y_ref, idx_ref, _, L_ref = orc.moe_forward(fmt, E, k, H, F, ns, w["router_W"],
                                                   w["w_gate"], w["w_up"], w["w_down"],
                                                   w["sh_gate"], w["sh_up"], w["sh_down"], xh, 1, T)
        ig = idx.cpu().numpy()
        for t in range(T):   # a near-tie routed differently: the oracle under that selection
            if not np.array_equal(ig[t], idx_ref[t]):
                y_ref[t] = ref_under_selection(orc, fmt, w, E, k, H, F, ns, xh, 1, t, ig[t], L_ref)
        assert rel_err(ys, y_ref) <= MOE_TOL
        assert rel_err(yr, y_ref) <= MOE_TOL
        assert rel_err(ys, yr) <= MOE_TOL
        distinct += len(np.unique(idx.cpu().numpy()))
    st = cache.stats()
    assert st["hits"] + st["misses"] == distinct
    assert st["bytes_copied"] == st["misses"] * expert_bytes
    assert st["misses"] >= len(np.unique(idx.cpu().numpy()))   # at least the first call's
    cache.close()


def test_streamed_lru_reuse(dq):
    # the same tokens twice: the second call finds every expert in the cache
    E, k, H, F = 32, 2, 512, 512
    w, dev, host = _layer(9300, Q4_K, E, H, F, 0)
    cache = dq.ExpertCache(E, k, H, F, 0, Q4_K, dev["router_W"], host["w_gate"], host["w_up"],
                           host["w_down"], max_tokens=4, slots=8, phases=2)
    x = dev_act(synth.activations(synth.streams(9301, 1)[0], (4, H), 1), 1)
    y1 = cache.forward(x)
    s1 = cache.stats()
    y2 = cache.forward(x)
    s2 = cache.stats()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y1.cpu().numpy(), y2.cpu().numpy())
    assert s2["misses"] == s1["misses"] and s2["hits"] - s1["hits"] == s1["misses"]
    cache.close()


def test_streamed_wide_against_oracle(dq, orc):
    # experts above 32 tokens: the streamed layer keeps them on the grouped
    # kernel (the resident one takes the tensor-core GEMM), so the check is
    # against the oracle
    E, k, H, F, ns, T = 4, 2, 512, 512, 1, 40
    w, dev, host = _layer(9400, Q4_K, E, H, F, ns)
    cache = dq.ExpertCache(E, k, H, F, ns, Q4_K, dev["router_W"], host["w_gate"], host["w_up"],
                           host["w_down"], dev["sh_gate"], dev["sh_up"], dev["sh_down"],
                           max_tokens=T, phases=3)
    x = synth.activations(synth.streams(9401, 1)[0], (T, H), 2)
    y = cache.forward(dev_act(x, 2)).cpu().numpy()
    assert dq.device_status() == 0
    y_ref, _, _, _ = orc.moe_forward(Q4_K, E, k, H, F, ns, w["router_W"], w["w_gate"], w["w_up"],
                                     w["w_down"], w["sh_gate"], w["sh_up"], w["sh_down"], x, 2, T)
    assert rel_err(y, y_ref) <= MOE_TOL
    cache.close()
