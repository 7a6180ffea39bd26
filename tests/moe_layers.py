"""Seeded MoE layers for the GPU tests, kept once per process.

The full-size layers (Mixtral-shaped: 8 experts of 14336 x 4096; DeepSeek-V3-
shaped: 256 experts of 2048 x 7168 plus one shared expert) take seconds to
draw, so each is drawn once and its host bytes and device copies are shared by
the tests that use it.
"""
import numpy as np
import torch

import synth
from gpu_util import dev_bytes

_LAYERS = {}


def layer(seed, fmt, E, k, H, F, ns):
    """(host weights dict, device tensors dict, descriptor) of one seeded layer."""
    import dequant_gemv_moe_gb300 as dq
    key = (seed, fmt, E, k, H, F, ns)
    if key not in _LAYERS:
        w = synth.moe_weights(seed, E, H, F, ns, fmt)
        dev = {kk: (dev_bytes(v) if v is not None and v.dtype == np.uint8 else
                    (torch.from_numpy(v).cuda() if v is not None else None))
               for kk, v in w.items()}
        desc = dq.ops.make_desc(E, k, H, F, ns, fmt, dev["router_W"], dev["w_gate"], dev["w_up"],
                                dev["w_down"], dev["sh_gate"], dev["sh_up"], dev["sh_down"])
        _LAYERS[key] = (w, dev, desc)
    return _LAYERS[key]


def drop(seed, fmt, E, k, H, F, ns):
    _LAYERS.pop((seed, fmt, E, k, H, F, ns), None)
    torch.cuda.empty_cache()


def deepseek():
    c = synth.MOE_DEEPSEEK
    return layer(synth.BASE_SEED + 4, c["fmt"], c["E"], c["top_k"], c["H"], c["F"], c["n_shared"])


def mixtral():
    c = synth.MOE_MIXTRAL
    return layer(synth.BASE_SEED + 3, c["fmt"], c["E"], c["top_k"], c["H"], c["F"], c["n_shared"])


def ref_under_selection(orc, fmt, w, E, k, H, F, ns, x, xdt, t, sel, L_ref):
    """The oracle's layer output for token t with the experts `sel` selected
    (the oracle's gates over those experts' exact logits L_ref[t]): the
    reference for a token whose selection the GPU took differently at a
    near-tie of the fp32 logits."""
    qk, nb = synth.BLOCK[fmt]
    gu = F * (H // qk) * nb
    dn = H * (F // qk) * nb
    masked = np.full((1, E), -1e300)
    masked[0, sel] = L_ref[t, sel]
    idx_m, gate_m = orc.topk(masked, k)
    v = orc.act_to_f64(xdt, x[t:t + 1]).reshape(H)
    y = np.zeros(H)
    for i in range(k):
        e = int(idx_m[0, i])
        y += gate_m[0, i] * orc.expert_ffn(fmt, w["w_gate"][e * gu:(e + 1) * gu],
                                           w["w_up"][e * gu:(e + 1) * gu],
                                           w["w_down"][e * dn:(e + 1) * dn], H, F, v)
    for s in range(ns):
        y += orc.expert_ffn(fmt, w["sh_gate"][s * gu:(s + 1) * gu], w["sh_up"][s * gu:(s + 1) * gu],
                            w["sh_down"][s * dn:(s + 1) * dn], H, F, v)
    return y.astype(np.float32)
