"""GPU parity of the MoE steps and the whole layer against the CPU oracle (-m gpu).

Router logits: within the fp32 summation bound (gamma_n * sum |W x|).
Top-k indices: bit-exact against the oracle's stable sort applied to the GPU's
own logits; against the oracle's own (double) logits every disagreement must
be a near-tie (gap below twice the bound).  Permute: bit-exact.  Layer output:
max|y - y_ref| / max|y_ref| <= 2e-3 (16-bit operands on the tensor cores).
"""
import numpy as np
import pytest
import torch

import synth
import moe_layers
from gpu_util import dev_act, dev_bytes, rel_err
from moe_layers import ref_under_selection

pytestmark = pytest.mark.gpu

Q4_K, Q6_K, Q8_0, NVFP4 = 1, 2, 3, 6
MOE_TOL = 2e-3


@pytest.fixture(scope="module")
def dq():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import dequant_gemv_moe_gb300 as dq
    return dq


def _fp32_bound(Wr, xf, H):
    # |fl(sum) - sum| <= gamma_n * sum |terms|, gamma_n = n u / (1 - n u), n = H + splits
    u = 2.0 ** -24
    n = H + 64
    gam = n * u / (1 - n * u)
    return gam * (np.abs(xf) @ np.abs(Wr.astype(np.float64)).T)


def _check_router(orc, Wr, x, xdt, E, H, T, k, logits, idx, gate):
    xf = orc.act_to_f64(xdt, x).reshape(T, H)
    L_ref = orc.router_logits(Wr, E, H, x, xdt, T)
    bound = _fp32_bound(Wr, xf, H)
    assert np.all(np.abs(logits.astype(np.float64) - L_ref) <= bound)
    # (ii) selection and tie-break exactly as the stable sort of the GPU's logits
    idx_g, gate_g = orc.topk(logits.astype(np.float64), k)
    np.testing.assert_array_equal(idx, idx_g)
    np.testing.assert_allclose(gate, gate_g, rtol=2e-6, atol=1e-7)
    # (iii) against the exact logits: only near-ties may differ
    idx_r, _ = orc.topk(L_ref, k)
    bad = np.nonzero(np.any(idx != idx_r, axis=1))[0]
    for t in bad:
        srt = np.sort(L_ref[t])[::-1]
        gap = np.min(np.abs(np.diff(srt[max(0, k - 2):k + 1])))
        assert gap <= 2 * bound[t].max(), (t, gap)
    return len(bad)


@pytest.mark.parametrize("E,k,H,T,xdt", [(8, 2, 4096, 16, 1), (256, 8, 7168, 8, 2),
                                         (256, 8, 7168, 1, 2), (64, 6, 1024, 37, 0),
                                         (3, 3, 256, 5, 1)])
def test_router_topk(dq, orc, E, k, H, T, xdt):
    g = synth.streams(900 + E + T, 2)
    Wr = synth.router_weights(g[0], E, H)
    x = synth.activations(g[1], (T, H), xdt)
    logits, idx, gate = dq.moe_router(torch.from_numpy(Wr).cuda(), E, H, dev_act(x, xdt), k)
    _check_router(orc, Wr, x, xdt, E, H, T, k, logits.cpu().numpy(), idx.cpu().numpy(),
                  gate.cpu().numpy())


def test_router_argument_errors(dq):
    # the logits buffer is required (the sums are formed there); pointers need
    # 4-byte alignment; nothing is launched on an error
    import ctypes
    E, k, H, T = 16, 2, 256, 2
    Wr = torch.zeros(E, H, dtype=torch.float32, device="cuda")
    x = torch.zeros(T, H, dtype=torch.float16, device="cuda")
    lg = torch.full((T, E), 7.0, dtype=torch.float32, device="cuda")
    idx = torch.full((T, k), -3, dtype=torch.int32, device="cuda")
    gate = torch.full((T, k), 7.0, dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    st = P(torch.cuda.current_stream().cuda_stream)
    f = dq.lib.dq_moe_router
    assert f(P(Wr.data_ptr()), E, H, P(x.data_ptr()), 1, T, k, None, P(idx.data_ptr()),
             P(gate.data_ptr()), st) == -1
    assert f(P(Wr.data_ptr() + 2), E, H, P(x.data_ptr()), 1, T, k, P(lg.data_ptr()),
             P(idx.data_ptr()), P(gate.data_ptr()), st) == -2
    assert f(P(Wr.data_ptr()), E, 100, P(x.data_ptr()), 1, T, k, P(lg.data_ptr()),
             P(idx.data_ptr()), P(gate.data_ptr()), st) == -1
    torch.cuda.synchronize()
    assert bool((idx == -3).all()) and bool((lg == 7.0).all())


def test_topk_ties_lowest_index(dq):
    # zero router weights: every logit is 0, the selection is experts 0..k-1
    E, k, H, T = 32, 4, 256, 3
    Wr = torch.zeros(E, H, dtype=torch.float32, device="cuda")
    x = torch.randn(T, H, device="cuda").half()
    logits, idx, gate = dq.moe_router(Wr, E, H, x, k)
    assert idx.cpu().numpy().tolist() == [[0, 1, 2, 3]] * T
    np.testing.assert_allclose(gate.cpu().numpy(), 0.25, rtol=1e-7)


@pytest.mark.parametrize("T,k,E", [(16, 2, 8), (8, 8, 256), (256, 8, 256), (1, 1, 1),
                                   (1000, 4, 60)])
def test_permute_bit_exact(dq, orc, T, k, E):
    rng = np.random.default_rng(T * 31 + E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    offs, srt = dq.moe_permute(torch.from_numpy(idx).cuda(), E)
    counts, offsets, sorted_ = orc.permute(idx, E)
    np.testing.assert_array_equal(offs.cpu().numpy(), offsets)
    np.testing.assert_array_equal(srt.cpu().numpy(), sorted_)


def _moe_case(dq, orc, fmt, E, k, H, F, ns, T, xdt, seed, tokens=None, cached=None):
    """The whole layer on the GPU against the oracle for the listed tokens (all
    T if None).  A token whose GPU selection differs from the oracle's exact
    one must sit at a near-tie of the logits (checked by _check_router); it is
    compared with the oracle's layer under the GPU's selection instead."""
    if cached is not None:
        w, dev, desc = cached
    else:
        w = synth.moe_weights(seed, E, H, F, ns, fmt)
        dev = {kk: (dev_bytes(v) if v is not None and v.dtype == np.uint8 else
                    (torch.from_numpy(v).cuda() if v is not None else None)) for kk, v in w.items()}
        desc = dq.ops.make_desc(E, k, H, F, ns, fmt, dev["router_W"], dev["w_gate"], dev["w_up"],
                                dev["w_down"], dev["sh_gate"], dev["sh_up"], dev["sh_down"])
    x = synth.activations(synth.streams(seed + 1, 1)[0], (T, H), xdt)
    y, idx, gate, logits = dq.moe_forward(desc, dev_act(x, xdt), want_routing=True)
    y = y.cpu().numpy()
    idx = idx.cpu().numpy()
    assert dq.device_status() == 0
    assert np.isfinite(y).all()
    nb = _check_router(orc, w["router_W"], x, xdt, E, H, T, k, logits.cpu().numpy(), idx,
                       gate.cpu().numpy())
    y_ref, idx_ref, _, L_ref = orc.moe_forward(fmt, E, k, H, F, ns, w["router_W"], w["w_gate"],
                                               w["w_up"], w["w_down"], w["sh_gate"], w["sh_up"],
                                               w["sh_down"], x, xdt, T, tokens=tokens)
    rows = np.arange(T) if tokens is None else np.asarray(tokens)
    assert y_ref.shape == (len(rows), H)
    ref = y_ref.copy()
    for i, t in enumerate(rows):
        if not np.array_equal(idx[t], idx_ref[t]):
            ref[i] = ref_under_selection(orc, fmt, w, E, k, H, F, ns, x, xdt, t, idx[t], L_ref)
    err = rel_err(y[rows], ref)
    if cached is None:
        del dev
        torch.cuda.empty_cache()
    return err, nb


@pytest.mark.parametrize("fmt,E,k,H,F,ns,T,xdt", [
    (Q4_K, 8, 2, 512, 1024, 0, 5, 1),
    (Q4_K, 8, 2, 512, 1024, 1, 16, 2),
    (Q4_K, 16, 4, 1024, 512, 2, 33, 1),     # > 8 tokens on some experts: several groups
    (Q8_0, 8, 3, 768, 512, 1, 9, 2),
    (Q6_K, 4, 2, 2048, 2048, 1, 7, 1),
    (Q4_K, 4, 4, 256, 256, 0, 3, 2),        # every expert active
    (Q4_K, 1, 1, 256, 512, 0, 1, 1),        # one expert, one token
    (Q4_K, 4, 2, 512, 512, 1, 40, 1),       # ~20 tokens per expert: 32-column groups
    (Q8_0, 4, 2, 256, 512, 0, 64, 2),       # ~32 tokens per expert: some groups split
    # more than 32 tokens on an expert: the tcgen05 grouped GEMM (units of <= 128)
    (Q4_K, 4, 2, 512, 512, 1, 64, 1),
    (Q6_K, 2, 1, 2048, 2048, 0, 100, 2),
    (Q8_0, 2, 2, 256, 256, 1, 300, 1),
    # many one-token experts beside a 3-token shared expert
    (Q4_K, 64, 2, 1024, 512, 1, 3, 2),
    (Q4_K, 32, 8, 2048, 1024, 0, 2, 1),
    # NVFP4 experts: one-token decode, 16-column groups, 32-column groups,
    # and the tcgen05 path
    (NVFP4, 8, 2, 512, 1024, 1, 1, 2),
    (NVFP4, 8, 2, 512, 512, 0, 30, 1),
    (NVFP4, 4, 2, 768, 512, 1, 50, 2),
    (NVFP4, 2, 2, 512, 256, 1, 90, 1),
    # one token with shared experts (hidden > 1024: the streaming router;
    # hidden 1024: the tiled router)
    (Q4_K, 16, 4, 2048, 512, 2, 1, 2),
    (Q8_0, 8, 2, 2048, 1024, 1, 1, 1),
    (Q6_K, 4, 2, 4096, 2048, 1, 1, 2),
    (Q4_K, 16, 4, 1024, 512, 1, 1, 1),
    # few down units for the grid: the down products split over K (two and
    # four parts, shared expert included), summed in part order by the combine
    (Q6_K, 4, 2, 2048, 2048, 1, 6, 2),
    (Q8_0, 8, 2, 1024, 4096, 1, 12, 2),
    (NVFP4, 8, 2, 1024, 4096, 0, 1, 1),
    # two bf16 tokens: the permute CTA converts x to fp16 itself
    (Q4_K, 32, 4, 2048, 512, 1, 2, 2),
    # Q6_K / Q8_0 one-token experts at T > 1 beside experts with two tokens
    # (each seed's routing gives 1-4 of them; the last case also one 3-token
    # expert), which run on the general kernel in the same layer
    (Q6_K, 16, 2, 2048, 2048, 1, 3, 1),
    (Q6_K, 32, 8, 2048, 2048, 0, 2, 2),
    (Q8_0, 16, 2, 1024, 1024, 0, 4, 2),
    (Q4_K, 32, 4, 2048, 512, 1, 4, 1),
    (Q8_0, 64, 4, 1024, 512, 1, 8, 1),
])
def test_moe_forward_small(dq, orc, fmt, E, k, H, F, ns, T, xdt):
    err, _ = _moe_case(dq, orc, fmt, E, k, H, F, ns, T, xdt, seed=3000 + E * 7 + T)
    assert err <= MOE_TOL, err


def test_moe_mixtral_config(dq, orc):
    # every token of the Mixtral-shaped layer
    c = synth.MOE_MIXTRAL
    err, nb = _moe_case(dq, orc, c["fmt"], c["E"], c["top_k"], c["H"], c["F"], c["n_shared"],
                        16, c["xdt"], seed=synth.BASE_SEED + 3, cached=moe_layers.mixtral())
    assert err <= MOE_TOL, err


def _deepseek_t256_tokens(orc, w, x, xdt, c):
    """Tokens of the T=256 chunk to compare: the first and last column of
    every 32-column box of the shared expert's tcgen05 units (units of 128
    tokens), every token of the three most-loaded routed experts, and a
    seeded spread over the rest."""
    T = x.shape[0]
    L = orc.router_logits(w["router_W"], c["E"], c["H"], x, xdt, T)
    idx, _ = orc.topk(L, c["top_k"])
    cnt = np.bincount(idx.ravel(), minlength=c["E"])
    busy = np.argsort(-cnt, kind="stable")[:3]
    toks = set()
    for b in range(0, T, 32):
        toks.update((b, min(T - 1, b + 31)))
    for e in busy:
        toks.update(np.nonzero(np.any(idx == e, axis=1))[0].tolist())
    toks.update(np.random.default_rng(256).choice(T, 12, replace=False).tolist())
    return sorted(int(t) for t in toks)


@pytest.mark.parametrize("T", [1, 8, 256])
def test_moe_deepseek_config(dq, orc, T):
    # every token at T = 1 and 8; at T = 256 (the shared expert on the tcgen05
    # GEMM) every 32-column box edge, the busiest experts' tokens and a spread
    c = synth.MOE_DEEPSEEK
    lay = moe_layers.deepseek()
    tokens = None
    if T == 256:
        x = synth.activations(synth.streams(synth.BASE_SEED + 5, 1)[0], (T, c["H"]), c["xdt"])
        tokens = _deepseek_t256_tokens(orc, lay[0], x, c["xdt"], c)
        assert len(tokens) >= 32
    err, nb = _moe_case(dq, orc, c["fmt"], c["E"], c["top_k"], c["H"], c["F"], c["n_shared"], T,
                        c["xdt"], seed=synth.BASE_SEED + 4, tokens=tokens, cached=lay)
    assert err <= MOE_TOL, err


def test_moe_refuses_fp32_activations(dq):
    # the layer computes with 16-bit tensor-core operands, which cannot hold
    # the 1e-5 bar of fp32 activations: fp32 x is refused before any launch
    import ctypes
    E, k, H, F = 8, 2, 256, 256
    d = dq.ops.make_desc(E, k, H, F, 0, 1, torch.zeros(E, H, device="cuda"),
                         torch.zeros(E * F * 144, dtype=torch.uint8, device="cuda"),
                         torch.zeros(E * F * 144, dtype=torch.uint8, device="cuda"),
                         torch.zeros(E * H * 144, dtype=torch.uint8, device="cuda"))
    T = 4
    x = torch.zeros(T, H, dtype=torch.float32, device="cuda")
    y = torch.full((T, H), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(dq.moe_workspace_size(d, T), dtype=torch.uint8, device="cuda")
    rc = dq.lib.dq_moe_forward(ctypes.byref(d), ctypes.c_void_p(x.data_ptr()), 0, T,
                               ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                               ws.numel(), None, None, None, None)
    assert rc == -3
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


def test_moe_workspace_errors(dq):
    import ctypes
    E, k, H, F = 8, 2, 256, 256
    d = dq.ops.make_desc(E, k, H, F, 0, 1, torch.zeros(E, H, device="cuda"),
                         torch.zeros(E * F * 144, dtype=torch.uint8, device="cuda"),
                         torch.zeros(E * F * 144, dtype=torch.uint8, device="cuda"),
                         torch.zeros(E * H * 144, dtype=torch.uint8, device="cuda"))
    need = dq.moe_workspace_size(d, 4)
    x = torch.zeros(4, H, dtype=torch.float16, device="cuda")
    y = torch.empty(4, H, device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    rc = dq.lib.dq_moe_forward(ctypes.byref(d), ctypes.c_void_p(x.data_ptr()), 1, 4,
                               ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                               need - 1, None, None, None, None)
    assert rc == -4
