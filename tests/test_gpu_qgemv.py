"""GPU parity of block decode and qGEMV against the CPU oracle (-m gpu).

Bars: decoded weights bit-exact; y within max|y - y_ref| / max|y_ref| <= 1e-5
for fp32 activations and <= 2e-3 for fp16 / bf16 activations.
"""
import numpy as np
import pytest
import torch

import synth
from golden_io import read_block_cases
from gpu_util import TOL, dev_act, dev_bytes, rel_err

pytestmark = pytest.mark.gpu

Q4_K, Q6_K, Q8_0 = 1, 2, 3


@pytest.fixture(scope="module")
def dq():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import dequant_gemv_moe_gb300 as dq
    return dq


@pytest.mark.parametrize("fmt,qk", [(Q4_K, 256), (Q6_K, 256), (Q8_0, 32)])
def test_dequant_bit_exact_random(dq, orc, fmt, qk):
    g = synth.streams(31 + fmt, 1)[0]
    raw = synth.quant_matrix(g, fmt, 37, 4096)
    n = 37 * 4096
    got = dq.dequant(fmt, dev_bytes(raw), n).cpu().numpy()
    ref = orc.dequant(fmt, raw, n)
    assert got.view(np.uint32).tolist() == ref.view(np.uint32).tolist()


@pytest.mark.parametrize("fname,fmt,qk", [("q4_k_blocks.txt", Q4_K, 256),
                                          ("q6_k_blocks.txt", Q6_K, 256),
                                          ("q8_0_blocks.txt", Q8_0, 32)])
def test_dequant_golden(dq, fname, fmt, qk):
    for c in read_block_cases(fname):
        got = dq.dequant(fmt, dev_bytes(c["bytes"]), qk).cpu().numpy().astype(np.float64)
        np.testing.assert_array_equal(got, c["expect"], err_msg=c["name"])


def _case(dq, orc, fmt, N, K, B, xdt, seed, ksplit=None, rows=None, xscale=1.0):
    g = synth.streams(seed, 2)
    W = synth.quant_matrix(g[0], fmt, N, K)
    if xscale != 1.0:
        x = synth.activations(g[1], (B, K), 0) * np.float32(xscale)
        x = x if xdt == 0 else (x.astype(np.float16) if xdt == 1 else synth.f32_to_bf16_bits(x))
    else:
        x = synth.activations(g[1], (B, K), xdt)
    y = dq.qgemv(fmt, dev_bytes(W), N, K, dev_act(x, xdt), ksplit=ksplit).cpu().numpy()
    assert dq.device_status() == 0
    if rows is None:
        ref = orc.qgemv(fmt, W, N, K, x, xdt, B)
        got = y
    else:
        rows = np.asarray(rows, dtype=np.int64)
        ref = orc.qgemv(fmt, W, N, K, x, xdt, B, rows=rows)
        got = y[:, rows]
    assert np.isfinite(got).all()
    return rel_err(got, ref)


@pytest.mark.parametrize("fmt", [Q4_K, Q6_K, Q8_0])
@pytest.mark.parametrize("xdt", [0, 1, 2])
@pytest.mark.parametrize("B", [1, 3, 8])
def test_qgemv_small_ragged(dq, orc, fmt, xdt, B):
    # several 64-row tiles plus a ragged tail; K spans several pipeline stages
    N, K = 200, 4096
    err = _case(dq, orc, fmt, N, K, B, xdt, seed=fmt * 100 + xdt * 10 + B)
    assert err <= TOL[xdt], err


@pytest.mark.parametrize("fmt", [Q4_K, Q6_K, Q8_0])
@pytest.mark.parametrize("ks", [1, 2, 3, 5, 8])
def test_qgemv_cluster_ksplit(dq, orc, fmt, ks):
    N, K = 130, 8192
    err = _case(dq, orc, fmt, N, K, 4, 1, seed=500 + fmt * 10 + ks, ksplit=ks)
    assert err <= TOL[1], err


def test_qgemv_edge_shapes(dq, orc):
    # one row, one super-block, odd batch; Q6_K needs K % 2048 == 0
    for fmt, N, K in [(Q4_K, 1, 256), (Q8_0, 1, 256), (Q6_K, 1, 2048), (Q4_K, 65, 256),
                      (Q8_0, 63, 512)]:
        for xdt in (0, 1, 2):
            err = _case(dq, orc, fmt, N, K, 5, xdt, seed=N + K + xdt)
            assert err <= TOL[xdt], (fmt, N, K, xdt, err)


def test_qgemv_bf16_large_values(dq, orc):
    # activations far above the fp16 range: the per-stage power-of-two scale
    # must keep the 16-bit operands finite
    for fmt in (Q4_K, Q6_K, Q8_0):
        err = _case(dq, orc, fmt, 96, 4096, 8, 2, seed=77 + fmt, xscale=3.0e6)
        assert err <= TOL[2], err


def test_single_gemv_config(dq, orc):
    c = synth.GEMV_SINGLE
    err = _case(dq, orc, c["fmt"], c["N"], c["K"], c["batch"], c["xdt"], seed=synth.BASE_SEED)
    assert err <= TOL[0], err


@pytest.mark.parametrize("name,N,K", synth.LLAMA8B_LINEARS)
@pytest.mark.parametrize("B", [1, 4, 8])
def test_llama8b_linears(dq, orc, name, N, K, B):
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(N + B).integers(0, N, 96)]))
    err = _case(dq, orc, Q4_K, N, K, B, 1, seed=synth.BASE_SEED + 1, rows=rows)
    assert err <= TOL[1], err


@pytest.mark.parametrize("fmt", [Q4_K, Q6_K, Q8_0])
@pytest.mark.parametrize("name,N,K", synth.LLAMA70B_LINEARS[2:] + synth.LLAMA70B_LINEARS[:1])
@pytest.mark.parametrize("B", [1, 8])
def test_llama70b_linears(dq, orc, fmt, name, N, K, B):
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(N * B).integers(0, N, 48)]))
    err = _case(dq, orc, fmt, N, K, B, 1, seed=synth.BASE_SEED + 2, rows=rows)
    assert err <= TOL[1], err
    torch.cuda.empty_cache()
