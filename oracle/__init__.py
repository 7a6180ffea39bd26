"""CPU oracle for the block-quantized GEMV and the sparse MoE layer.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library (dequant_gemv_moe_gb300)
never does and shares no code with it.  The arithmetic lives in oracle.cpp
(plain loops in double); this module only marshals numpy arrays through
ctypes.
"""
import ctypes
import os

import numpy as np

from . import build as _build

OR_Q4_K, OR_Q6_K, OR_Q8_0, OR_Q4_0, OR_Q5_K, OR_NVFP4, OR_Q2_K, OR_Q3_K = 1, 2, 3, 4, 5, 6, 7, 8
OR_F32, OR_F16, OR_BF16 = 0, 1, 2

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        sigs = {
            "or_geometry": [i32, P, P],
            "or_dequant": [i32, P, i64, P],
            "or_act_to_f64": [i32, P, i64, P],
            "or_qgemv": [i32, P, i64, i64, P, i32, i32, P, i64, P, i32],
            "or_router_logits": [P, i32, i32, P, i32, i32, P, i32],
            "or_topk": [P, i32, i32, i32, P, P],
            "or_permute": [P, i32, i32, i32, P, P, P],
            "or_expert_ffn": [i32, P, P, P, i32, i32, P, P],
            "or_moe_forward": [i32, i32, i32, i32, i32, i32, P, P, P, P, P, P,
                               P, P, i32, i32, P, i32, P, P, P, P, i32],
        }
        for name, argt in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = argt
            fn.restype = ctypes.c_int
        L.or_silu.argtypes = [dbl]
        L.or_silu.restype = dbl
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def default_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def geometry(fmt):
    qk, nb = ctypes.c_int(), ctypes.c_int()
    _check(lib().or_geometry(fmt, ctypes.byref(qk), ctypes.byref(nb)), "geometry")
    return qk.value, nb.value


def dequant(fmt, blocks, n):
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    out = np.empty(n, dtype=np.float32)
    _check(lib().or_dequant(fmt, _p(blocks), n, _p(out)), "dequant")
    return out


def act_to_f64(dtype, x):
    x = np.ascontiguousarray(x)
    out = np.empty(x.size, dtype=np.float64)
    _check(lib().or_act_to_f64(dtype, _p(x), x.size, _p(out)), "act_to_f64")
    return out.reshape(x.shape)


def qgemv(fmt, W, N, K, x, xdt, batch, rows=None, nthreads=None):
    """y [batch][len(rows) or N] fp32, computed in double and rounded once."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x)
    nthreads = nthreads or default_threads()
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nr = rows.size
    else:
        nr = N
    y = np.empty((batch, nr), dtype=np.float32)
    _check(lib().or_qgemv(fmt, _p(W), N, K, _p(x), xdt, batch, _p(rows), nr,
                          _p(y), nthreads), "qgemv")
    return y


def router_logits(Wr, E, H, x, xdt, T, nthreads=None):
    Wr = np.ascontiguousarray(Wr, dtype=np.float32)
    x = np.ascontiguousarray(x)
    out = np.empty((T, E), dtype=np.float64)
    _check(lib().or_router_logits(_p(Wr), E, H, _p(x), xdt, T, _p(out),
                                  nthreads or default_threads()), "router_logits")
    return out


def topk(logits, k):
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    gate = np.empty((T, k), dtype=np.float64)
    _check(lib().or_topk(_p(logits), T, E, k, _p(idx), _p(gate)), "topk")
    return idx, gate


def permute(idx, E):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    sorted_ = np.empty(T * k, dtype=np.int32)
    _check(lib().or_permute(_p(idx), T, k, E, _p(counts), _p(offsets),
                            _p(sorted_)), "permute")
    return counts, offsets, sorted_


def silu(g):
    return lib().or_silu(float(g))


def expert_ffn(fmt, Wg, Wu, Wd, H, F, v):
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(H, dtype=np.float64)
    _check(lib().or_expert_ffn(fmt, _p(np.ascontiguousarray(Wg)),
                               _p(np.ascontiguousarray(Wu)),
                               _p(np.ascontiguousarray(Wd)), H, F, _p(v),
                               _p(out)), "expert_ffn")
    return out


def moe_forward(fmt, E, k, H, F, n_shared, Wr, w_gate, w_up, w_down, sh_gate,
                sh_up, sh_down, x, xdt, T, tokens=None, nthreads=None):
    """Returns (y [ntok][H] fp32, idx [T][k], gate [T][k] f64, logits [T][E] f64)."""
    x = np.ascontiguousarray(x)
    if tokens is not None:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        nt = tokens.size
    else:
        nt = T
    y = np.empty((nt, H), dtype=np.float32)
    idx = np.empty((T, k), dtype=np.int32)
    gate = np.empty((T, k), dtype=np.float64)
    logits = np.empty((T, E), dtype=np.float64)
    c = np.ascontiguousarray
    _check(lib().or_moe_forward(
        fmt, E, k, H, F, n_shared, _p(c(Wr, dtype=np.float32)), _p(c(w_gate)),
        _p(c(w_up)), _p(c(w_down)),
        _p(c(sh_gate) if sh_gate is not None else None),
        _p(c(sh_up) if sh_up is not None else None),
        _p(c(sh_down) if sh_down is not None else None),
        _p(x), xdt, T, _p(tokens), nt, _p(y), _p(idx), _p(gate), _p(logits),
        nthreads or default_threads()), "moe_forward")
    return y, idx, gate, logits
