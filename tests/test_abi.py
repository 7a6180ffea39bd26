"""The C-ABI library loads and exports every symbol include/dqmoe.h declares
(CPU only: no compute call without a GPU), and host-side validation rejects
bad arguments before anything is launched."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "dqmoe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def so():
    import importlib.util
    path = os.path.join(ROOT, "dequant_gemv_moe_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_dqmoe_build", path)
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return ctypes.CDLL(b.build())


def test_header_symbols_exported(so):
    names = _declared()
    assert "dq_qgemv" in names and "dq_moe_forward" in names and "dq_dequant" in names
    for n in names:
        assert hasattr(so, n), n


def test_status_strings(so):
    so.dq_status_string.restype = ctypes.c_char_p
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert so.dq_status_string(code)
    assert so.dq_status_string(12345) == b"unknown status"


def test_qgemv_argument_errors_without_launch(so):
    f = so.dq_qgemv
    P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [I, P, L, L, P, I, I, P, P]
    a = P(4096)                # fake, aligned; never dereferenced on the error paths
    assert f(9, a, 64, 256, a, 1, 1, a, None) == -1            # bad format
    assert f(1, None, 64, 256, a, 1, 1, a, None) == -1         # null W
    assert f(1, a, 64, 100, a, 1, 1, a, None) == -1            # K % 256
    assert f(1, a, 64, 256, a, 1, 0, a, None) == -1            # batch 0
    assert f(1, a, 64, 256, a, 1, 9, a, None) == -1            # batch 9
    assert f(1, a, 64, 256, a, 7, 1, a, None) == -1            # bad dtype
    assert f(1, P(4097), 64, 256, a, 1, 1, a, None) == -2      # misaligned W
    assert f(2, a, 64, 1024, a, 1, 1, a, None) == -2           # Q6_K needs K % 2048
    assert f(7, a, 64, 512, a, 1, 1, a, None) == -2            # Q2_K needs K % 1024
    assert f(8, a, 64, 1024, a, 1, 1, a, None) == -2           # Q3_K needs K % 2048
    assert f(1, a, 0, 256, a, 1, 1, a, None) == -1             # N = 0


def test_qgemv_ex_argument_errors_without_launch(so):
    f = so.dq_qgemv_ex
    P, I, L, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint
    f.argtypes = [I, P, L, L, P, I, I, P, I, U, P]
    a = P(4096)
    assert f(1, a, 64, 256, a, 1, 1, a, 0, 2, None) == -1      # unknown flag bit
    assert f(1, a, 64, 256, a, 1, 1, a, 9, 1, None) == -1      # ksplit > 8
    assert f(1, a, 64, 256, a, 1, 1, a, -1, 0, None) == -1     # ksplit < 0
    assert f(1, P(4097), 64, 256, a, 1, 1, a, 0, 1, None) == -2  # misaligned W


def test_dequant_argument_errors(so):
    f = so.dq_dequant
    P = ctypes.c_void_p
    f.argtypes = [ctypes.c_int, P, ctypes.c_int64, P, P]
    a = P(4096)
    assert f(1, a, 100, a, None) == -1
    assert f(3, a, 0, a, None) == -1
    assert f(3, P(4097), 32, a, None) == -2


def test_block_geometry_all_formats(so):
    f = so.dq_block_geometry
    qk, nb = ctypes.c_int(), ctypes.c_int()
    # Q4_K, Q6_K, Q8_0, Q4_0, Q5_K, NVFP4, Q2_K, Q3_K: the block sizes
    for fmt, want in [(1, (256, 144)), (2, (256, 210)), (3, (32, 34)), (4, (32, 18)),
                      (5, (256, 176)), (6, (256, 144)), (7, (256, 84)), (8, (256, 110))]:
        assert f(fmt, ctypes.byref(qk), ctypes.byref(nb)) == 0
        assert (qk.value, nb.value) == want
    assert f(9, ctypes.byref(qk), ctypes.byref(nb)) == -1
    assert f(0, ctypes.byref(qk), ctypes.byref(nb)) == -1


def test_moe_rejects_gemv_only_formats(so):
    # the MoE layer takes Q4_K / Q6_K / Q8_0 / NVFP4 experts; Q4_0 and Q5_K
    # are dequant / qGEMV formats: refused before anything is launched
    class Desc(ctypes.Structure):
        _fields_ = [("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("hidden", ctypes.c_int32),
                    ("ffn", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("fmt", ctypes.c_int32),
                    ("router_W", ctypes.c_void_p), ("w_gate", ctypes.c_void_p),
                    ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                    ("sh_gate", ctypes.c_void_p), ("sh_up", ctypes.c_void_p),
                    ("sh_down", ctypes.c_void_p)]
    a = ctypes.c_void_p(4096)
    n = ctypes.c_size_t()
    f = so.dq_moe_workspace_size
    f.argtypes = [ctypes.POINTER(Desc), ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
    for fmt, rc in [(1, 0), (6, 0), (4, -3), (5, -3), (7, -3), (8, -3), (9, -1)]:
        d = Desc(8, 2, 512, 512, 0, fmt, a, a, a, a, None, None, None)
        assert f(ctypes.byref(d), 4, ctypes.byref(n)) == rc, fmt


def test_expert_cache_argument_errors(so):
    # checks that fail before any CUDA call: no cache pointer, tokens, phases,
    # too few slots; null handles everywhere else
    class Desc(ctypes.Structure):
        _fields_ = [("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("hidden", ctypes.c_int32),
                    ("ffn", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("fmt", ctypes.c_int32),
                    ("router_W", ctypes.c_void_p), ("w_gate", ctypes.c_void_p),
                    ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                    ("sh_gate", ctypes.c_void_p), ("sh_up", ctypes.c_void_p),
                    ("sh_down", ctypes.c_void_p)]
    a = ctypes.c_void_p(4096)
    d = Desc(8, 2, 512, 512, 0, 1, a, a, a, a, None, None, None)
    f = so.dq_expert_cache_create
    f.argtypes = [ctypes.POINTER(Desc), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    h = ctypes.c_void_p()
    assert f(ctypes.byref(d), 4, a, a, a, 2, 2, None) == -1             # no handle pointer
    assert f(ctypes.byref(d), 4, a, a, a, 0, 2, ctypes.byref(h)) == -1  # max_tokens
    assert f(ctypes.byref(d), 4, a, a, a, 2, 0, ctypes.byref(h)) == -1  # phases
    assert f(ctypes.byref(d), 4, a, a, a, 2, 9, ctypes.byref(h)) == -1
    assert f(ctypes.byref(d), 3, a, a, a, 2, 2, ctypes.byref(h)) == -1  # slots < 2 * 2
    assert f(ctypes.byref(d), 9, a, a, a, 2, 2, ctypes.byref(h)) == -1  # slots > E
    assert f(ctypes.byref(d), 4, None, a, a, 2, 2, ctypes.byref(h)) == -1
    assert f(ctypes.byref(d), 4, ctypes.c_void_p(4100), a, a, 2, 2, ctypes.byref(h)) == -2
    d.fmt = 4   # Q4_0 experts are not supported by the layer
    assert f(ctypes.byref(d), 4, a, a, a, 2, 2, ctypes.byref(h)) == -3
    assert h.value is None
    g = so.dq_moe_forward_streamed
    g.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]
    assert g(None, a, 1, 1, a, a, 1 << 20, None, a) == -1
    so.dq_expert_cache_stats.argtypes = [ctypes.c_void_p] * 4
    assert so.dq_expert_cache_stats(None, a, a, a) == -1
    so.dq_expert_cache_destroy.argtypes = [ctypes.c_void_p]
    assert so.dq_expert_cache_destroy(None) == -1
    so.dq_expert_cache_workspace_size.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    n = ctypes.c_size_t()
    assert so.dq_expert_cache_workspace_size(None, 1, ctypes.byref(n)) == -1
