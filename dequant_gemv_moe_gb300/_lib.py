"""ctypes binding of libdqmoe.so: argument marshalling only.

Every function takes torch CUDA tensors, passes their data pointers, sizes and
the current CUDA stream to the C ABI of include/dqmoe.h, and raises on a
non-zero status.  No computation happens here, and there is no fallback: if
the shared library is missing the import fails.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdqmoe.so")

Q4_K, Q6_K, Q8_0 = 1, 2, 3
F32, F16, BF16 = 0, 1, 2

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t


class DqError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (fn, status_string(status), status))


class MoeDesc(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int32), ("top_k", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("ffn", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("fmt", ctypes.c_int32),
                ("router_W", _P), ("w_gate", _P), ("w_up", _P), ("w_down", _P),
                ("sh_gate", _P), ("sh_up", _P), ("sh_down", _P)]


_SIGS = {
    "dq_block_geometry": [_I, _P, _P],
    "dq_dequant": [_I, _P, _I64, _P, _P],
    "dq_qgemv": [_I, _P, _I64, _I64, _P, _I, _I, _P, _P],
    "dq_qgemv_ksplit": [_I, _P, _I64, _I64, _P, _I, _I, _P, _I, _P],
    "dq_qgemv_ex": [_I, _P, _I64, _I64, _P, _I, _I, _P, _I, ctypes.c_uint, _P],
    "dq_device_status": [_P],
    "dq_stage": [_P, _P, _I64, _P],
}
_OPTIONAL_SIGS = {
    "dq_moe_workspace_size": [ctypes.POINTER(MoeDesc), _I, _P],
    "dq_moe_router": [_P, _I, _I, _P, _I, _I, _I, _P, _P, _P, _P],
    "dq_moe_permute": [_P, _I, _I, _I, _P, _P, _P],
    "dq_moe_forward": [ctypes.POINTER(MoeDesc), _P, _I, _I, _P, _P, _SZ, _P, _P, _P, _P],
    "dq_moe_forward_noalloc": [ctypes.POINTER(MoeDesc), _P, _I, _I, _P, _P, _P, _P, _P],
    "dq_expert_cache_create": [ctypes.POINTER(MoeDesc), _I, _P, _P, _P, _I, _I, _P],
    "dq_expert_cache_workspace_size": [_P, _I, _P],
    "dq_moe_forward_streamed": [_P, _P, _I, _I, _P, _P, _SZ, _P, _P],
    "dq_expert_cache_stats": [_P, _P, _P, _P],
    "dq_expert_cache_destroy": [_P],
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libdqmoe.so is not built (run __graft_entry__.build() or "
                          "python dequant_gemv_moe_gb300/build.py)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, argt in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = argt
        fn.restype = _I
    for name, argt in _OPTIONAL_SIGS.items():
        fn = getattr(lib, name, None)
        if fn is not None:
            fn.argtypes = argt
            fn.restype = _I
    lib.dq_status_string.argtypes = [_I]
    lib.dq_status_string.restype = ctypes.c_char_p
    return lib


lib = _load()


def status_string(status):
    return lib.dq_status_string(int(status)).decode()


def exported_symbols():
    return sorted(list(_SIGS) + list(_OPTIONAL_SIGS) + ["dq_status_string"])
