"""torch-facing wrappers of the C ABI (marshalling only; see include/dqmoe.h)."""
import ctypes

import torch

from ._lib import F16, F32, BF16, DqError, MoeDesc, lib

_DT = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _call(name, *args):
    rc = getattr(lib, name)(*args)
    if rc != 0:
        raise DqError(name, rc)


def _dtype_code(x):
    if x.dtype not in _DT:
        raise TypeError("activation dtype must be float32, float16 or bfloat16, got %s" % x.dtype)
    return _DT[x.dtype]


def block_geometry(fmt):
    qk, nb = ctypes.c_int(), ctypes.c_int()
    _call("dq_block_geometry", fmt, ctypes.byref(qk), ctypes.byref(nb))
    return qk.value, nb.value


def dequant(fmt, blocks, n_weights, out=None):
    """Decode n_weights weights of packed blocks (uint8 CUDA tensor) to fp32."""
    if out is None:
        out = torch.empty(n_weights, dtype=torch.float32, device=blocks.device)
    _call("dq_dequant", fmt, _ptr(blocks), n_weights, _ptr(out), _stream())
    return out


QGEMV_WEIGHTS_EARLY = 1


def qgemv(fmt, W, N, K, x, y=None, ksplit=None, weights_early=False):
    """y[b][n] = sum_k W[n][k] x[b][k]; x is [batch][K] (float32/float16/bfloat16).

    weights_early: W is not written by the kernel issued just before on the
    stream, so its first stages may stream in while that kernel drains
    (dq_qgemv_ex with DQ_QGEMV_WEIGHTS_EARLY).
    """
    x = x.reshape(-1, K)
    batch = x.shape[0]
    if y is None:
        y = torch.empty(batch, N, dtype=torch.float32, device=x.device)
    if weights_early:
        _call("dq_qgemv_ex", fmt, _ptr(W), N, K, _ptr(x), _dtype_code(x), batch, _ptr(y),
              int(ksplit or 0), QGEMV_WEIGHTS_EARLY, _stream())
    elif ksplit is None:
        _call("dq_qgemv", fmt, _ptr(W), N, K, _ptr(x), _dtype_code(x), batch, _ptr(y), _stream())
    else:
        _call("dq_qgemv_ksplit", fmt, _ptr(W), N, K, _ptr(x), _dtype_code(x), batch, _ptr(y),
              int(ksplit), _stream())
    return y


def stage(dst, src):
    """Copy src into dst (same number of bytes; CUDA or page-locked CPU tensors)
    with the library's copy kernel on the current stream (dq_stage)."""
    nb = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nb:
        raise ValueError("stage: dst and src sizes differ")
    _call("dq_stage", _ptr(dst), _ptr(src), nb, _stream())
    return dst


def device_status():
    v = ctypes.c_int()
    _call("dq_device_status", ctypes.byref(v))
    return v.value


# ---------------------------------------------------------------- MoE layer
def make_desc(E, top_k, hidden, ffn, n_shared, fmt, router_W, w_gate, w_up, w_down,
              sh_gate=None, sh_up=None, sh_down=None):
    d = MoeDesc()
    d.E, d.top_k, d.hidden, d.ffn, d.n_shared, d.fmt = E, top_k, hidden, ffn, n_shared, fmt
    d.router_W, d.w_gate, d.w_up, d.w_down = (router_W.data_ptr(), w_gate.data_ptr(),
                                              w_up.data_ptr(), w_down.data_ptr())
    d.sh_gate = sh_gate.data_ptr() if sh_gate is not None else None
    d.sh_up = sh_up.data_ptr() if sh_up is not None else None
    d.sh_down = sh_down.data_ptr() if sh_down is not None else None
    return d


def moe_workspace_size(desc, T):
    n = ctypes.c_size_t()
    _call("dq_moe_workspace_size", ctypes.byref(desc), T, ctypes.byref(n))
    return n.value


def moe_router(router_W, E, H, x, top_k, logits=None):
    T = x.shape[0]
    dev = x.device
    if logits is None:
        logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    idx = torch.empty(T, top_k, dtype=torch.int32, device=dev)
    gate = torch.empty(T, top_k, dtype=torch.float32, device=dev)
    _call("dq_moe_router", _ptr(router_W), E, H, _ptr(x), _dtype_code(x), T, top_k, _ptr(logits),
          _ptr(idx), _ptr(gate), _stream())
    return logits, idx, gate


def moe_permute(topk_idx, E):
    T, k = topk_idx.shape
    dev = topk_idx.device
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_ = torch.empty(T * k, dtype=torch.int32, device=dev)
    _call("dq_moe_permute", _ptr(topk_idx), T, k, E, _ptr(offsets), _ptr(sorted_), _stream())
    return offsets, sorted_


def moe_forward(desc, x, y=None, ws=None, want_routing=False):
    """The whole MoE layer.  Returns y (and idx, gate, logits if want_routing)."""
    T = x.shape[0]
    dev = x.device
    if y is None:
        y = torch.empty(T, desc.hidden, dtype=torch.float32, device=dev)
    need = moe_workspace_size(desc, T)
    if ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    idx = gate = logits = None
    if want_routing:
        idx = torch.empty(T, desc.top_k, dtype=torch.int32, device=dev)
        gate = torch.empty(T, desc.top_k, dtype=torch.float32, device=dev)
        logits = torch.empty(T, desc.E, dtype=torch.float32, device=dev)
    _call("dq_moe_forward", ctypes.byref(desc), _ptr(x), _dtype_code(x), T, _ptr(y), _ptr(ws),
          ws.numel(), _ptr(idx), _ptr(gate), _ptr(logits), _stream())
    if want_routing:
        return y, idx, gate, logits
    return y


# ------------------------------------------------------- expert streaming
class ExpertCache:
    """A device cache of `slots` experts for a layer whose routed experts live
    in page-locked host memory (dq_expert_cache_*; marshalling only).

    host_w_gate / host_w_up / host_w_down: pinned CPU uint8 tensors of all E
    experts; router_W and the shared experts (optional) are CUDA tensors.  The
    slot buffers are allocated here as CUDA tensors and kept by this object.
    """

    def __init__(self, E, top_k, hidden, ffn, n_shared, fmt, router_W, host_w_gate, host_w_up,
                 host_w_down, sh_gate=None, sh_up=None, sh_down=None, slots=None,
                 max_tokens=1, phases=2):
        self.desc = make_desc(E, top_k, hidden, ffn, n_shared, fmt, router_W, host_w_gate,
                              host_w_up, host_w_down, sh_gate, sh_up, sh_down)
        self._keep = (router_W, host_w_gate, host_w_up, host_w_down, sh_gate, sh_up, sh_down)
        if slots is None:
            slots = min(E, max_tokens * top_k)
        dev = router_W.device
        gu = host_w_gate.numel() // E
        dn = host_w_down.numel() // E
        self.slot_gate = torch.empty(slots * gu, dtype=torch.uint8, device=dev)
        self.slot_up = torch.empty(slots * gu, dtype=torch.uint8, device=dev)
        self.slot_down = torch.empty(slots * dn, dtype=torch.uint8, device=dev)
        self.max_tokens = max_tokens
        h = ctypes.c_void_p()
        _call("dq_expert_cache_create", ctypes.byref(self.desc), slots, _ptr(self.slot_gate),
              _ptr(self.slot_up), _ptr(self.slot_down), max_tokens, phases, ctypes.byref(h))
        self.handle = h
        self.copy_stream = torch.cuda.Stream(device=dev)

    def workspace_size(self, T):
        n = ctypes.c_size_t()
        _call("dq_expert_cache_workspace_size", self.handle, T, ctypes.byref(n))
        return n.value

    def forward(self, x, y=None, ws=None):
        """The layer for x [T][hidden] on the current stream (copies on this
        cache's copy stream)."""
        T = x.shape[0]
        if y is None:
            y = torch.empty(T, self.desc.hidden, dtype=torch.float32, device=x.device)
        if ws is None:
            ws = torch.empty(self.workspace_size(T), dtype=torch.uint8, device=x.device)
        _call("dq_moe_forward_streamed", self.handle, _ptr(x), _dtype_code(x), T, _ptr(y),
              _ptr(ws), ws.numel(), _stream(), ctypes.c_void_p(self.copy_stream.cuda_stream))
        return y

    def stats(self):
        h, m, b = ctypes.c_longlong(), ctypes.c_longlong(), ctypes.c_longlong()
        _call("dq_expert_cache_stats", self.handle, ctypes.byref(h), ctypes.byref(m),
              ctypes.byref(b))
        return {"hits": h.value, "misses": m.value, "bytes_copied": b.value}

    def close(self):
        if self.handle:
            _call("dq_expert_cache_destroy", self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
