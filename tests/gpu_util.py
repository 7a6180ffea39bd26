"""Helpers for the GPU parity tests: move synth arrays to the device."""
import numpy as np
import torch


def dev_bytes(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_act(a, xdt):
    """numpy activations from synth.activations -> torch CUDA tensor of the dtype."""
    if xdt == 0:
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    if xdt == 1:
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16)).cuda()
    bits = np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(bits).cuda().view(torch.bfloat16)


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.abs(ref).max()
    return np.abs(got - ref).max() / (scale if scale > 0 else 1.0)


TOL = {0: 1e-5, 1: 2e-3, 2: 2e-3}   # fp32 / fp16 / bf16 activations
