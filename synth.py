"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method: it only draws random bytes and
numbers in the shapes and distributions of the workloads and packs them into
the block byte layouts (field placement only).  Both the CUDA library and the
CPU oracle receive exactly these arrays.

Recipe (the pages name no dataset; everything is synthetic):
  * numpy Generator(PCG64(seed)); one spawned child stream per tensor, so a
    tensor's values do not depend on the shapes of the others.
  * Q4_K: d, dmin = |N(0,1)| * 0.01 rounded to fp16; the 12 scale bytes and
    128 quant bytes uniform over 0..255 (so every 6-bit field is uniform).
  * Q6_K: ql, qh and the 16 int8 scale bytes uniform over 0..255; d as Q4_K.
  * Q8_0: d as Q4_K; the 32 int8 quants uniform over -127..127.
  * Q4_0: d as Q4_K; the 16 quant bytes uniform.  Q5_K: as Q4_K, plus the
    32 fifth-bit bytes uniform.
  * Q2_K: the 16 scale/min bytes and 64 quant bytes uniform; d at 80 and
    dmin at 82 as Q4_K.  Q3_K: hmask, quants and the 12 scale bytes uniform;
    d at 108 as Q4_K.
  * NVFP4: the 128 code bytes uniform; the 16 E4M3 scale bytes positive with
    exponent field uniform over 1..6 and mantissa field uniform (scales
    2^-6 .. 2^-1 * 1.875: weights within +-0.7, the range of Q4_K's).
  * activations N(0,1), drawn in fp32 and rounded to nearest-even into the
    activation dtype; router weights N(0, 0.02) fp32.
"""
import numpy as np

BLOCK = {1: (256, 144), 2: (256, 210), 3: (32, 34), 4: (32, 18), 5: (256, 176),
         6: (256, 144), 7: (256, 84), 8: (256, 110)}  # fmt -> (weights, bytes)
FMT_NAMES = {"q4_k": 1, "q6_k": 2, "q8_0": 3, "q4_0": 4, "q5_k": 5, "nvfp4": 6, "q2_k": 7,
             "q3_k": 8}
DT_NAMES = {"f32": 0, "f16": 1, "bf16": 2}
BASE_SEED = 20261202


def streams(seed, n):
    """n independent child generators of one seed."""
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(n)]


def _scale_f16(rng, n):
    return (np.abs(rng.standard_normal(n, dtype=np.float32)) * np.float32(0.01)).astype(np.float16)


def quant_matrix(rng, fmt, rows, cols):
    """Random blocks of `fmt` for a [rows][cols] matrix, as a flat uint8 array."""
    qk, nbytes = BLOCK[fmt]
    assert cols % qk == 0
    nblk = rows * (cols // qk)
    raw = np.frombuffer(rng.bytes(nblk * nbytes), dtype=np.uint8).copy()
    blk = raw.reshape(nblk, nbytes)
    if fmt == 1:        # Q4_K: d at 0, dmin at 2
        blk[:, 0:2] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
        blk[:, 2:4] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
    elif fmt == 2:      # Q6_K: d at 208
        blk[:, 208:210] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
    elif fmt == 3:      # Q8_0: d at 0, quants -127..127
        blk[:, 0:2] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
        blk[:, 2:34] = rng.integers(-127, 128, size=(nblk, 32), dtype=np.int8).view(np.uint8)
    elif fmt == 4:      # Q4_0: d at 0
        blk[:, 0:2] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
    elif fmt == 5:      # Q5_K: d at 0, dmin at 2 (as Q4_K)
        blk[:, 0:2] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
        blk[:, 2:4] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
    elif fmt == 7:      # Q2_K: d at 80, dmin at 82
        blk[:, 80:82] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
        blk[:, 82:84] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
    elif fmt == 8:      # Q3_K: d at 108
        blk[:, 108:110] = _scale_f16(rng, nblk).view(np.uint8).reshape(nblk, 2)
    else:               # NVFP4: 16 positive E4M3 scale bytes with exponent field 1..6
        ef = rng.integers(1, 7, size=(nblk, 16), dtype=np.uint8)
        mf = rng.integers(0, 8, size=(nblk, 16), dtype=np.uint8)
        blk[:, 0:16] = (ef << 3) | mf
    return raw


def f32_to_bf16_bits(a):
    """Round fp32 to bfloat16 (nearest-even), returned as uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(rng, shape, dtype):
    """N(0,1) activations in dtype 0=f32, 1=f16, 2=bf16 (bf16 as uint16 bits)."""
    a = rng.standard_normal(shape, dtype=np.float32)
    if dtype == 0:
        return a
    if dtype == 1:
        return a.astype(np.float16)
    return f32_to_bf16_bits(a)


def router_weights(rng, E, H):
    return (rng.standard_normal((E, H), dtype=np.float32) * np.float32(0.02)).astype(np.float32)


# ---------------------------------------------------------------------------
# The five workloads: shapes exactly as specified.
# ---------------------------------------------------------------------------
LLAMA8B_LINEARS = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096),
                   ("o", 4096, 4096), ("gate", 14336, 4096), ("up", 14336, 4096),
                   ("down", 4096, 14336)]
# the same matrices as inference engines store them: q, k, v stacked into one
# [6144 x 4096] matrix and gate, up into one [28672 x 4096] matrix (identical
# bytes and products; four GEMV launches per layer instead of seven)
LLAMA8B_MERGED = [("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 28672, 4096),
                  ("down", 4096, 14336)]
LLAMA70B_LINEARS = [("gate", 28672, 8192), ("up", 28672, 8192),
                    ("down", 8192, 28672), ("q", 8192, 8192)]

GEMV_SINGLE = dict(name="q4k_256x1024_b1_f32", fmt=1, N=256, K=1024, batch=1, xdt=0)
MOE_MIXTRAL = dict(name="mixtral_moe", E=8, top_k=2, H=4096, F=14336, n_shared=0,
                   fmt=1, T=(16,), xdt=1)
MOE_DEEPSEEK = dict(name="deepseek_v3_moe", E=256, top_k=8, H=7168, F=2048, n_shared=1,
                    fmt=1, T=(1, 8, 256), xdt=2)


def moe_weights(seed, E, H, F, n_shared, fmt):
    """Router and stacked expert matrices of one MoE layer."""
    g = streams(seed, 8)
    return dict(
        router_W=router_weights(g[0], E, H),
        w_gate=quant_matrix(g[1], fmt, E * F, H),
        w_up=quant_matrix(g[2], fmt, E * F, H),
        w_down=quant_matrix(g[3], fmt, E * H, F),
        sh_gate=quant_matrix(g[4], fmt, n_shared * F, H) if n_shared else None,
        sh_up=quant_matrix(g[5], fmt, n_shared * F, H) if n_shared else None,
        sh_down=quant_matrix(g[6], fmt, n_shared * H, F) if n_shared else None,
    )
