"""Writes q2_k_blocks.txt and q3_k_blocks.txt: hand-packed Q2_K / Q3_K
super-blocks and their decoded weights.

Each case packs its bytes from a few stated field values and computes every
expected weight from the format's closed form (stated on the case's '#'
line), with plain integer and float arithmetic: it calls neither the oracle
nor the CUDA library, so the fixtures pin the oracle from outside it.

    python tests/golden/make_low_bit_blocks.py     # rewrites both files
"""
import os
import struct

HERE = os.path.dirname(os.path.abspath(__file__))


def f16(v):
    return struct.pack("<e", v)


def hexs(b):
    return " ".join("%02x" % x for x in b)


def floats(ws):
    return " ".join(repr(float(w)) for w in ws)


# ---------------------------------------------------------------------------
# Q2_K: scales[16] (scale | min << 4 per 16-weight sub-block), qs[64], fp16 d,
# fp16 dmin.  Weight 128h + 32r + l takes bits 2r..2r+1 of qs[32h + l];
# w = d*(sc & 15)*q - dmin*(sc >> 4).
# ---------------------------------------------------------------------------
def q2k_block(sc, qs, d, dmin):
    assert len(sc) == 16 and len(qs) == 64
    return bytes(sc) + bytes(qs) + f16(d) + f16(dmin)


def q2k_weights(sc, qs, d, dmin):
    w = [0.0] * 256
    for h in range(2):
        for r in range(4):
            for l in range(32):
                i = 128 * h + 32 * r + l
                q = (qs[32 * h + l] >> (2 * r)) & 3
                s = sc[i // 16]
                w[i] = d * (s & 15) * q - dmin * (s >> 4)
    return w


Q2K_HEAD = """# Hand-packed Q2_K super-blocks (84 B) and their decoded weights.
# Format named by: KTransformers, section 支持的量化格式 (Q2_K_L / Q2_K_XS mixes).
# Byte layout: GGUF/llama.cpp reading (scales[16] = scale | min << 4 per
# 16-weight sub-block, qs[64] of 2-bit quants, fp16 d, fp16 dmin).  Weight
# 128h + 32r + l takes bits 2r..2r+1 of qs[32h + l], closed form
# w = d*(sc & 15)*q - dmin*(sc >> 4).  Each case's values follow from it by hand
# (stated on the '#' line).
"""

Q2K_CASES = [
    ("scale_walk", "q = 1, sc_j = j, min 0, d = 1: w[i] = i//16",
     list(range(16)), [0x55] * 64, 1.0, 0.0),
    ("min_walk", "q = 0, min_j = j, dmin = 0.5: w[i] = -0.5*(i//16)",
     [j << 4 for j in range(16)], [0] * 64, 1.0, 0.5),
    ("field_walk", "qs bytes 0xE4 (fields 0,1,2,3), sc 1, d 1: w[128h+32r+l] = r",
     [1] * 16, [0xE4] * 64, 1.0, 0.0),
    ("byte_walk", "qs[32h+l] = l, sc 1, d 1: w[128h+32r+l] = (l >> 2r) & 3",
     [1] * 16, list(range(32)) * 2, 1.0, 0.0),
    ("scale_and_min", "q = 3, scale 1, min 3, d 2, dmin 1: w = 2*3 - 3 = 3",
     [0x31] * 16, [0xFF] * 64, 2.0, 1.0),
]


# ---------------------------------------------------------------------------
# Q3_K: hmask[32], qs[64] of 2-bit low quants, 12 bytes of sixteen 6-bit
# scales, fp16 d.  Weight 128h + 32r + l: low bits 2r..2r+1 of qs[32h + l],
# high bit = bit 4h + r of hmask[l]; q = low - 4 when the high bit is clear.
# Scale j: low nibble = nibble j//8 of scales[j % 8], high two bits = bits
# 2(j//4).. of scales[8 + j % 4]; w = d*(s_j - 32)*q.
# ---------------------------------------------------------------------------
def q3k_pack_scales(s):
    assert len(s) == 16 and all(0 <= v < 64 for v in s)
    b = [0] * 12
    for j in range(16):
        b[j % 8] |= (s[j] & 15) << (4 * (j // 8))
        b[8 + j % 4] |= (s[j] >> 4) << (2 * (j // 4))
    return bytes(b)


def q3k_block(hmask, qs, s, d):
    assert len(hmask) == 32 and len(qs) == 64
    return bytes(hmask) + bytes(qs) + q3k_pack_scales(s) + f16(d)


def q3k_weights(hmask, qs, s, d):
    w = [0.0] * 256
    for h in range(2):
        for r in range(4):
            for l in range(32):
                i = 128 * h + 32 * r + l
                low = (qs[32 * h + l] >> (2 * r)) & 3
                high = (hmask[l] >> (4 * h + r)) & 1
                q = low if high else low - 4
                w[i] = d * (s[i // 16] - 32) * q
    return w


Q3K_HEAD = """# Hand-packed Q3_K super-blocks (110 B) and their decoded weights.
# Format named by: KTransformers, section 支持的量化格式 (Q3_K_M mix).
# Byte layout: GGUF/llama.cpp reading (hmask[32], qs[64] of 2-bit low quants,
# 12 bytes of sixteen 6-bit scales, fp16 d).  Weight 128h + 32r + l: low bits
# 2r..2r+1 of qs[32h + l], high bit = bit 4h + r of hmask[l]; q = low - 4 when
# the high bit is clear.  Scale j: low nibble = nibble j//8 of scales[j % 8],
# high two bits = bits 2(j//4).. of scales[8 + j % 4]; w = d*(s_j - 32)*q.
# Each case's values follow from the closed form by hand (stated on the '#' line).
"""

Q3K_CASES = [
    ("high_set", "hmask all set, qs 0xE4, every s_j = 33, d = 1: w[128h+32r+l] = r",
     [0xFF] * 32, [0xE4] * 64, [33] * 16, 1.0),
    ("high_clear", "hmask clear, qs 0xE4, every s_j = 33, d = 1: w = r - 4",
     [0x00] * 32, [0xE4] * 64, [33] * 16, 1.0),
    ("scale_low_walk", "q = 1, s_j = j (high scale bits 0), d = 1: w[i] = i//16 - 32",
     [0xFF] * 32, [0x55] * 64, list(range(16)), 1.0),
    ("scale_high_walk", "q = 1, s_j = 16*(j % 4), d = 0.5: w[i] = 8*((i//16) % 4) - 16",
     [0xFF] * 32, [0x55] * 64, [16 * (j % 4) for j in range(16)], 0.5),
    ("hmask_walk", "hmask[l] = 1 << (l % 8), low quants 0, s_j = 33, d = 1:\n"
     "# w[128h+32r+l] = 0 where l % 8 == 4h + r, else -4",
     [1 << (l % 8) for l in range(32)], [0] * 64, [33] * 16, 1.0),
]


def write(path, head, cases, block, weights):
    lines = [head.rstrip("\n")]
    for name, note, *args in cases:
        lines.append("case " + name)
        lines.append("# " + note)
        lines.append("bytes " + hexs(block(*args)))
        lines.append("expect " + floats(weights(*args)))
    with open(path, "w", encoding="utf-8") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    write(os.path.join(HERE, "q2_k_blocks.txt"), Q2K_HEAD, Q2K_CASES, q2k_block, q2k_weights)
    write(os.path.join(HERE, "q3_k_blocks.txt"), Q3K_HEAD, Q3K_CASES, q3k_block, q3k_weights)
