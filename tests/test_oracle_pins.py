"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks the oracle against something the formats' closed forms, the
mathematics or a library routine fix independently:
  * hand-packed blocks whose decoded values follow by hand from the closed
    forms (tests/golden/*.txt);
  * exact conversions of every fp16 / bf16 bit pattern (numpy's own);
  * brute force with numpy's matmul on tiny shapes, plus an integer case that
    is exact in any precision;
  * numpy's stable sort for top-k / permute, scipy's softmax for k = E;
  * the MoE invariant: the layer equals a dense all-experts
    compute masked to the selected experts.
A plausible slip anywhere in the oracle (a swapped nibble, a wrong 6-bit
field, a transposed operand, a dropped min term, a reversed tie-break, a
missing renormalisation or shared expert) fails at least one of these.
"""
import numpy as np
import pytest
from scipy.special import softmax

import synth
from golden_io import read_block_cases

Q4_K, Q6_K, Q8_0, Q4_0, Q5_K, NVFP4, Q2_K, Q3_K = 1, 2, 3, 4, 5, 6, 7, 8


# ---------------------------------------------------------------------------
# block decode: hand-packed special cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fname,fmt,qk", [("q4_k_blocks.txt", Q4_K, 256),
                                          ("q6_k_blocks.txt", Q6_K, 256),
                                          ("q8_0_blocks.txt", Q8_0, 32),
                                          ("q2_k_blocks.txt", Q2_K, 256),
                                          ("q3_k_blocks.txt", Q3_K, 256)])
def test_dequant_golden_blocks(orc, fname, fmt, qk):
    cases = read_block_cases(fname)
    assert len(cases) >= 3
    for c in cases:
        got = orc.dequant(fmt, c["bytes"], qk).astype(np.float64)
        np.testing.assert_array_equal(got, c["expect"], err_msg=c["name"])


def test_dequant_blocks_independent(orc):
    # decoding two blocks at once equals decoding each alone (no state leaks
    # across blocks; the block stride is the format's byte size)
    g = synth.streams(7, 3)
    for i, (fmt, qk, nb) in enumerate([(Q4_K, 256, 144), (Q6_K, 256, 210), (Q8_0, 32, 34),
                                       (Q2_K, 256, 84), (Q3_K, 256, 110)]):
        raw = synth.quant_matrix(g[i % 3], fmt, 3, qk)
        both = orc.dequant(fmt, raw, 3 * qk)
        for i in range(3):
            one = orc.dequant(fmt, raw[i * nb:(i + 1) * nb], qk)
            np.testing.assert_array_equal(both[i * qk:(i + 1) * qk], one)


def test_q4k_scale_bits_each_feed_one_field(orc):
    # Every one of the 96 bits of the 12 scale bytes changes exactly one
    # sub-block (32 consecutive weights) and by a power of two of d or dmin:
    # no bit is dropped and no two fields overlap.
    base = np.zeros(144, dtype=np.uint8)
    base[0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)   # d = 1
    base[2:4] = np.array([1.0], dtype=np.float16).view(np.uint8)   # dmin = 1
    base[16:] = 0x11                                               # q = 1
    ref = orc.dequant(Q4_K, base, 256).astype(np.float64)
    np.testing.assert_array_equal(ref, 0.0)
    seen = set()
    for byte in range(12):
        for bit in range(8):
            blk = base.copy()
            blk[4 + byte] = 1 << bit
            diff = orc.dequant(Q4_K, blk, 256).astype(np.float64) - ref
            nz = np.nonzero(diff)[0]
            assert nz.size == 32, (byte, bit)
            sb = nz[0] // 32
            assert np.all(nz // 32 == sb)
            v = diff[nz[0]]
            assert np.all(diff[nz] == v)
            mag = abs(v)
            assert mag == 2.0 ** round(np.log2(mag)) and 1 <= mag <= 32
            field = (sb, v > 0, int(np.log2(mag)))   # (sub-block, scale vs min, bit)
            assert field not in seen
            seen.add(field)
    # 8 sub-blocks x (6 scale bits + 6 min bits) = 96 distinct fields
    assert len(seen) == 96


def test_q6k_bits_each_feed_one_weight(orc):
    # Each bit of ql / qh changes exactly one weight (d = 1, all scales 1), by
    # 2^(bit position inside that weight's 6-bit q); every weight is reached
    # by exactly 6 bits.
    base = np.zeros(210, dtype=np.uint8)
    base[192:208] = 1
    base[208:210] = np.array([1.0], dtype=np.float16).view(np.uint8)
    ref = orc.dequant(Q6_K, base, 256).astype(np.float64)
    np.testing.assert_array_equal(ref, -32.0)
    hits = np.zeros(256, dtype=np.int64)
    mags = [set() for _ in range(256)]
    for byte in range(192):
        for bit in range(8):
            blk = base.copy()
            blk[byte] = 1 << bit
            diff = orc.dequant(Q6_K, blk, 256).astype(np.float64) - ref
            nz = np.nonzero(diff)[0]
            assert nz.size == 1, (byte, bit)
            w = nz[0]
            hits[w] += 1
            mags[w].add(diff[w])
            # the four low bits come from ql, the two high bits from qh
            assert (byte < 128) == (diff[w] < 16)
    assert np.all(hits == 6)
    assert all(m == {1.0, 2.0, 4.0, 8.0, 16.0, 32.0} for m in mags)


# ---------------------------------------------------------------------------
# activation conversions: every bit pattern
# ---------------------------------------------------------------------------
def test_f16_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = orc.act_to_f64(1, bits)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    assert np.all(np.isnan(got[np.isnan(ref)]))
    assert np.all(got[np.isinf(ref)] == ref[np.isinf(ref)])


def test_bf16_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = orc.act_to_f64(2, bits)
    fin = np.isfinite(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])


def test_synth_bf16_rounding_is_nearest_even():
    # input-generator check: bf16 rounding equals the exact nearest bf16
    x = np.random.default_rng(3).standard_normal(10000).astype(np.float32)
    b = synth.f32_to_bf16_bits(x)
    v = synth.bf16_bits_to_f32(b).astype(np.float64)
    up = synth.bf16_bits_to_f32(b + 1).astype(np.float64)
    dn = synth.bf16_bits_to_f32(b - 1).astype(np.float64)
    err = np.abs(v - x)
    assert np.all(err <= np.abs(up - x)) and np.all(err <= np.abs(dn - x))


# ---------------------------------------------------------------------------
# Q4_0 and Q5_K: reductions to the pinned formats, and bit walks
# ---------------------------------------------------------------------------
def test_q40_equals_q80_with_shifted_quants(orc):
    # a Q4_0 block is a Q8_0 block whose int8 quants are the nibbles minus 8,
    # low nibbles first (weights 0..15), then high nibbles (16..31)
    rng = np.random.default_rng(404)
    nblk = 64
    q40 = np.frombuffer(rng.bytes(nblk * 18), dtype=np.uint8).copy().reshape(nblk, 18)
    q40[:, 0:2] = (np.abs(rng.standard_normal(nblk)) * 0.01).astype(np.float16).view(np.uint8).reshape(nblk, 2)
    q80 = np.zeros((nblk, 34), dtype=np.uint8)
    q80[:, 0:2] = q40[:, 0:2]
    nib = q40[:, 2:18]
    q80[:, 2:18] = ((nib & 15).astype(np.int16) - 8).astype(np.int8).view(np.uint8)
    q80[:, 18:34] = ((nib >> 4).astype(np.int16) - 8).astype(np.int8).view(np.uint8)
    a = orc.dequant(Q4_0, q40.reshape(-1), nblk * 32)
    b = orc.dequant(Q8_0, q80.reshape(-1), nblk * 32)
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_q40_nibble_walk(orc):
    # d = 0.5, every nibble 8 (weight 0); raising one nibble to 11 gives 1.5 at
    # exactly one position: low nibble of byte j -> weight j, high -> j + 16
    base = np.zeros(18, dtype=np.uint8)
    base[0:2] = np.array([0.5], dtype=np.float16).view(np.uint8)
    base[2:18] = 0x88
    assert np.all(orc.dequant(Q4_0, base, 32) == 0.0)
    for j in range(16):
        for hi in (0, 1):
            b = base.copy()
            b[2 + j] = 0x8B if hi == 0 else 0xB8
            w = orc.dequant(Q4_0, b, 32)
            want = np.zeros(32, dtype=np.float32)
            want[j + 16 * hi] = 1.5
            np.testing.assert_array_equal(w, want)


def test_q5k_without_fifth_bits_is_q4k(orc):
    # with every qh byte zero a Q5_K block decodes as the Q4_K block made of
    # the same d, dmin, scale bytes and low quants
    rng = np.random.default_rng(505)
    q4 = synth.quant_matrix(rng, Q4_K, 8, 1024).reshape(-1, 144)
    q5 = np.zeros((q4.shape[0], 176), dtype=np.uint8)
    q5[:, 0:16] = q4[:, 0:16]
    q5[:, 48:176] = q4[:, 16:144]
    n = q4.shape[0] * 256
    a = orc.dequant(Q5_K, q5.reshape(-1), n)
    b = orc.dequant(Q4_K, q4.reshape(-1), n)
    np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_q5k_fifth_bit_walk(orc):
    # d = 1, dmin = 0, every 6-bit scale 1 and min 0, low quants 0: all weights
    # 0.  Setting bit i of qh[l] must add 16 to exactly one weight:
    # 64*(i//2) + l for even i, 64*(i//2) + 32 + l for odd i.
    base = np.zeros(176, dtype=np.uint8)
    base[0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
    base[4:8] = 1          # sc_0..3 = 1 (m_0..3 = 0 from bytes 8..11)
    base[12:16] = 0x01     # sc_4..7 = 1, m_4..7 = 0
    assert np.all(orc.dequant(Q5_K, base, 256) == 0.0)
    for i in range(8):
        for l in (0, 1, 17, 31):
            b = base.copy()
            b[16 + l] = 1 << i
            w = orc.dequant(Q5_K, b, 256)
            want = np.zeros(256, dtype=np.float32)
            want[64 * (i // 2) + 32 * (i % 2) + l] = 16.0
            np.testing.assert_array_equal(w, want)


# ---------------------------------------------------------------------------
# Q2_K / Q3_K: bit walks, a reduction of one to the other
# ---------------------------------------------------------------------------
def _q2k_block(sc, qs, d, dmin):
    b = np.zeros(84, dtype=np.uint8)
    b[0:16] = sc
    b[16:80] = qs
    b[80:82] = np.array([d], dtype=np.float16).view(np.uint8)
    b[82:84] = np.array([dmin], dtype=np.float16).view(np.uint8)
    return b


def _q3k_block(hm, qs, sc, d):
    b = np.zeros(110, dtype=np.uint8)
    b[0:32] = hm
    b[32:96] = qs
    b[96:108] = sc
    b[108:110] = np.array([d], dtype=np.float16).view(np.uint8)
    return b


def test_q2k_quant_bits_each_feed_one_weight(orc):
    # d = 1, every scale 1, min 0: each of the 512 quant bits moves exactly one
    # weight, by 1 (low bit of its field) or 2 (high bit); every weight is
    # reached by exactly two bits, one of each.
    base = _q2k_block(np.full(16, 1), np.zeros(64), 1.0, 0.0)
    assert np.all(orc.dequant(Q2_K, base, 256) == 0.0)
    mags = [[] for _ in range(256)]
    for byte in range(64):
        for bit in range(8):
            b = base.copy()
            b[16 + byte] = 1 << bit
            w = orc.dequant(Q2_K, b, 256).astype(np.float64)
            nz = np.nonzero(w)[0]
            assert nz.size == 1, (byte, bit)
            mags[nz[0]].append(w[nz[0]])
    assert all(sorted(m) == [1.0, 2.0] for m in mags)


def test_q2k_scale_bits_each_feed_one_field(orc):
    # q = 1 everywhere, d = dmin = 1: bit k of scale byte j changes exactly the
    # 16 weights of sub-block j, by +2^k (scale nibble) or -2^(k-4) (min nibble)
    base = _q2k_block(np.zeros(16), np.full(64, 0x55), 1.0, 1.0)
    assert np.all(orc.dequant(Q2_K, base, 256) == 0.0)
    for j in range(16):
        for k in range(8):
            b = base.copy()
            b[j] = 1 << k
            w = orc.dequant(Q2_K, b, 256).astype(np.float64)
            want = np.zeros(256)
            want[16 * j:16 * j + 16] = 2.0 ** k if k < 4 else -(2.0 ** (k - 4))
            np.testing.assert_array_equal(w, want, err_msg=str((j, k)))


def test_q3k_bits_each_feed_one_weight(orc):
    # d = 1, every scale s = 33 (factor 1), all high bits set, low quants 0: all
    # weights 0.  Each low-quant bit raises exactly one weight by 1 or 2 and
    # each hmask bit, cleared, lowers exactly one weight by 4; every weight
    # is reached by two low bits and one hmask bit.
    sc = np.array([0x11] * 8 + [0xAA] * 4, dtype=np.uint8)
    base = _q3k_block(np.full(32, 0xFF), np.zeros(64), sc, 1.0)
    assert np.all(orc.dequant(Q3_K, base, 256) == 0.0)
    mags = [[] for _ in range(256)]
    for byte in range(64):
        for bit in range(8):
            b = base.copy()
            b[32 + byte] = 1 << bit
            w = orc.dequant(Q3_K, b, 256).astype(np.float64)
            nz = np.nonzero(w)[0]
            assert nz.size == 1, (byte, bit)
            mags[nz[0]].append(w[nz[0]])
    for byte in range(32):
        for bit in range(8):
            b = base.copy()
            b[byte] = 0xFF ^ (1 << bit)
            w = orc.dequant(Q3_K, b, 256).astype(np.float64)
            nz = np.nonzero(w)[0]
            assert nz.size == 1, (byte, bit)
            mags[nz[0]].append(w[nz[0]])
    assert all(sorted(m) == [-4.0, 1.0, 2.0] for m in mags)


def test_q3k_scale_bits_each_feed_one_field(orc):
    # q = 1 everywhere, d = 1, all scale bytes 0 (s = 0, w = -32): each of the
    # 96 scale bits raises exactly one sub-block of 16 weights by a power of
    # two from 1 to 32; the 96 bits make 16 sub-blocks x 6 distinct bits.
    base = _q3k_block(np.full(32, 0xFF), np.full(64, 0x55), np.zeros(12), 1.0)
    np.testing.assert_array_equal(orc.dequant(Q3_K, base, 256), -32.0)
    seen = set()
    for byte in range(12):
        for bit in range(8):
            b = base.copy()
            b[96 + byte] = 1 << bit
            diff = orc.dequant(Q3_K, b, 256).astype(np.float64) + 32.0
            nz = np.nonzero(diff)[0]
            assert nz.size == 16 and nz[0] % 16 == 0 and np.all(np.diff(nz) == 1), (byte, bit)
            v = diff[nz[0]]
            assert np.all(diff[nz] == v) and v == 2.0 ** round(np.log2(v)) and 1 <= v <= 32
            field = (nz[0] // 16, int(np.log2(v)))
            assert field not in seen
            seen.add(field)
            # the low nibbles (bytes 0..7) carry the four low scale bits
            assert (byte < 8) == (v < 16)
    assert len(seen) == 96


def test_q3k_with_high_bits_set_is_q2k(orc):
    # every hmask bit set and every 6-bit scale 33 (factor 1): Q3_K decodes as
    # the Q2_K block of the same quant bytes and d with scale 1, min 0
    rng = np.random.default_rng(707)
    sc3 = np.array([0x11] * 8 + [0xAA] * 4, dtype=np.uint8)
    for _ in range(4):
        qs = rng.integers(0, 256, size=64)
        d = float(np.float16(abs(rng.standard_normal()) * 0.01))
        a = orc.dequant(Q3_K, _q3k_block(np.full(32, 0xFF), qs, sc3, d), 256)
        b = orc.dequant(Q2_K, _q2k_block(np.full(16, 1), qs, d, 0.0), 256)
        np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# NVFP4: the E2M1 and E4M3 value tables, a reduction to Q8_0, placement walks
# ---------------------------------------------------------------------------
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]   # codes 0..15


def _nvfp4_block(scales, codes):
    b = np.zeros(144, dtype=np.uint8)
    b[0:16] = scales
    c = np.asarray(codes, dtype=np.uint8)
    b[16:144] = c[0::2] | (c[1::2] << 4)
    return b


def test_nvfp4_e2m1_table(orc):
    # scale 0x38 = 1.0: weight i shows the code's E2M1 value
    codes = np.arange(256) % 16
    w = orc.dequant(NVFP4, _nvfp4_block(np.full(16, 0x38), codes), 256)
    np.testing.assert_array_equal(w, np.array([E2M1_TABLE[c] for c in codes], dtype=np.float32))
    assert np.signbit(w[8])                       # code 8 is -0


def test_nvfp4_e4m3_scale_values(orc):
    # code 2 (= 1.0) times the block's scale: E4M3 values of the FP8 definition
    # (bias 7; exponent 0 subnormal m/8 * 2^-6; max 448)
    cases = {0x38: 1.0, 0x30: 0.5, 0x3F: 1.875, 0x40: 2.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
             0x08: 2.0 ** -6, 0x7E: 448.0, 0xC0: -2.0, 0x00: 0.0, 0x5C: 24.0}
    items = list(cases.items())
    for i in range(0, len(items), 16):
        chunk = items[i:i + 16]
        scales = np.full(16, 0x38, dtype=np.uint8)
        for j, (byte, _) in enumerate(chunk):
            scales[j] = byte
        w = orc.dequant(NVFP4, _nvfp4_block(scales, np.full(256, 2)), 256)
        for j, (byte, val) in enumerate(chunk):
            np.testing.assert_array_equal(w[16 * j:16 * j + 16], np.float32(val), err_msg=hex(byte))


def test_nvfp4_equals_q80_at_unit_scale(orc):
    # with every scale 1.0 an NVFP4 super-block is eight Q8_0 blocks with
    # d = 0.5 and q = 2 * the E2M1 value (integers 0, +-1, .., +-12)
    rng = np.random.default_rng(606)
    codes = rng.integers(0, 16, size=256)
    a = orc.dequant(NVFP4, _nvfp4_block(np.full(16, 0x38), codes), 256)
    q80 = np.zeros((8, 34), dtype=np.uint8)
    q80[:, 0:2] = np.array([0.5], dtype=np.float16).view(np.uint8)
    q = np.array([int(2 * E2M1_TABLE[c]) for c in codes], dtype=np.int8).reshape(8, 32)
    q80[:, 2:34] = q.view(np.uint8)
    b = orc.dequant(Q8_0, q80.reshape(-1), 256)
    np.testing.assert_array_equal(np.abs(a), np.abs(b))
    np.testing.assert_array_equal(a[a != 0], b[a != 0])


def test_nvfp4_placement_walk(orc):
    # one scale byte doubled -> exactly its 16 weights double; one code set ->
    # exactly weight 2i (low nibble of byte i) or 2i+1 (high nibble)
    for blk in range(16):
        scales = np.full(16, 0x38, dtype=np.uint8)
        scales[blk] = 0x40
        w = orc.dequant(NVFP4, _nvfp4_block(scales, np.full(256, 2)), 256)
        want = np.ones(256, dtype=np.float32)
        want[16 * blk:16 * blk + 16] = 2.0
        np.testing.assert_array_equal(w, want)
    for i in (0, 1, 2, 127, 128, 254, 255):
        codes = np.zeros(256, dtype=np.int64)
        codes[i] = 7
        w = orc.dequant(NVFP4, _nvfp4_block(np.full(16, 0x38), codes), 256)
        want = np.zeros(256, dtype=np.float32)
        want[i] = 6.0
        np.testing.assert_array_equal(w, want)


# ---------------------------------------------------------------------------
# qGEMV: brute force against numpy on tiny shapes; an exact integer case
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [Q4_K, Q6_K, Q8_0, Q4_0, Q5_K, NVFP4, Q2_K, Q3_K])
@pytest.mark.parametrize("xdt", [0, 1, 2])
def test_qgemv_brute_force(orc, fmt, xdt):
    g = synth.streams(100 + fmt * 10 + xdt, 4)
    for N, K, B in [(1, 256, 1), (5, 512, 3), (8, 256, 8), (3, 768, 4)]:
        W = synth.quant_matrix(g[0], fmt, N, K)
        x = synth.activations(g[1], (B, K), xdt)
        y = orc.qgemv(fmt, W, N, K, x, xdt, B)
        Wd = orc.dequant(fmt, W, N * K).astype(np.float64).reshape(N, K)
        xd = orc.act_to_f64(xdt, x).reshape(B, K)
        ref = (xd @ Wd.T).astype(np.float32)
        np.testing.assert_allclose(y, ref, rtol=2e-7, atol=1e-6 * np.abs(ref).max())
        # rows subset gives the same rows
        rows = np.array([N - 1, 0], dtype=np.int64)
        ys = orc.qgemv(fmt, W, N, K, x, xdt, B, rows=rows)
        np.testing.assert_array_equal(ys, y[:, rows])


def test_qgemv_exact_integer_case(orc):
    # Q8_0 with d = 1 and small integer quants, integer activations in fp16:
    # the product is an integer matrix product, exact in every precision.
    N, K, B = 6, 96, 3
    rng = np.random.default_rng(11)
    q = rng.integers(-9, 10, size=(N, K)).astype(np.int64)
    blocks = np.zeros((N, K // 32, 34), dtype=np.uint8)
    blocks[:, :, 0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
    blocks[:, :, 2:] = q.reshape(N, K // 32, 32).astype(np.int8).view(np.uint8)
    xi = rng.integers(-5, 6, size=(B, K)).astype(np.int64)
    y = orc.qgemv(Q8_0, blocks.ravel(), N, K, xi.astype(np.float16), 1, B)
    np.testing.assert_array_equal(y, (xi @ q.T).astype(np.float32))


def test_qgemv_transposition_sensitive(orc):
    # a non-square case where W and W^T would both fit: y[b][n] must use row n
    N, K = 2, 256
    W = np.zeros((N, 34 * 8), dtype=np.uint8).reshape(N, 8, 34)
    W[:, :, 0:2] = np.array([1.0], dtype=np.float16).view(np.uint8)
    W[0, 0, 2] = 1            # W[0][0] = 1
    W[1, 7, 2 + 31] = 3       # W[1][255] = 3
    x = np.zeros((1, K), dtype=np.float32)
    x[0, 0], x[0, 255] = 2.0, 5.0
    y = orc.qgemv(Q8_0, W.ravel(), N, K, x, 0, 1)
    np.testing.assert_array_equal(y, [[2.0, 15.0]])


# ---------------------------------------------------------------------------
# router, top-k, gates
# ---------------------------------------------------------------------------
def test_router_logits_vs_matmul(orc):
    g = synth.streams(5, 2)
    E, H, T = 16, 512, 7
    Wr = synth.router_weights(g[0], E, H)
    for xdt in (0, 1, 2):
        x = synth.activations(g[1], (T, H), xdt)
        L = orc.router_logits(Wr, E, H, x, xdt, T)
        ref = orc.act_to_f64(xdt, x).reshape(T, H) @ Wr.astype(np.float64).T
        np.testing.assert_allclose(L, ref, rtol=1e-12, atol=1e-12)


def test_topk_matches_stable_sort(orc):
    rng = np.random.default_rng(9)
    T, E = 40, 32
    # coarse values make many exact ties
    L = rng.integers(-3, 4, size=(T, E)).astype(np.float64)
    for k in (1, 2, 5, 8, 32):
        idx, gate = orc.topk(L, k)
        for t in range(T):
            order = np.lexsort((np.arange(E), -L[t]))   # by -logit, then index
            np.testing.assert_array_equal(idx[t], order[:k])
        np.testing.assert_allclose(gate.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_topk_ties_take_lowest_index(orc):
    L = np.zeros((1, 8))
    idx, gate = orc.topk(L, 3)
    np.testing.assert_array_equal(idx[0], [0, 1, 2])
    np.testing.assert_allclose(gate[0], [1 / 3] * 3, rtol=1e-15)
    L = np.array([[1.0, 5.0, 5.0, 2.0, 5.0]])
    idx, _ = orc.topk(L, 2)
    np.testing.assert_array_equal(idx[0], [1, 2])


def test_gates_full_softmax_when_k_equals_e(orc):
    rng = np.random.default_rng(2)
    L = rng.standard_normal((5, 8)) * 3
    idx, gate = orc.topk(L, 8)
    for t in range(5):
        np.testing.assert_allclose(gate[t], softmax(L[t])[idx[t]], rtol=1e-13)


def test_gates_renormalised_softmax(orc):
    # gate_i = p_i / sum_sel p_j with p the full softmax over all E
    rng = np.random.default_rng(4)
    L = rng.standard_normal((6, 16)) * 2
    idx, gate = orc.topk(L, 4)
    for t in range(6):
        p = softmax(L[t])
        np.testing.assert_allclose(gate[t], p[idx[t]] / p[idx[t]].sum(), rtol=1e-13)
        assert np.all(np.diff(gate[t]) <= 0)      # slots in descending order


# ---------------------------------------------------------------------------
# permute
# ---------------------------------------------------------------------------
def test_permute_matches_stable_argsort(orc):
    rng = np.random.default_rng(1)
    for T, k, E in [(16, 2, 8), (8, 8, 256), (256, 8, 256), (3, 1, 4)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        counts, offsets, sorted_ = orc.permute(idx, E)
        np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
        np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        np.testing.assert_array_equal(sorted_, np.argsort(idx.ravel(), kind="stable"))
        assert counts.sum() == T * k
        assert np.array_equal(np.sort(sorted_), np.arange(T * k))


# ---------------------------------------------------------------------------
# SiLU and the MoE layer
# ---------------------------------------------------------------------------
def test_silu_special_values(orc):
    assert orc.silu(0.0) == 0.0
    assert orc.silu(1.0) == pytest.approx(0.7310585786300049, rel=1e-15)  # 1/(1+e^-1)
    assert orc.silu(-1.0) == pytest.approx(-0.2689414213699951, rel=1e-15)
    assert orc.silu(50.0) == pytest.approx(50.0, rel=1e-20)
    v = orc.silu(-1000.0)   # exp overflows to +inf: result -0, never NaN
    assert v == 0.0 and np.signbit(v)


def _dense_masked_moe(orc, fmt, E, k, H, F, n_shared, w, x_f64):
    """Every expert on every token, then masked to the selection (numpy)."""
    qk, nb = orc.geometry(fmt)
    T = x_f64.shape[0]
    L = x_f64 @ w["router_W"].astype(np.float64).T
    p = np.exp(L - L.max(axis=1, keepdims=True))
    y = np.zeros((T, H))
    mask = np.zeros((T, E))
    for t in range(T):
        sel = np.lexsort((np.arange(E), -L[t]))[:k]
        mask[t, sel] = p[t, sel] / p[t, sel].sum()

    def mat(raw, i, rows, cols):
        n = rows * (cols // qk) * nb
        return orc.dequant(fmt, raw[i * n:(i + 1) * n], rows * cols).astype(np.float64).reshape(rows, cols)

    def ffn(Wg, Wu, Wd):
        gg = x_f64 @ Wg.T
        uu = x_f64 @ Wu.T
        return ((gg / (1.0 + np.exp(-gg))) * uu) @ Wd.T

    for e in range(E):
        y += mask[:, e:e + 1] * ffn(mat(w["w_gate"], e, F, H), mat(w["w_up"], e, F, H),
                                    mat(w["w_down"], e, H, F))
    for s in range(n_shared):
        y += ffn(mat(w["sh_gate"], s, F, H), mat(w["sh_up"], s, F, H), mat(w["sh_down"], s, H, F))
    return y


@pytest.mark.parametrize("fmt,E,k,H,F,n_shared,T,xdt", [
    (Q4_K, 8, 2, 256, 512, 0, 5, 1),
    (Q4_K, 6, 3, 512, 256, 1, 4, 2),
    (Q8_0, 4, 4, 64, 96, 0, 3, 0),
    (Q6_K, 3, 1, 256, 256, 2, 2, 1),
    (Q4_K, 1, 1, 256, 256, 0, 2, 0),
])
def test_moe_equals_dense_masked(orc, fmt, E, k, H, F, n_shared, T, xdt):
    g = synth.streams(1000 + E * 10 + k, 2)
    w = synth.moe_weights(2000 + E, E, H, F, n_shared, fmt)
    x = synth.activations(g[0], (T, H), xdt)
    y, idx, gate, logits = orc.moe_forward(fmt, E, k, H, F, n_shared, w["router_W"], w["w_gate"],
                                           w["w_up"], w["w_down"], w["sh_gate"], w["sh_up"],
                                           w["sh_down"], x, xdt, T)
    ref = _dense_masked_moe(orc, fmt, E, k, H, F, n_shared, w, orc.act_to_f64(xdt, x).reshape(T, H))
    scale = np.abs(ref).max()
    assert scale > 0
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-6 * scale)
    np.testing.assert_allclose(gate.sum(axis=1), 1.0, atol=1e-12)
    # token subset returns the same rows
    sub = np.array([T - 1, 0], dtype=np.int32)
    ys, *_ = orc.moe_forward(fmt, E, k, H, F, n_shared, w["router_W"], w["w_gate"], w["w_up"],
                             w["w_down"], w["sh_gate"], w["sh_up"], w["sh_down"], x, xdt, T,
                             tokens=sub)
    np.testing.assert_array_equal(ys, y[sub])


def test_moe_single_expert_is_plain_ffn(orc):
    # E = k = 1: gate is 1 and the layer is the expert's SwiGLU FFN
    fmt, H, F = Q4_K, 256, 512
    w = synth.moe_weights(77, 1, H, F, 0, fmt)
    x = synth.activations(synth.streams(78, 1)[0], (1, H), 1)
    y, idx, gate, _ = orc.moe_forward(fmt, 1, 1, H, F, 0, w["router_W"], w["w_gate"], w["w_up"],
                                      w["w_down"], None, None, None, x, 1, 1)
    assert idx[0, 0] == 0 and gate[0, 0] == 1.0
    o = orc.expert_ffn(fmt, w["w_gate"], w["w_up"], w["w_down"], H, F,
                       orc.act_to_f64(1, x).ravel())
    np.testing.assert_array_equal(y[0], o.astype(np.float32))


def test_ref_under_selection_reproduces_the_layer(orc):
    # the parity tests' reference for a near-tie token (the oracle's expert
    # FFNs and gates under a given selection) equals the oracle's layer when
    # given the oracle's own selection, and differs under another one
    from moe_layers import ref_under_selection
    E, k, H, F, ns, T, fmt, xdt = 8, 2, 256, 512, 1, 4, 1, 1
    w = synth.moe_weights(4100, E, H, F, ns, fmt)
    x = synth.activations(synth.streams(4101, 1)[0], (T, H), xdt)
    y, idx, gate, L = orc.moe_forward(fmt, E, k, H, F, ns, w["router_W"], w["w_gate"], w["w_up"],
                                      w["w_down"], w["sh_gate"], w["sh_up"], w["sh_down"], x, xdt, T)
    for t in range(T):
        r = ref_under_selection(orc, fmt, w, E, k, H, F, ns, x, xdt, t, idx[t], L)
        np.testing.assert_allclose(r, y[t], rtol=1e-6, atol=1e-6 * np.abs(y[t]).max())
        other = np.array([e for e in range(E) if e not in idx[t]][:k])
        r2 = ref_under_selection(orc, fmt, w, E, k, H, F, ns, x, xdt, t, other, L)
        assert np.abs(r2 - y[t]).max() > 1e-3 * np.abs(y[t]).max()
