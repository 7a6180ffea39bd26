// qgemv_mma.cuh — the streaming quantized GEMV core for 16-bit-operand
// tensor-core products, shared by dq_qgemv and the grouped MoE kernels.
//
// What it computes: for a 64-row tile of a quantized matrix W (N x K, blocks
// of dqmoe.h) and up to 8 activation columns, acc[row][col] = sum_k W x, fp32
// accumulate — the decode linear of [NTransformer, §核心性能] and the expert
// projections of [Titan Engine, §MoE 专家流式加载].
//
// How (sm_103a):
//   * warp 0 is the loader.  Per pipeline stage it issues one 1-D bulk copy
//     (TMA engine, L2 evict-first) per weight row of C super-blocks into a
//     padded shared-memory row, and converts the activation chunk of the stage
//     into fp16 (with a per-column power-of-two scale for bf16/fp32 inputs, so
//     no value overflows fp16), writing it in a bank-skewed layout.
//   * warps 1..4 are consumers, 16 rows each.  Lane (g = lane/4, t = lane%4)
//     owns 64 weights of every super-block of rows g and g+8: it decodes them
//     in registers to fp16 (exact integer unpack, then one fused scale/min per
//     pair; Q4_K in per-row power-of-two units) straight into the A fragment of
//     mma.m16n8k16 (rows = weights, k = 16 weights, n = 8 activation columns).
//     Scales are folded into A, so the k order inside an mma is free; the
//     activation B fragment is read in natural k order.
//   * fp32 accumulators per stage are scaled by the column's inverse scale and
//     summed into the running accumulator.
//   * stages flow through full/empty mbarriers with bounded waits.
// Arithmetic per weight: ~1.3 integer/half2 instructions (Q4_K); the tensor
// core does the multiply-accumulate.
#pragma once

#include "common.cuh"

namespace dqmoe {

constexpr int kConsumerWarps = 4;
constexpr int kTileRows = 16 * kConsumerWarps;   // 64
constexpr int kThreads = 32 * (kConsumerWarps + 1);

// fp16 element offset of activation k inside a stage column: 8 halves (16 B)
// of padding after every 64 so that the 4 lanes of a quad, which read 64
// elements apart, hit distinct banks; 8-element runs stay 16-byte aligned.
__host__ __device__ constexpr int xoff(int k) { return k + 8 * (k >> 6); }

template <int FMT>
struct Layout {
  static constexpr int SBB = Fmt<FMT>::SB_BYTES;
  // one super-block (256 weights) per row per pipeline stage
  static constexpr int C = 1;
  // bytes of a row's TMA box per stage: the super-block, for Q6_K / Q2_K /
  // Q3_K a 16-byte aligned superset of its 210 / 84 / 110 bytes (starts up to
  // 14 / 12 / 14 bytes early)
  static constexpr int BOX = (FMT == DQ_Q4_K || FMT == DQ_Q4_0 || FMT == DQ_NVFP4) ? 144
                             : (FMT == DQ_Q6_K)                   ? 240
                             : (FMT == DQ_Q5_K)                   ? 176
                             : (FMT == DQ_Q2_K)                   ? 112
                             : (FMT == DQ_Q3_K)                   ? 144
                                                                  : 272;
  // TMA writes box rows densely: pitch = BOX; BOX/16 is odd for every format,
  // so rows g and g+1 fall on different bank halves for 16-byte reads
  static constexpr int ROW_PITCH = BOX;
  static constexpr int W_STAGE = kTileRows * ROW_PITCH;
  // activation column pitch: 32 (mod 128) bytes
  static constexpr int XCOL_RAW = xoff(C * 256) * 2;
  static constexpr int XCOL = XCOL_RAW + ((32 - XCOL_RAW % 128) + 128) % 128;
};

// Per-stage column-scale slots: 8 per 8 activation columns.
__host__ __device__ constexpr int xinv_stride(int cols) { return 8 * ((cols + 7) / 8); }

// Dynamic shared memory layout of one CTA (offsets in bytes).
struct SmemPlan {
  int nstage, batch, ksplit;
  int off_bar, off_w, off_x, off_xinv, off_red, total;
};

template <int FMT>
__host__ __device__ inline SmemPlan make_plan(int nstage, int batch, int ksplit) {
  SmemPlan p;
  p.nstage = nstage;
  p.batch = batch;
  p.ksplit = ksplit;
  p.off_bar = 0;                                       // full[ns], empty[ns], red
  p.off_w = 1024;                                      // 128-byte aligned TMA stages
  p.off_x = p.off_w + nstage * Layout<FMT>::W_STAGE;
  p.off_xinv = p.off_x + nstage * batch * Layout<FMT>::XCOL;
  p.off_red = p.off_xinv + nstage * xinv_stride(batch) * 4;
  p.off_red = (p.off_red + 15) / 16 * 16;
  p.total = p.off_red + (ksplit > 1 ? (ksplit - 1) * kConsumerWarps * 32 * 16 : 0);
  return p;
}

// ---------------------------------------------------------------------------
// Activation sources: the loader converts a column chunk of 8 values.
// ---------------------------------------------------------------------------
struct XSrc {
  const void* base;   // element 0 of row 0
  int dtype;          // DQ_F16 / DQ_BF16 / DQ_F32
  int64_t col_stride; // elements between rows
  const int* rows;    // column c reads row rows[c] (gather); nullptr: row c
};

__device__ __forceinline__ int64_t xrow(const XSrc& xs, int c) {
  return xs.rows ? (int64_t)__ldg(xs.rows + c) : (int64_t)c;
}

__device__ __forceinline__ void load8_f32(const XSrc& xs, int col, int64_t k, float (&v)[8]) {
  if (xs.dtype == DQ_F32) {
    const float4* p = (const float4*)((const float*)xs.base + xrow(xs, col) * xs.col_stride + k);
    const float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = __ldg((const uint4*)((const uint16_t*)xs.base + xrow(xs, col) * xs.col_stride + k));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    if (xs.dtype == DQ_BF16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(u32_as_h2(w[i]));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
    }
  }
}

// scale = 2^(14 - e) where max|x| in [2^e, 2^(e+1)): scaled values < 2^15.
__device__ __forceinline__ void pow2_scale(float amax, float& scale, float& inv) {
  const uint32_t bits = __float_as_uint(amax);
  int e = (int)((bits >> 23) & 255) - 127;
  if (amax == 0.f || e == 128) {   // zero column (or non-finite: out of contract)
    scale = 1.f;
    inv = 1.f;
    return;
  }
  if (e < -126) e = -126;
  int se = 14 - e;                 // in [-113, 140]
  if (se > 126) se = 126;          // keep both 2^se and 2^-se normal
  scale = __uint_as_float((uint32_t)(127 + se) << 23);
  inv = __uint_as_float((uint32_t)(127 - se) << 23);
}

// Arrivals per phase of a stage's full barrier: the loader's lane 0 with the
// TMA byte count, one cp.async arrival per loader lane, and for converted
// (bf16 / fp32) activations one more arrival per lane after its stores.
__host__ __device__ constexpr int full_arrivals(int dtype) { return dtype == DQ_F16 ? 33 : 65; }

// fp16 activations need no scale: every stage's column scale is 1.
__device__ __forceinline__ void init_xinv(float* xinv, int n, int dtype) {
  if (dtype == DQ_F16)
    for (int i = threadIdx.x; i < n; i += blockDim.x) xinv[i] = 1.f;
}

// Loader: stage the activation columns of one stage (nsb_stage super-blocks
// starting at activation index k0) as fp16 at xdst (column pitch XCOL bytes)
// and arrive on `full` for this lane: asynchronously once its cp.async copies
// of the stage have landed, and (bf16 / fp32 input only) once more after its
// own shared-memory stores.  fp16 input is copied asynchronously; bf16 / fp32
// input is converted with a per-column power-of-two scale.  The full barrier
// therefore expects full_arrivals(dtype) arrivals per phase.
template <int FMT>
__device__ __forceinline__ void stage_x(const XSrc& xs, int ncols, int64_t k0, int nsb_stage,
                                        uint8_t* xdst, float* xinv, int lane, uint64_t* full) {
  if (xs.dtype == DQ_F16) {
    for (int c = 0; c < ncols; ++c) {
      uint8_t* col = xdst + c * Layout<FMT>::XCOL;
      const uint16_t* src = (const uint16_t*)xs.base + xrow(xs, c) * xs.col_stride + k0;
      for (int j = 0; j < nsb_stage; ++j) {
        const int k = j * 256 + 8 * lane;
        cp_async16(col + 2 * xoff(k), src + k);
      }
    }
    // xinv stays 1 for fp16 input: set once per CTA before the pipeline starts
    cp_async_arrive_noinc(full);
    return;
  }
  // four columns at a time: their global loads are all issued before any
  // value is used (a use inside the same branch as its load would wait for
  // each load in turn)
  static_assert(Layout<FMT>::C == 1, "one super-block per stage");
  for (int c0 = 0; c0 < ncols; c0 += 4) {
    float v[4][8];
    float amax[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (c0 + j < ncols && nsb_stage > 0) load8_f32(xs, c0 + j, k0 + 8 * lane, v[j]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax[j] = 0.f;
      if (c0 + j < ncols && nsb_stage > 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) amax[j] = fmaxf(amax[j], fabsf(v[j][i]));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int j = 0; j < 4; ++j) amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], o));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (c0 + j < ncols && nsb_stage > 0) {
        float sc, inv;
        pow2_scale(amax[j], sc, inv);
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          h[i] = h2_as_u32(__floats2half2_rn(v[j][2 * i] * sc, v[j][2 * i + 1] * sc));
        *(uint4*)(xdst + (c0 + j) * Layout<FMT>::XCOL + 2 * xoff(8 * lane)) =
            make_uint4(h[0], h[1], h[2], h[3]);
        if (lane == 0) xinv[c0 + j] = inv;
      }
    }
  }
  cp_async_arrive_noinc(full);
  mbar_arrive(full);
}

// ---------------------------------------------------------------------------
// Consumer: one super-block of 16 rows (rows g, g+8 of lane) x 256 weights.
// wrow: shared address of row g's super-block; pitch: bytes to row g+8.
// xcol: shared address of this lane's activation column, at the stage start
// (column 0 for lanes past the batch);
// kb: k offset of the super-block inside the stage (j*256).
// ---------------------------------------------------------------------------
// The decode cores below read shared memory with plain (schedulable) loads:
// callers pass addresses derived from order_after_wait() of the stage's full
// barrier and pass the accumulators through keep_before_release() before the
// stage is released.
//
// B fragment (k, k+1 | k+2, k+3) of this lane's activation column.  Lanes
// whose column is past the batch read column 0: their output column is never
// stored, and an mma output column depends only on its own B column.
__device__ __forceinline__ void ldx(uint32_t xcol, int k, uint32_t& b0, uint32_t& b1) {
  const uint2 v = lds_u64_nv(xcol + 2 * xoff(k));
  b0 = v.x;
  b1 = v.y;
}

// One A fragment times NT activation tiles of 8 columns: NT mma into the
// accumulator chain `ch` of each tile.
template <int NT>
__device__ __forceinline__ void mma_x(float (&acc)[NT][2][4], int ch, uint32_t a0, uint32_t a1,
                                      uint32_t a2, uint32_t a3, const uint32_t (&xcol)[NT],
                                      int k) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    uint32_t b0, b1;
    ldx(xcol[nt], k, b0, b1);
    mma_16816_nv(acc[nt][ch], a0, a1, a2, a3, b0, b1);
  }
}

template <int FMT>
struct SBDot;

// acc += (D0 + D1) * row scale * column scale for one 8-column tile: D0, D1
// are the two accumulator chains of a super-block in row-scaled units (r0 for
// row g, r8 for row g+8); c0, c1 undo the activation scale of columns 2t, 2t+1.
__device__ __forceinline__ void fold_tile(float (&acc)[4], const float (&d)[2][4], float r0,
                                          float r8, float c0, float c1) {
  acc[0] = fmaf(d[0][0] + d[1][0], r0 * c0, acc[0]);
  acc[1] = fmaf(d[0][1] + d[1][1], r0 * c1, acc[1]);
  acc[2] = fmaf(d[0][2] + d[1][2], r8 * c0, acc[2]);
  acc[3] = fmaf(d[0][3] + d[1][3], r8 * c1, acc[3]);
}

// Q4_K: lane t owns qs group t (bytes 32t..32t+31): sub-blocks 2t (low
// nibbles) and 2t+1 (high nibbles), weights 64t + [0,64).
//
// Decode: a masked nibble pair, read as two fp16 bit patterns, is the exact
// subnormal pair (q * 2^-24); one fp16 FMA then gives q * S + O with
// S = sc * d * F and O = -m * dmin * F * 2^-24, F = 2^(24 - e) for e the larger
// exponent field of d and dmin.  The A operand is therefore the weight times
// the power of two 2^-e, normal and within fp16 range for any d, dmin, and the
// fp32 result of the super-block is multiplied back by 2^e (rinv).  One integer
// AND and one FMA per weight pair, no magic-number subtraction.
template <>
struct SBDot<DQ_Q4_K> {
  static constexpr bool kRowScale = true;

  __device__ __forceinline__ static void scales(uint4 hd, int t, __half2& slo, __half2& olo,
                                                __half2& shi, __half2& ohi, float& rinv) {
    const int jj = 2 * (t & 1);
    const uint32_t sel = (uint32_t)jj | (4u << 4) | ((uint32_t)(jj + 1) << 8) | (4u << 12);
    const uint32_t hy = __byte_perm(hd.y, 0, sel);
    const uint32_t hz = __byte_perm(hd.z, 0, sel);
    const uint32_t hw = __byte_perm(hd.w, 0, sel);
    uint32_t sc, mn;
    if (t < 2) {
      sc = hy & 0x003F003Fu;
      mn = hz & 0x003F003Fu;
    } else {
      sc = (hw & 0x000F000Fu) | ((hy >> 2) & 0x00300030u);
      mn = ((hw >> 4) & 0x000F000Fu) | ((hz >> 2) & 0x00300030u);
    }
    const __half2 magic = u32_as_h2(0x64006400u);
    const __half2 sch = __hsub2(u32_as_h2(sc | 0x64006400u), magic);   // exact ints
    const float2 mnf = __half22float2(__hsub2(u32_as_h2(mn | 0x64006400u), magic));
    // e: larger biased exponent field of d and dmin (0 when both are
    // subnormal or zero: then F = 2^24 maps d = k * 2^-24 to the integer k)
    const uint32_t e = max(hd.x & 0x7C00u, (hd.x >> 16) & 0x7C00u) >> 10;
    const float F = __uint_as_float((151u - e) << 23);     // 2^(24 - e)
    const float Fm = __uint_as_float((127u - e) << 23);    // 2^-e = F * 2^-24
    rinv = __uint_as_float((127u + e) << 23);              // 2^e
    // d * F < 1024: exact in fp16; sc * d * F <= 63 * 1023.5 < 65504
    const float df = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFF))) * F;
    const float dm = -__half2float(__ushort_as_half((unsigned short)(hd.x >> 16))) * Fm;
    const __half2 s = __hmul2(__float2half2_rn(df), sch);   // (S_lo, S_hi)
    const __half2 o = __floats2half2_rn(mnf.x * dm, mnf.y * dm);
    slo = __low2half2(s);
    olo = __low2half2(o);
    shi = __hmul2(__high2half2(s), __float2half2_rn(0.0625f));   // high nibbles carry x16
    ohi = __high2half2(o);
  }

  // Absolute scales for decoding real fp16 weights (the tensor-core prefill
  // tiles, whose K runs across super-blocks): (d*sc, -dmin*m) of sub-blocks
  // 2t (lo) and 2t+1 (hi, with the x16 of high nibbles folded in).
  __device__ __forceinline__ static void scales_abs(uint4 hd, int t, __half2& slo, __half2& olo,
                                                    __half2& shi, __half2& ohi) {
    const int jj = 2 * (t & 1);
    const uint32_t sel = (uint32_t)jj | (4u << 4) | ((uint32_t)(jj + 1) << 8) | (4u << 12);
    const uint32_t hy = __byte_perm(hd.y, 0, sel);
    const uint32_t hz = __byte_perm(hd.z, 0, sel);
    const uint32_t hw = __byte_perm(hd.w, 0, sel);
    uint32_t sc, mn;
    if (t < 2) {
      sc = hy & 0x003F003Fu;
      mn = hz & 0x003F003Fu;
    } else {
      sc = (hw & 0x000F000Fu) | ((hy >> 2) & 0x00300030u);
      mn = ((hw >> 4) & 0x000F000Fu) | ((hz >> 2) & 0x00300030u);
    }
    const __half2 magic = u32_as_h2(0x64006400u);
    const __half2 sch = __hsub2(u32_as_h2(sc | 0x64006400u), magic);
    const __half2 mnh = __hsub2(u32_as_h2(mn | 0x64006400u), magic);
    const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)(hd.x & 0xFFFF)));
    const __half2 dm2 = __half2half2(__hneg(__ushort_as_half((unsigned short)(hd.x >> 16))));
    const __half2 s = __hmul2(d2, sch);
    const __half2 o = __hmul2(dm2, mnh);
    slo = __low2half2(s);
    olo = __low2half2(o);
    shi = __hmul2(__high2half2(s), __float2half2_rn(0.0625f));
    ohi = __high2half2(o);
  }

  // A fragments of one step: words w0 (row g) and w8 (row g+8) hold bytes
  // b0..b3 = weights 4s..4s+3 of sub-block 2t (low nibbles) and 2t+1 (high).
  // lo / hi: the fragments of the low / high nibbles, weights in k order.
  // s*h is the high sub-block's S/16 (the scale of 16*q).
  __device__ __forceinline__ static void frags(uint32_t w0, uint32_t w8, __half2 s0l, __half2 o0l,
                                               __half2 s0h, __half2 o0h, __half2 s8l,
                                               __half2 o8l, __half2 s8h, __half2 o8h,
                                               uint32_t (&lo)[4], uint32_t (&hi)[4]) {
    // whole bytes in 16-bit lanes: (b0, b1) and (b2, b3), each the exact
    // subnormal (lo + 16 hi) * 2^-24.  The low term is one AND and one HFMA2;
    // the high term s_h * (b - lo) + o_h takes two HFMA2 and no mask, which
    // moves work from the integer pipe (the busier one) to the fp16 pipe.
    const uint32_t r0 = __byte_perm(w0, 0, 0x4140), r0s = __byte_perm(w0, 0, 0x4342);
    const uint32_t r8 = __byte_perm(w8, 0, 0x4140), r8s = __byte_perm(w8, 0, 0x4342);
    const uint32_t l0 = r0 & 0x000F000Fu, l0s = r0s & 0x000F000Fu;
    const uint32_t l8 = r8 & 0x000F000Fu, l8s = r8s & 0x000F000Fu;
    lo[0] = h2_as_u32(__hfma2(u32_as_h2(l0), s0l, o0l));
    lo[1] = h2_as_u32(__hfma2(u32_as_h2(l8), s8l, o8l));
    lo[2] = h2_as_u32(__hfma2(u32_as_h2(l0s), s0l, o0l));
    lo[3] = h2_as_u32(__hfma2(u32_as_h2(l8s), s8l, o8l));
    const __half2 n0h = __hneg2(s0h), n8h = __hneg2(s8h);
    hi[0] = h2_as_u32(__hfma2(u32_as_h2(r0), s0h, __hfma2(u32_as_h2(l0), n0h, o0h)));
    hi[1] = h2_as_u32(__hfma2(u32_as_h2(r8), s8h, __hfma2(u32_as_h2(l8), n8h, o8h)));
    hi[2] = h2_as_u32(__hfma2(u32_as_h2(r0s), s0h, __hfma2(u32_as_h2(l0s), n0h, o0h)));
    hi[3] = h2_as_u32(__hfma2(u32_as_h2(r8s), s8h, __hfma2(u32_as_h2(l8s), n8h, o8h)));
  }

  // acc: this super-block's products in units of 2^-e per row (rows g and
  // g+8: r0, r8 = 2^e of each row's super-block).  PAIRX: fetch the B
  // fragments of two consecutive steps with one 16-byte load (faster in the
  // grouped kernel, slower in the single-matrix one, measured on GB300).
  template <int NT, bool PAIRX = false>
  __device__ __forceinline__ static void run(uint32_t wrow, int pitch8,
                                             const uint32_t (&xcol)[NT], int kb, int t,
                                             float (&acc)[NT][2][4], float& r0, float& r8) {
    const uint32_t ra = wrow, rb = wrow + pitch8;
    const uint4 h0 = lds_u128_nv(ra), h8 = lds_u128_nv(rb);
    __half2 s0l, o0l, s0h, o0h, s8l, o8l, s8h, o8h;
    scales(h0, t, s0l, o0l, s0h, o0h, r0);
    scales(h8, t, s8l, o8l, s8h, o8h, r8);
    const uint32_t qa = ra + 16 + 32 * t;      // this lane's 32 quant bytes of row g
    const uint4 qa0 = lds_u128_nv(qa), qb0 = lds_u128_nv(qa + 16);
    const uint4 qa8 = lds_u128_nv(qa + pitch8), qb8 = lds_u128_nv(qa + pitch8 + 16);
    const uint32_t q0[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qb0.x, qb0.y, qb0.z, qb0.w};
    const uint32_t q8[8] = {qa8.x, qa8.y, qa8.z, qa8.w, qb8.x, qb8.y, qb8.z, qb8.w};
    if constexpr (PAIRX) {
      // activation kb + 64t + c (c < 64) of a tile sits at xb + 2c: the B
      // fragments of two consecutive steps come from one 16-byte load
      uint32_t xb[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) xb[nt] = xcol[nt] + 2 * xoff(kb + 64 * t);
#pragma unroll
      for (int sp = 0; sp < 4; ++sp) {
        uint4 xl[NT], xh[NT];                      // steps 2sp, 2sp+1: low / high nibbles
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          xl[nt] = lds_u128_nv(xb[nt] + 16 * sp);
          xh[nt] = lds_u128_nv(xb[nt] + 16 * sp + 64);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int s = 2 * sp + h;
          uint32_t lo[4], hi[4];
          frags(q0[s], q8[s], s0l, o0l, s0h, o0h, s8l, o8l, s8h, o8h, lo, hi);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_16816_nv(acc[nt][0], lo[0], lo[1], lo[2], lo[3], h ? xl[nt].z : xl[nt].x,
                      h ? xl[nt].w : xl[nt].y);
            mma_16816_nv(acc[nt][1], hi[0], hi[1], hi[2], hi[3], h ? xh[nt].z : xh[nt].x,
                      h ? xh[nt].w : xh[nt].y);
          }
        }
      }
    } else {
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        // weights kb + 64t + 4s + 0..3 (low nibbles), 32 further (high)
        const int k = kb + 64 * t + 4 * s;
        uint32_t lo[4], hi[4];
        frags(q0[s], q8[s], s0l, o0l, s0h, o0h, s8l, o8l, s8h, o8h, lo, hi);
        mma_x<NT>(acc, 0, lo[0], lo[1], lo[2], lo[3], xcol, k);
        mma_x<NT>(acc, 1, hi[0], hi[1], hi[2], hi[3], xcol, k + 32);
      }
    }
  }
};

// Q6_K: lane t owns, in each half h, positions l in [8t, 8t+8) of the four
// 32-weight runs r = 0..3: weights 128h + 32r + l, scale index 8h + 2r + t/2.
// Blocks are 210 bytes, so every other block is only 2-byte aligned.
//
// Decode: q is assembled in place in each 16-bit lane (runs 0-1: the low
// nibble at bits 0-3 and the two qh bits at 4-5, value q; runs 2-3: the high
// nibble at bits 4-7 and the qh bits at 8-9, value 16 q), read as the exact
// fp16 subnormal, and one HFMA2 with S = d sc F (runs 2-3: S / 16) and
// O = -32 d sc F 2^-24 gives (q - 32) d sc F 2^-24: the weight times the
// row's power of two F 2^-24 = 2^-(e+1), e the exponent field of d (undone in
// fp32 after the super-block).  d F < 512 and |sc| <= 128 keep |S| <= 65504.
template <>
struct SBDot<DQ_Q6_K> {
  static constexpr bool kRowScale = true;

  // (q - 32) of two weights as an exact fp16 pair, for decoders that produce
  // absolute weights (the tensor-core prefill slabs): nib holds 4-bit values
  // in bits 0-3 of each 16-bit lane, hq 2-bit values already in bits 4-5
  __device__ __forceinline__ static uint32_t q6_pair(uint32_t nib, uint32_t hq) {
    const uint32_t v = (nib & 0x000F000Fu) | (hq & 0x00300030u) | 0x64006400u;
    return h2_as_u32(__hsub2(u32_as_h2(v), u32_as_h2(0x64206420u)));   // 1024+q - 1056
  }

  // 32-bit word at a 2-byte aligned address whose misalignment (0 or 2
  // bytes, MIS) is uniform for the stage
  template <bool MIS>
  __device__ __forceinline__ static uint32_t ldw(uint32_t a) {
    if constexpr (MIS) return __funnelshift_r(lds_u32_nv(a - 2), lds_u32_nv(a + 2), 16);
    else return lds_u32_nv(a);
  }

  template <int NT, bool PAIRX = false>
  __device__ __forceinline__ static void run(uint32_t wrow, int pitch8,
                                             const uint32_t (&xcol)[NT], int kb, int t,
                                             float (&acc)[NT][2][4], float& r0, float& r8) {
    // the 210-byte super-blocks start 0 or 2 bytes off a word, the same for
    // every row of a stage: a uniform branch
    if (wrow & 2u) run_impl<NT, true>(wrow, pitch8, xcol, kb, t, acc, r0, r8);
    else run_impl<NT, false>(wrow, pitch8, xcol, kb, t, acc, r0, r8);
  }

  template <int NT, bool MIS>
  __device__ __forceinline__ static void run_impl(uint32_t wrow, int pitch8,
                                                  const uint32_t (&xcol)[NT], int kb, int t,
                                                  float (&acc)[NT][2][4], float& r0,
                                                  float& r8) {
    const uint32_t rows[2] = {wrow, wrow + pitch8};
    // this lane's 8 scales per row, sc[8h + 2r + t/2] (h = 0..1, r = 0..3), as
    // S and O pairs
    __half2 S[2][8], O[2][8];
    float rinv[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const uint32_t rb = rows[rr];
      const uint32_t dh = lds_u16_nv(rb + 208);
      const uint32_t e = (dh >> 10) & 31u;
      const float F = __uint_as_float((150u - e) << 23);   // 2^(23 - e)
      rinv[rr] = __uint_as_float((128u + e) << 23);        // 2^(e + 1)
      const float df = __half2float(__ushort_as_half((unsigned short)dh)) * F;   // exact
      const uint32_t s0 = ldw<MIS>(rb + 192), s1 = ldw<MIS>(rb + 196);
      const uint32_t s2 = ldw<MIS>(rb + 200), s3 = ldw<MIS>(rb + 204);
      const uint32_t sw[4] = {s0, s1, s2, s3};
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int idx = 8 * h + 2 * r;    // + t/2
          const uint32_t word = sw[idx >> 2];
          const int byte = (idx & 3) + (t >> 1);
          const int sc = (int)(int8_t)((word >> (8 * byte)) & 0xFF);
          // d F sc is exact in fp32 (11 + 8 bits); one rounding to fp16
          const __half2 sv = __float2half2_rn(df * (float)sc * ((r & 2) ? 0.0625f : 1.f));
          S[rr][4 * h + r] = sv;
          O[rr][4 * h + r] = __hmul2(sv, __float2half2_rn((r & 2) ? -0x1p-15f : -0x1p-19f));
        }
    }
    r0 = rinv[0];
    r8 = rinv[1];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        // per row: ql words of runs 0/2 (A) and 1/3 (B), the qh word (H), each
        // as bytes (b0 b2 | b1 b3) in 16-bit lanes; the weights k+2, k+3 of
        // each step come from the words shifted down by 8
        uint32_t Q[2][2][2], H2[2][2], H4[2][2];   // [row][hi pair][run&1], [row][hi pair]
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const uint32_t rb = rows[rr];
          const uint32_t A = __byte_perm(ldw<MIS>(rb + 64 * h + 8 * t + 4 * p), 0, 0x3120);
          const uint32_t B = __byte_perm(ldw<MIS>(rb + 64 * h + 32 + 8 * t + 4 * p), 0, 0x3120);
          const uint32_t H = __byte_perm(ldw<MIS>(rb + 128 + 32 * h + 8 * t + 4 * p), 0, 0x3120);
          Q[rr][0][0] = A;
          Q[rr][0][1] = B;
          Q[rr][1][0] = A >> 8;
          Q[rr][1][1] = B >> 8;
          H4[rr][0] = H << 4;
          H2[rr][0] = H << 2;
          H4[rr][1] = (H >> 8) << 4;
          H2[rr][1] = (H >> 8) << 2;
        }
        const int kbase = kb + 128 * h + 8 * t + 4 * p;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          // qh bits 2r..2r+1 land at 4-5 (runs 0-1) or 8-9 (runs 2-3) after a
          // left shift by 4 (r even) or 2 (r odd)
          const uint32_t qm = (r & 2) ? 0x00F000F0u : 0x000F000Fu;
          const uint32_t hm = (r & 2) ? 0x03000300u : 0x00300030u;
          uint32_t a[4];
#pragma unroll
          for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
              const uint32_t hq = (r & 1) ? H2[rr][hp] : H4[rr][hp];
              const uint32_t u = lop3_and_or(hq, hm, Q[rr][hp][r & 1] & qm);
              a[2 * hp + rr] =
                  h2_as_u32(__hfma2(u32_as_h2(u), S[rr][4 * h + r], O[rr][4 * h + r]));
            }
          mma_x<NT>(acc, r & 1, a[0], a[1], a[2], a[3], xcol, kbase + 32 * r);
        }
      }
    }
  }
};

// Q8_0: 8 blocks of 34 bytes per 256 weights; block s is step s; lane t owns
// quants 8t..8t+7 of each block.
template <>
struct SBDot<DQ_Q8_0> {
  static constexpr bool kRowScale = false;
  template <int NT>
  __device__ __forceinline__ static void run(uint32_t wrow, int pitch8,
                                             const uint32_t (&xcol)[NT], int kb, int t,
                                             float (&acc)[NT][2][4]) {
    const __half2 bias = __float2half2_rn(1152.f);   // 1024 + 128
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t a[2][4];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const uint32_t blk = wrow + (rr ? pitch8 : 0) + 34 * s;
        const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)lds_u16_nv(blk)));
        const uint32_t w0 = lds_u32_a2_nv(blk + 2 + 8 * t) ^ 0x80808080u;   // q + 128, unsigned
        const uint32_t w1 = lds_u32_a2_nv(blk + 6 + 8 * t) ^ 0x80808080u;
        const uint32_t ws[2] = {w0, w1};
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t lo = __byte_perm(ws[m], 0x64646464u, 0x4140);   // bytes 0,1
          const uint32_t hi = __byte_perm(ws[m], 0x64646464u, 0x4342);   // bytes 2,3
          a[m][rr] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(lo), bias), d2));
          a[m][2 + rr] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(hi), bias), d2));
        }
      }
      mma_x<NT>(acc, 0, a[0][0], a[0][1], a[0][2], a[0][3], xcol, kb + 32 * s + 8 * t);
      mma_x<NT>(acc, 1, a[1][0], a[1][1], a[1][2], a[1][3], xcol, kb + 32 * s + 8 * t + 4);
    }
  }
};

// Q5_K: Q4_K's scales and nibble layout plus a fifth bit per weight (qh[l]
// bit 2t for the low nibble of byte l of group t, bit 2t+1 for the high one).
// Lane t owns group t as in Q4_K; the fifth bits are merged into the masked
// nibbles before the same one-HFMA2 decode (q up to 31: still an exact fp16
// subnormal).
template <>
struct SBDot<DQ_Q5_K> {
  static constexpr bool kRowScale = true;

  template <int NT, bool PAIRX = false>
  __device__ __forceinline__ static void run(uint32_t wrow, int pitch8,
                                             const uint32_t (&xcol)[NT], int kb, int t,
                                             float (&acc)[NT][2][4], float& r0, float& r8) {
    const uint32_t ra = wrow, rb = wrow + pitch8;
    const uint4 h0 = lds_u128_nv(ra), h8 = lds_u128_nv(rb);
    __half2 s0l, o0l, s0h, o0h, s8l, o8l, s8h, o8h;
    SBDot<DQ_Q4_K>::scales(h0, t, s0l, o0l, s0h, o0h, r0);
    SBDot<DQ_Q4_K>::scales(h8, t, s8l, o8l, s8h, o8h, r8);
    const uint32_t qa = ra + 48 + 32 * t;      // this lane's 32 low-quant bytes of row g
    const uint4 qa0 = lds_u128_nv(qa), qb0 = lds_u128_nv(qa + 16);
    const uint4 qa8 = lds_u128_nv(qa + pitch8), qb8 = lds_u128_nv(qa + pitch8 + 16);
    const uint4 ea0 = lds_u128_nv(ra + 16), eb0 = lds_u128_nv(ra + 32);   // qh[0..31] of row g
    const uint4 ea8 = lds_u128_nv(rb + 16), eb8 = lds_u128_nv(rb + 32);
    const uint32_t q0[8] = {qa0.x, qa0.y, qa0.z, qa0.w, qb0.x, qb0.y, qb0.z, qb0.w};
    const uint32_t q8[8] = {qa8.x, qa8.y, qa8.z, qa8.w, qb8.x, qb8.y, qb8.z, qb8.w};
    const uint32_t e0[8] = {ea0.x, ea0.y, ea0.z, ea0.w, eb0.x, eb0.y, eb0.z, eb0.w};
    const uint32_t e8[8] = {ea8.x, ea8.y, ea8.z, ea8.w, eb8.x, eb8.y, eb8.z, eb8.w};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      // bytes (b0 b1 b2 b3) -> (b0 b2 b1 b3): 16-bit lanes hold weights k, k+1;
      // the qh bytes follow the same permutation, shifted so that bit 2t of
      // each byte is bit 0 of its lane and bit 2t+1 is bit 1
      const uint32_t p0 = __byte_perm(q0[s], 0, 0x3120), p8 = __byte_perm(q8[s], 0, 0x3120);
      const uint32_t f0 = __byte_perm(e0[s], 0, 0x3120) >> (2 * t);
      const uint32_t f8 = __byte_perm(e8[s], 0, 0x3120) >> (2 * t);
      const uint32_t pv[4] = {p0, p8, p0 >> 8, p8 >> 8};
      const uint32_t fv[4] = {f0, f8, f0 >> 8, f8 >> 8};
      const int k = kb + 64 * t + 4 * s;
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 sl = (i & 1) ? s8l : s0l, ol = (i & 1) ? o8l : o0l;
        const __half2 sh = (i & 1) ? s8h : s0h, oh = (i & 1) ? o8h : o0h;
        // q * 2^-24 with q = nibble | fifth bit << 4; high nibbles as 16 * q
        const uint32_t ql = (pv[i] & 0x000F000Fu) | ((fv[i] << 4) & 0x00100010u);
        const uint32_t qh = (pv[i] & 0x00F000F0u) | ((fv[i] << 7) & 0x01000100u);
        lo[i] = h2_as_u32(__hfma2(u32_as_h2(ql), sl, ol));
        hi[i] = h2_as_u32(__hfma2(u32_as_h2(qh), sh, oh));
      }
      mma_x<NT>(acc, 0, lo[0], lo[1], lo[2], lo[3], xcol, k);
      mma_x<NT>(acc, 1, hi[0], hi[1], hi[2], hi[3], xcol, k + 32);
    }
  }
};

// Q4_0: 8 blocks of 18 bytes per 256 weights; block s is step s.  Lane t owns
// quant bytes 4t..4t+3 of each block: weights 4t..4t+3 (low nibbles) and
// 16+4t..16+4t+3 (high nibbles).  Absolute fp16 weights (q - 8 exact by the
// 1024 magic, one multiply by d).
template <>
struct SBDot<DQ_Q4_0> {
  static constexpr bool kRowScale = false;
  template <int NT, bool PAIRX = false>
  __device__ __forceinline__ static void run(uint32_t wrow, int pitch8,
                                             const uint32_t (&xcol)[NT], int kb, int t,
                                             float (&acc)[NT][2][4]) {
    const __half2 bias = __float2half2_rn(1032.f);   // 1024 + 8
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const uint32_t blk = wrow + (rr ? pitch8 : 0) + 18 * s;
        const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)lds_u16_nv(blk)));
        const uint32_t p = __byte_perm(lds_u32_a2_nv(blk + 2 + 4 * t), 0, 0x3120);
        const uint32_t pv[2] = {p, p >> 8};
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t l = lop3_and_or(pv[m], 0x000F000Fu, 0x64006400u);
          const uint32_t h = lop3_and_or(pv[m] >> 4, 0x000F000Fu, 0x64006400u);
          lo[2 * m + rr] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(l), bias), d2));
          hi[2 * m + rr] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(h), bias), d2));
        }
      }
      mma_x<NT>(acc, 0, lo[0], lo[1], lo[2], lo[3], xcol, kb + 32 * s + 4 * t);
      mma_x<NT>(acc, 1, hi[0], hi[1], hi[2], hi[3], xcol, kb + 32 * s + 16 + 4 * t);
    }
  }
};

// Q2_K / Q3_K: lane t owns the 16 quant bytes 16t..16t+15 of qs, i.e. half
// hq = t/2 and positions l = 16(t&1) + [0, 16): weights 128hq + 32r + l of
// the four 2-bit fields r, one 16-weight sub-block (8hq + 2r + (t&1)) per r.
// Step i reads the lane's quant word w = (i + t) & 3 (bytes 4w..4w+3 of its
// 16): with row pitches of an odd number of 16-byte units the 32 lanes of
// each 4-byte load then fall on 32 distinct banks.  The k order inside an mma
// is free, so each step's B fragment is read at the activations of its word.
//
// Decode: field r of each byte is masked in place (value q 4^r), the bytes
// are spread to 16-bit lanes and read as exact fp16 subnormals q 4^r 2^-24,
// and one HFMA2 with S/4^r and O yields the weight times a power of two per
// row (undone in fp32 after the super-block, as Q4_K).

// B fragments of one step at byte offset `off` from the lane's base xb.
template <int NT>
__device__ __forceinline__ void mma_xb(float (&acc)[NT][2][4], int ch, uint32_t a0, uint32_t a1,
                                       uint32_t a2, uint32_t a3, const uint32_t (&xb)[NT],
                                       int off) {
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint2 b = lds_u64_nv(xb[nt] + off);
    mma_16816_nv(acc[nt][ch], a0, a1, a2, a3, b.x, b.y);
  }
}

// Byte offset of field r's activations from those of field 0 of a word: the
// word's positions sit below 32 inside their 64-activation group, so field r
// is 32r further on and crosses r/2 group paddings of 8 halves.
__device__ __forceinline__ constexpr int field_xoff(int r) { return 2 * (32 * r + 8 * (r >> 1)); }

template <>
struct SBDot<DQ_Q2_K> {
  static constexpr bool kRowScale = true;

  // S[r] = d sc F / 4^r and O[r] = -dmin m F 2^-24 of the lane's sub-block of
  // field r (as broadcast pairs), F = 2^(26 - e) for e the larger exponent
  // field of d and dmin: d F < 4096 and sc <= 15 keep S < 61440; rinv = 2^(e-2)
  // undoes F 2^-24.  S is rounded once to fp16, O once from fp32.
  __device__ __forceinline__ static void scales(uint32_t rb, int t, __half2 (&S)[4],
                                                __half2 (&O)[4], float& rinv) {
    const uint32_t dd = lds_u32_nv(rb + 80);   // d | dmin << 16
    const uint32_t w0 = lds_u32_nv(rb + 8 * (t >> 1)), w1 = lds_u32_nv(rb + 8 * (t >> 1) + 4);
    // scale bytes 8hq + 2r + (t&1): (r = 0, 1) from w0, (2, 3) from w1
    const uint32_t tt = (uint32_t)(t & 1);
    const uint32_t sel = tt | (4u << 4) | ((tt + 2u) << 8) | (4u << 12);
    const uint32_t p0 = __byte_perm(w0, 0, sel), p1 = __byte_perm(w1, 0, sel);
    const __half2 magic = u32_as_h2(0x64006400u);
    const __half2 sc01 = __hsub2(u32_as_h2(lop3_and_or(p0, 0x000F000Fu, 0x64006400u)), magic);
    const __half2 sc23 = __hsub2(u32_as_h2(lop3_and_or(p1, 0x000F000Fu, 0x64006400u)), magic);
    const float2 m01 =
        __half22float2(__hsub2(u32_as_h2(lop3_and_or(p0 >> 4, 0x000F000Fu, 0x64006400u)), magic));
    const float2 m23 =
        __half22float2(__hsub2(u32_as_h2(lop3_and_or(p1 >> 4, 0x000F000Fu, 0x64006400u)), magic));
    const uint32_t e = max(dd & 0x7C00u, (dd >> 16) & 0x7C00u) >> 10;
    const float F = __uint_as_float((153u - e) << 23);    // 2^(26 - e)
    const float Fm = __uint_as_float((129u - e) << 23);   // 2^(2 - e) = F 2^-24
    rinv = __uint_as_float((125u + e) << 23);             // 2^(e - 2)
    const float df = __half2float(__ushort_as_half((unsigned short)(dd & 0xFFFF))) * F;
    const float dm = -__half2float(__ushort_as_half((unsigned short)(dd >> 16))) * Fm;
    const __half2 s01 = __hmul2(sc01, __floats2half2_rn(df, df * 0.25f));
    const __half2 s23 = __hmul2(sc23, __floats2half2_rn(df * 0.0625f, df * 0.015625f));
    const __half2 o01 = __floats2half2_rn(m01.x * dm, m01.y * dm);
    const __half2 o23 = __floats2half2_rn(m23.x * dm, m23.y * dm);
    S[0] = __low2half2(s01);
    S[1] = __high2half2(s01);
    S[2] = __low2half2(s23);
    S[3] = __high2half2(s23);
    O[0] = __low2half2(o01);
    O[1] = __high2half2(o01);
    O[2] = __low2half2(o23);
    O[3] = __high2half2(o23);
  }

  template <int NT, bool PAIRX = false>
  __device__ __forceinline__ static void run(uint32_t wrow, int pitch8,
                                             const uint32_t (&xcol)[NT], int kb, int t,
                                             float (&acc)[NT][2][4], float& r0, float& r8) {
    __half2 S0[4], O0[4], S8[4], O8[4];
    scales(wrow, t, S0, O0, r0);
    scales(wrow + pitch8, t, S8, O8, r8);
    const int kl = kb + 128 * (t >> 1) + 16 * (t & 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int w = (i + t) & 3;
      const uint32_t qa = wrow + 16 + 16 * t + 4 * w;
      const uint32_t q0 = lds_u32_nv(qa), q8 = lds_u32_nv(qa + pitch8);
      // bytes (0, 1) and (2, 3) of each word in 16-bit lanes: weights (k, k+1), (k+2, k+3)
      const uint32_t l0 = __byte_perm(q0, 0, 0x4140), h0 = __byte_perm(q0, 0, 0x4342);
      const uint32_t l8 = __byte_perm(q8, 0, 0x4140), h8 = __byte_perm(q8, 0, 0x4342);
      uint32_t xb[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) xb[nt] = xcol[nt] + 2 * xoff(kl + 4 * w);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t m = 0x00030003u << (2 * r);
        const uint32_t a0 = h2_as_u32(__hfma2(u32_as_h2(l0 & m), S0[r], O0[r]));
        const uint32_t a1 = h2_as_u32(__hfma2(u32_as_h2(l8 & m), S8[r], O8[r]));
        const uint32_t a2 = h2_as_u32(__hfma2(u32_as_h2(h0 & m), S0[r], O0[r]));
        const uint32_t a3 = h2_as_u32(__hfma2(u32_as_h2(h8 & m), S8[r], O8[r]));
        mma_xb<NT>(acc, r & 1, a0, a1, a2, a3, xb, field_xoff(r));
      }
    }
  }
};

// Q3_K: Q2_K's quant placement plus the high bit of each weight from hmask[l]
// (bit 4hq + r) and one signed 6-bit scale per sub-block.  With u = low + 4 *
// high = q + 4 in 0..7, w = d (s - 32) (u - 4).  Per word and field the bytes
// are assembled as u 2^b_r (b_r = 0, 2, 4, 5: the field's own position, and
// for r = 3 one lower so that the high bit still fits the byte), then spread
// and decoded as Q2_K's with S/2^b_r and O = -4 S 2^-24.  Blocks are 110
// bytes, so every other one starts 2 bytes off a 4-byte boundary: each word
// is then read as two aligned words and a funnel shift (MIS2).
template <>
struct SBDot<DQ_Q3_K> {
  static constexpr bool kRowScale = true;

  template <bool MIS2>
  __device__ __forceinline__ static uint32_t ld(uint32_t a) {
    if constexpr (MIS2) return __funnelshift_r(lds_u32_nv(a - 2), lds_u32_nv(a + 2), 16);
    else return lds_u32_nv(a);
  }

  // S[r] = d F (s - 32) / 2^b_r, O[r] = -4 d F (s - 32) 2^-24 of the lane's
  // sub-block of field r, F = 2^(25 - e) for e the exponent field of d:
  // d F < 2048 and |s - 32| <= 32 keep |S| <= 65504; rinv = 2^(e - 1).
  template <bool MIS2>
  __device__ __forceinline__ static void scales(uint32_t rb, int t, __half2 (&S)[4],
                                                __half2 (&O)[4], float& rinv) {
    const uint32_t dh = lds_u16_nv(rb + 108);
    const uint32_t s0 = ld<MIS2>(rb + 96), s1 = ld<MIS2>(rb + 100), s2 = ld<MIS2>(rb + 104);
    const uint32_t tt = (uint32_t)(t & 1), sh = 4u * (uint32_t)(t >> 1);
    const uint32_t sel = tt | (4u << 4) | ((tt + 2u) << 8) | (4u << 12);
    // sub-block j = 8hq + 2r + tt: low four bits = nibble hq of scale byte
    // 2r + tt (r = 0, 1 in s0, 2, 3 in s1); high two = field 2hq + r/2 of
    // byte 8 + tt (r even) or 10 + tt (r odd), bytes tt, tt + 2 of s2
    const uint32_t lo01 = __byte_perm(s0, 0, sel) >> sh, lo23 = __byte_perm(s1, 0, sel) >> sh;
    const uint32_t hb = __byte_perm(s2, 0, sel) >> sh;
    const uint32_t v01 =
        lop3_and_or(hb << 4, 0x00300030u, lop3_and_or(lo01, 0x000F000Fu, 0x64006400u));
    const uint32_t v23 =
        lop3_and_or(hb << 2, 0x00300030u, lop3_and_or(lo23, 0x000F000Fu, 0x64006400u));
    const __half2 bias = u32_as_h2(0x64206420u);   // 1024 + 32: s - 32, exact
    const __half2 c01 = __hsub2(u32_as_h2(v01), bias), c23 = __hsub2(u32_as_h2(v23), bias);
    const uint32_t e = (dh >> 10) & 31u;
    const float F = __uint_as_float((152u - e) << 23);   // 2^(25 - e)
    rinv = __uint_as_float((126u + e) << 23);            // 2^(e - 1)
    const float df = __half2float(__ushort_as_half((unsigned short)dh)) * F;
    const __half2 s01 = __hmul2(c01, __floats2half2_rn(df, df * 0.25f));
    const __half2 s23 = __hmul2(c23, __floats2half2_rn(df * 0.0625f, df * 0.03125f));
    // -4 S 2^-24 = -(S / 2^b_r) 2^(b_r - 22): exact power-of-two products
    const __half2 o01 = __hmul2(s01, __floats2half2_rn(-0x1p-22f, -0x1p-20f));
    const __half2 o23 = __hmul2(s23, __floats2half2_rn(-0x1p-18f, -0x1p-17f));
    S[0] = __low2half2(s01);
    S[1] = __high2half2(s01);
    S[2] = __low2half2(s23);
    S[3] = __high2half2(s23);
    O[0] = __low2half2(o01);
    O[1] = __high2half2(o01);
    O[2] = __low2half2(o23);
    O[3] = __high2half2(o23);
  }

  // u 2^b_r in each byte of a word, from its quant byte q and its hmask byte
  // h already shifted down by 4hq (bit r = this half's high bit of field r)
  __device__ __forceinline__ static uint32_t ubytes(uint32_t q, uint32_t h, int r) {
    if (r < 3)
      return lop3_and_or(h << (r + 2), 0x04040404u << (2 * r), q & (0x03030303u << (2 * r)));
    return lop3_and_or(h << 4, 0x80808080u, (q >> 1) & 0x60606060u);
  }

  template <int NT, bool MIS2>
  __device__ __forceinline__ static void run_impl(uint32_t wrow, int pitch8,
                                                  const uint32_t (&xcol)[NT], int kb, int t,
                                                  float (&acc)[NT][2][4], float& r0, float& r8) {
    __half2 S0[4], O0[4], S8[4], O8[4];
    scales<MIS2>(wrow, t, S0, O0, r0);
    scales<MIS2>(wrow + pitch8, t, S8, O8, r8);
    const uint32_t sh = 4u * (uint32_t)(t >> 1);
    const int kl = kb + 128 * (t >> 1) + 16 * (t & 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int w = (i + t) & 3;
      const uint32_t qa = wrow + 32 + 16 * t + 4 * w;      // qs[32hq + 16(t&1) + 4w]
      const uint32_t ha = wrow + 16 * (t & 1) + 4 * w;     // hmask[16(t&1) + 4w]
      const uint32_t q0 = ld<MIS2>(qa), q8 = ld<MIS2>(qa + pitch8);
      const uint32_t e0 = ld<MIS2>(ha) >> sh, e8 = ld<MIS2>(ha + pitch8) >> sh;
      uint32_t xb[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) xb[nt] = xcol[nt] + 2 * xoff(kl + 4 * w);
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t u0 = ubytes(q0, e0, r), u8 = ubytes(q8, e8, r);
        const __half2 s0 = S0[r], o0 = O0[r], s8 = S8[r], o8 = O8[r];
        const uint32_t a0 = h2_as_u32(__hfma2(u32_as_h2(__byte_perm(u0, 0, 0x4140)), s0, o0));
        const uint32_t a1 = h2_as_u32(__hfma2(u32_as_h2(__byte_perm(u8, 0, 0x4140)), s8, o8));
        const uint32_t a2 = h2_as_u32(__hfma2(u32_as_h2(__byte_perm(u0, 0, 0x4342)), s0, o0));
        const uint32_t a3 = h2_as_u32(__hfma2(u32_as_h2(__byte_perm(u8, 0, 0x4342)), s8, o8));
        mma_xb<NT>(acc, r & 1, a0, a1, a2, a3, xb, field_xoff(r));
      }
    }
  }

  template <int NT, bool PAIRX = false>
  __device__ __forceinline__ static void run(uint32_t wrow, int pitch8,
                                             const uint32_t (&xcol)[NT], int kb, int t,
                                             float (&acc)[NT][2][4], float& r0, float& r8) {
    // the block offset is the same for every row of a stage: a uniform branch
    if (wrow & 2u) run_impl<NT, true>(wrow, pitch8, xcol, kb, t, acc, r0, r8);
    else run_impl<NT, false>(wrow, pitch8, xcol, kb, t, acc, r0, r8);
  }
};

// NVFP4: lane t owns the four 16-weight blocks 4t..4t+3 (weights 64t..64t+63,
// code bytes 32t..32t+31) and their scales (scale bytes 4t..4t+3).  Step m
// (0..15) takes weights 64t+4m..+3: the hardware converts two code bytes to
// two fp16 pairs (exact) and one HMUL2 applies the block's E4M3 scale
// (exact: the products keep <= 6 significant bits and stay within
// 2^-10..2688).  Absolute fp16 weights.
template <>
struct SBDot<DQ_NVFP4> {
  static constexpr bool kRowScale = false;
  template <int NT, bool PAIRX = false>
  __device__ __forceinline__ static void run(uint32_t wrow, int pitch8,
                                             const uint32_t (&xcol)[NT], int kb, int t,
                                             float (&acc)[NT][2][4]) {
    const uint32_t rows[2] = {wrow, wrow + pitch8};
    uint32_t cw[2][8];
    __half2 sc[2][4];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const uint4 a = lds_u128_nv(rows[rr] + 16 + 32 * t), b = lds_u128_nv(rows[rr] + 32 + 32 * t);
      cw[rr][0] = a.x; cw[rr][1] = a.y; cw[rr][2] = a.z; cw[rr][3] = a.w;
      cw[rr][4] = b.x; cw[rr][5] = b.y; cw[rr][6] = b.z; cw[rr][7] = b.w;
      const uint32_t sw = lds_u32_nv(rows[rr] + 4 * t);            // scales of blocks 4t..4t+3
      const __half2 s01 = u32_as_h2(e4m3x2_to_h2((uint16_t)(sw & 0xFFFF)));
      const __half2 s23 = u32_as_h2(e4m3x2_to_h2((uint16_t)(sw >> 16)));
      sc[rr][0] = __low2half2(s01);
      sc[rr][1] = __high2half2(s01);
      sc[rr][2] = __low2half2(s23);
      sc[rr][3] = __high2half2(s23);
    }
#pragma unroll
    for (int wv = 0; wv < 8; ++wv) {                 // code word wv: steps 2wv, 2wv+1
      uint32_t h0[4], h8[4];
      e2m1x8_to_h2x4(cw[0][wv], h0);
      e2m1x8_to_h2x4(cw[1][wv], h8);
      const __half2 s0 = sc[0][wv >> 1], s8 = sc[1][wv >> 1];
#pragma unroll
      for (int hm = 0; hm < 2; ++hm) {
        const int m = 2 * wv + hm;
        const uint32_t a0 = h2_as_u32(__hmul2(u32_as_h2(h0[2 * hm]), s0));
        const uint32_t a1 = h2_as_u32(__hmul2(u32_as_h2(h8[2 * hm]), s8));
        const uint32_t a2 = h2_as_u32(__hmul2(u32_as_h2(h0[2 * hm + 1]), s0));
        const uint32_t a3 = h2_as_u32(__hmul2(u32_as_h2(h8[2 * hm + 1]), s8));
        mma_x<NT>(acc, m & 1, a0, a1, a2, a3, xcol, kb + 64 * t + 4 * m);
      }
    }
  }
};

// ---------------------------------------------------------------------------
// Q4_K with one activation column (decode at batch 1).
//
// With a single column, the 8 columns of mma.m16n8k16 are free to carry the 8
// sub-blocks of a super-block instead: B is block-diagonal (column j holds the
// activations of sub-block j, zeros elsewhere), so one accumulator keeps the 8
// per-sub-block dot products apart, and every scale and min is applied once per
// sub-block, in fp32, after the products:
//   y_row += d sc_j (sum_k q_k x_k) - dmin m_j (sum_k x_k)      (Q4_K, j = 0..7)
// with the sub-block sums of x computed once per activation vector.
//
// A holds quant bytes spread into 16-bit lanes, read as exact fp16
// subnormals: b * 2^-24 for a whole byte b = lo + 16 hi, lo * 2^-24 for its
// low nibble.  Byte j of qs group c carries weight j of sub-block 2c (low
// nibble) and of sub-block 2c+1 (high nibble), so with
//   mma 1:  A = b,   B column 2c+1 = +x(2c+1)
//   mma 2:  A = lo,  B column 2c = +x(2c),  column 2c+1 = -x(2c+1)
// column 2c gets sum lo x and column 2c+1 gets 16 sum hi x: the high nibble
// never needs its own mask.
//
// Lane (g, t) supplies rows g and g+8 and weights 8t..8t+7 of every
// sub-block; its B fragment is real only for sub-block g (16 bytes of x, or
// of -x for the second product of an odd sub-block) and reads zero bytes
// otherwise.  Its accumulator ends with sub-blocks 2t and 2t+1 of both rows.
// ---------------------------------------------------------------------------
struct Q4KB1 {
  // Per-lane constants, set once per kernel.
  struct Lane {
    int t;
    uint32_t sel_a;    // byte selector: scale bytes 2(t&1), +1 of hd.y (t < 2) or hd.w (t >= 2)
    uint32_t sel_b;    // the same bytes of the first source, zeros above them
    uint32_t sh_m;     // mins of sub-blocks 4..7 sit in the high nibbles: shift 4
    uint32_t mask_a;   // 6 (t < 2) or 4 (t >= 2) low bits per 16-bit lane
    uint32_t mask_b;   // bits 4-5 of each lane from the top 2 bits (t >= 2 only)
    uint32_t real[4];  // 1 for qs group c == g/2 (the group holding sub-block g), else 0
    uint32_t odd;      // g odd: this lane's sub-block is a high-nibble one
  };
  __device__ __forceinline__ static Lane lane_consts(int g, int t) {
    Lane L;
    L.t = t;
    const uint32_t jj = 2u * (uint32_t)(t & 1);
    const uint32_t hiw = t >= 2 ? 4u : 0u;   // PRMT indices 4-7 address the second source
    // bytes 1 and 3 of each result are don't-care (cleared by the masks)
    L.sel_a = (jj + hiw) | ((jj + 1 + hiw) << 8);
    L.sel_b = jj | (4u << 4) | ((jj + 1) << 8) | (4u << 12);
    L.sh_m = t >= 2 ? 4u : 0u;
    L.mask_a = t >= 2 ? 0x000F000Fu : 0x003F003Fu;
    L.mask_b = t >= 2 ? 0x00300030u : 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c) L.real[c] = (c == (g >> 1)) ? 1u : 0u;
    L.odd = (uint32_t)(g & 1);
    return L;
  }

  // Stage activations: [0, 512) fp16 x of sub-blocks 0..7 (16 bytes per lane
  // t at 64 j + 16 t); [512, 1024) -x of the odd sub-blocks at the same offsets.
  static constexpr int kStageX = 1024;

  // 6-bit scales and mins of sub-blocks 2t (x) and 2t+1 (y) as exact floats.
  // Sub-blocks 0-3: low 6 bits of scales[j] / scales[j+4]; 4-7: low / high
  // nibble of scales[j+4] with the top 2 bits of scales[j-4] / scales[j].
  __device__ __forceinline__ static void sub_scales(uint4 hd, const Lane& L, float2& sc,
                                                    float2& mn) {
    const uint32_t as = __byte_perm(hd.y, hd.w, L.sel_a);
    const uint32_t am = __byte_perm(hd.z, hd.w, L.sel_a) >> L.sh_m;
    const uint32_t bs = (__byte_perm(hd.y, 0, L.sel_b) >> 2) & L.mask_b;
    const uint32_t bm = (__byte_perm(hd.z, 0, L.sel_b) >> 2) & L.mask_b;
    const uint32_t s = (as & L.mask_a) | bs | 0x64006400u;
    const uint32_t m = (am & L.mask_a) | bm | 0x64006400u;
    const __half2 magic = u32_as_h2(0x64006400u);
    sc = __half22float2(__hsub2(u32_as_h2(s), magic));
    mn = __half22float2(__hsub2(u32_as_h2(m), magic));
  }

  // Shared addresses (wrow, xg, nsx) must come through order_after_wait() of
  // the stage's full barrier; acc must pass keep_before_release() before the
  // stage is released (the loads themselves are freely scheduled).
  // wrow: shared address of row g's super-block, row g+8 at wrow + pitch8.
  // xst: the stage's activations; xg = xst + 64 g + 16 t (this lane's x).
  // z: 16 zero bytes on banks 0-3 (no real lane of a quarter-warp reads them).
  // nsx: shared address of (-sum x of sub-block 2t, -sum of 2t+1).
  // inv: the activations' inverse power-of-two scale.
  // acc0 / acc8: rows g / g+8, as (sub-block 2t, 2t+1) pairs summed at the end.
  __device__ __forceinline__ static void run(uint32_t wrow, int pitch8, uint32_t xg, uint32_t z,
                                             uint32_t nsx, float inv, const Lane& L,
                                             float2& acc0, float2& acc8) {
    const uint4 h0 = lds_u128_nv(wrow), h8 = lds_u128_nv(wrow + pitch8);
    // first product: x of an odd sub-block; second: x (even) or -x (odd)
    const uint32_t d1 = L.odd * (xg - z), d2 = xg + L.odd * 512u - z;
    float D[4][4] = {};   // one chain per qs group
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint2 w0 = lds_u64_nv(wrow + 16 + 32 * c + 8 * L.t);
      const uint2 w8 = lds_u64_nv(wrow + pitch8 + 16 + 32 * c + 8 * L.t);
      const uint4 x1 = lds_u128_nv(z + L.real[c] * d1);
      const uint4 x2 = lds_u128_nv(z + L.real[c] * d2);
      const uint32_t b0[4] = {__byte_perm(w0.x, 0, 0x4140), __byte_perm(w0.x, 0, 0x4342),
                              __byte_perm(w0.y, 0, 0x4140), __byte_perm(w0.y, 0, 0x4342)};
      const uint32_t b8[4] = {__byte_perm(w8.x, 0, 0x4140), __byte_perm(w8.x, 0, 0x4342),
                              __byte_perm(w8.y, 0, 0x4140), __byte_perm(w8.y, 0, 0x4342)};
      // k slots (2t, 2t+1 | 2t+8, 2t+9) = weights (8t, 8t+1 | 8t+2, 8t+3), then +4
      mma_16816_nv(D[c], b0[0], b8[0], b0[1], b8[1], x1.x, x1.y);
      mma_16816_nv(D[c], b0[2], b8[2], b0[3], b8[3], x1.z, x1.w);
      mma_16816_nv(D[c], b0[0] & 0x000F000Fu, b8[0] & 0x000F000Fu, b0[1] & 0x000F000Fu,
                b8[1] & 0x000F000Fu, x2.x, x2.y);
      mma_16816_nv(D[c], b0[2] & 0x000F000Fu, b8[2] & 0x000F000Fu, b0[3] & 0x000F000Fu,
                b8[3] & 0x000F000Fu, x2.z, x2.w);
    }
    const uint2 nsu = lds_u64_nv(nsx);
    const float2 ns = make_float2(__uint_as_float(nsu.x), __uint_as_float(nsu.y));
    float2 sc0, mn0, sc8, mn8;
    sub_scales(h0, L, sc0, mn0);
    sub_scales(h8, L, sc8, mn8);
    // (d, dmin) of each row; with the activation scale undone
    float2 dm0 = __half22float2(u32_as_h2(h0.x)), dm8 = __half22float2(u32_as_h2(h8.x));
    dm0 = fmul2(dm0, make_float2(inv, inv));
    dm8 = fmul2(dm8, make_float2(inv, inv));
    // column 2t: low nibbles in units of 2^-24; column 2t+1: high, 16 * 2^-24
    const float2 unit = make_float2(16777216.f, 1048576.f);
    const float2 c0 = fmul2(fmul2(sc0, unit), make_float2(dm0.x, dm0.x));
    const float2 c8 = fmul2(fmul2(sc8, unit), make_float2(dm8.x, dm8.x));
    const float2 k0 = fmul2(mn0, make_float2(dm0.y, dm0.y));
    const float2 k8 = fmul2(mn8, make_float2(dm8.y, dm8.y));
    const float2 s0 = fadd2(fadd2(make_float2(D[0][0], D[0][1]), make_float2(D[1][0], D[1][1])),
                            fadd2(make_float2(D[2][0], D[2][1]), make_float2(D[3][0], D[3][1])));
    const float2 s8 = fadd2(fadd2(make_float2(D[0][2], D[0][3]), make_float2(D[1][2], D[1][3])),
                            fadd2(make_float2(D[2][2], D[2][3]), make_float2(D[3][2], D[3][3])));
    acc0 = ffma2(ns, k0, ffma2(s0, c0, acc0));
    acc8 = ffma2(ns, k8, ffma2(s8, c8, acc8));
  }
};

// ---------------------------------------------------------------------------
// Q6_K with one activation column: the block-diagonal core for 16-weight
// sub-blocks.  A super-block has 16 of them, so it takes two rounds of the 8
// mma columns: round h carries sub-blocks 8h + n in column n, n = 2r + lh,
// i.e. the 16 weights 128h + 32r + 16lh + [0, 16).  A holds q (6 bits) as
// exact fp16 subnormals q * 2^-24; each sub-block is scaled once in fp32:
//   y_row += d sc_j (sum_k q_k x_k - 32 sum_k x_k)               (j = 0..15)
// Lane (g, t) supplies rows g and g+8 and weights l = 16lh + 4t + [0, 4) of
// every sub-block: the low nibbles from ql[64h + 32(r&1) + l] (high nibbles
// for r >= 2), bits 2r..2r+1 from qh[32h + l].  Its accumulators end with
// sub-blocks 8h + 2t and 8h + 2t + 1 of both rows, h = 0, 1.
// ---------------------------------------------------------------------------
struct Q6KB1 {
  // 32-bit word at a 2-byte aligned shared address whose misalignment
  // (0 or 2 bytes, `mis`) is uniform for the stage
  template <bool MIS>
  __device__ __forceinline__ static uint32_t ldw(uint32_t a) {
    if constexpr (!MIS) {
      return lds_u32_nv(a);
    } else {
      const uint32_t lo = lds_u32_nv(a - 2), hi = lds_u32_nv(a + 2);
      return __funnelshift_r(lo, hi, 16);
    }
  }

  // q bytes (4 weights) of run r from the low-bit word (ql, run r&1) and the
  // high-bit word (qh)
  __device__ __forceinline__ static uint32_t q4(uint32_t ql, uint32_t qh, int r) {
    const uint32_t lo = (r & 2) ? (ql >> 4) : ql;
    const uint32_t hb = r == 0 ? (qh << 4) : r == 1 ? (qh << 2) : r == 2 ? qh : (qh >> 2);
    return (lo & 0x0F0F0F0Fu) | (hb & 0x30303030u);
  }

  // one round (half h of the super-block) of rows g / g+8 (ra / rb: their
  // super-block starts) into D[2][4]
  template <bool MIS>
  __device__ __forceinline__ static void round(uint32_t ra, uint32_t rb, int h, uint32_t xs,
                                               uint32_t z, const uint32_t (&real)[8], int t,
                                               float (&D)[2][4]) {
    uint32_t Q[2][2][2], H[2][2];   // [row][run&1][lh], [row][lh]
    const uint32_t rows[2] = {ra, rb};
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int lh = 0; lh < 2; ++lh) {
        Q[rr][0][lh] = ldw<MIS>(rows[rr] + 64 * h + 16 * lh + 4 * t);
        Q[rr][1][lh] = ldw<MIS>(rows[rr] + 64 * h + 32 + 16 * lh + 4 * t);
        H[rr][lh] = ldw<MIS>(rows[rr] + 128 + 32 * h + 16 * lh + 4 * t);
      }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int lh = 0; lh < 2; ++lh) {
        const int n = 2 * r + lh;   // column = sub-block 8h + n
        const uint32_t w0 = q4(Q[0][r & 1][lh], H[0][lh], r);
        const uint32_t w8 = q4(Q[1][r & 1][lh], H[1][lh], r);
        const uint2 xv = lds_u64_nv(z + real[n] * (xs + 32 * (8 * h + n) - z));
        // k slots (2t, 2t+1 | 2t+8, 2t+9) = weights l + (0, 1 | 2, 3)
        mma_16816_nv(D[lh], __byte_perm(w0, 0, 0x4140), __byte_perm(w8, 0, 0x4140),
                     __byte_perm(w0, 0, 0x4342), __byte_perm(w8, 0, 0x4342), xv.x, xv.y);
      }
  }

  // The two rounds and their scales.  ra / rb: shared addresses of the
  // super-block in rows g / g+8 (2-byte aligned; MIS: 2 mod 4), from
  // order_after_wait() of the stage barrier.  xs: the stage's activations
  // (fp16, natural order; this lane reads 8 bytes at xs + 32 j + 8 t);
  // z: 8 zero bytes; nsx: the stage's 16 negated sub-block sums (fp32);
  // inv: inverse activation scale.
  template <bool MIS>
  __device__ __forceinline__ static void run(uint32_t ra, uint32_t rb, uint32_t xs, uint32_t z,
                                             uint32_t nsx, float inv, const uint32_t (&real)[8],
                                             int t, float2& acc0, float2& acc8) {
    const uint32_t xl = xs + 8 * t;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float D[2][4] = {};
      round<MIS>(ra, rb, h, xl, z, real, t, D);
      // sub-blocks j = 8h + 2t + (0, 1): scales, d, -sum x
      const uint32_t s0 = lds_u16_nv(ra + 192 + 8 * h + 2 * t);
      const uint32_t s8 = lds_u16_nv(rb + 192 + 8 * h + 2 * t);
      const float d0 = __half2float(__ushort_as_half((unsigned short)lds_u16_nv(ra + 208))) * inv;
      const float d8 = __half2float(__ushort_as_half((unsigned short)lds_u16_nv(rb + 208))) * inv;
      const uint2 nsu = lds_u64_nv(nsx + 4 * (8 * h + 2 * t));
      const float2 ns = make_float2(__uint_as_float(nsu.x), __uint_as_float(nsu.y));
      const float2 sc0 = make_float2((float)(int8_t)(s0 & 0xFF), (float)(int8_t)(s0 >> 8));
      const float2 sc8 = make_float2((float)(int8_t)(s8 & 0xFF), (float)(int8_t)(s8 >> 8));
      // products in units of 2^-24; the -32 offset against the sums
      const float2 c0 = fmul2(sc0, make_float2(d0 * 16777216.f, d0 * 16777216.f));
      const float2 c8 = fmul2(sc8, make_float2(d8 * 16777216.f, d8 * 16777216.f));
      const float2 k0 = fmul2(sc0, make_float2(32.f * d0, 32.f * d0));
      const float2 k8 = fmul2(sc8, make_float2(32.f * d8, 32.f * d8));
      // column 2t (even sub-block) accumulates in chain 0, 2t+1 in chain 1
      acc0 = ffma2(ns, k0, ffma2(make_float2(D[0][0], D[1][1]), c0, acc0));
      acc8 = ffma2(ns, k8, ffma2(make_float2(D[0][2], D[1][3]), c8, acc8));
    }
  }
};

// ---------------------------------------------------------------------------
// Q2_K and Q3_K with one activation column: Q6_K's two block-diagonal rounds
// (round h: sub-block 8h + n in mma column n, n = 2r + lh; lane t supplies
// weights 16lh + 4t + [0, 4) of run r, i.e. one quant word per (h, lh) serves
// the four runs).  The 2-bit field r is masked in place, so column n sums
// (q 4^r 2^-24) x (Q3_K: u = q + 4 assembled as u 2^b_r, b_r = 0, 2, 4, 5) and
// every scale is applied per sub-block in fp32 after the products:
//   Q2_K: y_row += d sc_j (sum q x) - dmin m_j (sum x)
//   Q3_K: y_row += d (s_j - 32) (sum u x - 4 sum x)
// The lane's columns 2t, 2t+1 both hold run r = t: one factor 4^-t (2^-b_t).
// ---------------------------------------------------------------------------
struct Q2KB1 {
  // one round (half h) of rows g / g+8 (ra / rb: their super-block starts,
  // 4-byte aligned) into D[2][4]
  __device__ __forceinline__ static void round(uint32_t ra, uint32_t rb, int h, uint32_t xs,
                                               uint32_t z, const uint32_t (&real)[8], int t,
                                               float (&D)[2][4]) {
    uint32_t L[2][2], H[2][2];   // [row][lh]: bytes (0, 1) and (2, 3) in 16-bit lanes
    const uint32_t rows[2] = {ra, rb};
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int lh = 0; lh < 2; ++lh) {
        const uint32_t q = lds_u32_nv(rows[rr] + 16 + 32 * h + 16 * lh + 4 * t);
        L[rr][lh] = __byte_perm(q, 0, 0x4140);
        H[rr][lh] = __byte_perm(q, 0, 0x4342);
      }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int lh = 0; lh < 2; ++lh) {
        const int n = 2 * r + lh;
        const uint32_t m = 0x00030003u << (2 * r);
        const uint2 xv = lds_u64_nv(z + real[n] * (xs + 32 * (8 * h + n) - z));
        mma_16816_nv(D[lh], L[0][lh] & m, L[1][lh] & m, H[0][lh] & m, H[1][lh] & m, xv.x, xv.y);
      }
  }

  // ra / rb: shared addresses of the super-block in rows g / g+8 (from
  // order_after_wait() of the stage barrier); xs: the stage's activations;
  // z: 8 zero bytes; nsx: the stage's 16 negated sub-block sums; inv: inverse
  // activation scale; f: 2^24 4^-t.
  __device__ __forceinline__ static void run(uint32_t ra, uint32_t rb, uint32_t xs, uint32_t z,
                                             uint32_t nsx, float inv, float f,
                                             const uint32_t (&real)[8], int t, float2& acc0,
                                             float2& acc8) {
    const uint32_t xl = xs + 8 * t;
    const uint32_t dd0 = lds_u32_nv(ra + 80), dd8 = lds_u32_nv(rb + 80);   // d | dmin << 16
    const float d0 = __half2float(__ushort_as_half((unsigned short)(dd0 & 0xFFFF))) * inv;
    const float m0 = __half2float(__ushort_as_half((unsigned short)(dd0 >> 16))) * inv;
    const float d8 = __half2float(__ushort_as_half((unsigned short)(dd8 & 0xFFFF))) * inv;
    const float m8 = __half2float(__ushort_as_half((unsigned short)(dd8 >> 16))) * inv;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float D[2][4] = {};
      round(ra, rb, h, xl, z, real, t, D);
      // sub-blocks j = 8h + 2t + (0, 1): scale | min << 4 bytes, -sum x
      const uint32_t s0 = lds_u16_nv(ra + 8 * h + 2 * t), s8 = lds_u16_nv(rb + 8 * h + 2 * t);
      const uint2 nsu = lds_u64_nv(nsx + 4 * (8 * h + 2 * t));
      const float2 ns = make_float2(__uint_as_float(nsu.x), __uint_as_float(nsu.y));
      const float2 sc0 = make_float2((float)(s0 & 15), (float)((s0 >> 8) & 15));
      const float2 mn0 = make_float2((float)((s0 >> 4) & 15), (float)(s0 >> 12));
      const float2 sc8 = make_float2((float)(s8 & 15), (float)((s8 >> 8) & 15));
      const float2 mn8 = make_float2((float)((s8 >> 4) & 15), (float)(s8 >> 12));
      const float2 c0 = fmul2(sc0, make_float2(d0 * f, d0 * f));
      const float2 c8 = fmul2(sc8, make_float2(d8 * f, d8 * f));
      const float2 k0 = fmul2(mn0, make_float2(m0, m0));
      const float2 k8 = fmul2(mn8, make_float2(m8, m8));
      // column 2t (even sub-block) accumulates in chain 0, 2t+1 in chain 1
      acc0 = ffma2(ns, k0, ffma2(make_float2(D[0][0], D[1][1]), c0, acc0));
      acc8 = ffma2(ns, k8, ffma2(make_float2(D[0][2], D[1][3]), c8, acc8));
    }
  }
};

struct Q3KB1 {
  template <bool MIS>
  __device__ __forceinline__ static uint32_t ldw(uint32_t a) {
    if constexpr (!MIS) {
      return lds_u32_nv(a);
    } else {
      const uint32_t lo = lds_u32_nv(a - 2), hi = lds_u32_nv(a + 2);
      return __funnelshift_r(lo, hi, 16);
    }
  }

  // u 2^b_r in each byte from the quant word q and the hmask word h shifted
  // down by 4h (bit r = the high bit of run r)
  __device__ __forceinline__ static uint32_t ubytes(uint32_t q, uint32_t h, int r) {
    if (r < 3)
      return lop3_and_or(h << (r + 2), 0x04040404u << (2 * r), q & (0x03030303u << (2 * r)));
    return lop3_and_or(h << 4, 0x80808080u, (q >> 1) & 0x60606060u);
  }

  template <bool MIS>
  __device__ __forceinline__ static void round(uint32_t ra, uint32_t rb, int h, uint32_t xs,
                                               uint32_t z, const uint32_t (&real)[8], int t,
                                               float (&D)[2][4]) {
    uint32_t Q[2][2], E[2][2];   // [row][lh]: quant word, hmask word >> 4h
    const uint32_t rows[2] = {ra, rb};
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int lh = 0; lh < 2; ++lh) {
        Q[rr][lh] = ldw<MIS>(rows[rr] + 32 + 32 * h + 16 * lh + 4 * t);
        E[rr][lh] = ldw<MIS>(rows[rr] + 16 * lh + 4 * t) >> (4 * h);
      }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int lh = 0; lh < 2; ++lh) {
        const int n = 2 * r + lh;
        const uint32_t w0 = ubytes(Q[0][lh], E[0][lh], r), w8 = ubytes(Q[1][lh], E[1][lh], r);
        const uint2 xv = lds_u64_nv(z + real[n] * (xs + 32 * (8 * h + n) - z));
        mma_16816_nv(D[lh], __byte_perm(w0, 0, 0x4140), __byte_perm(w8, 0, 0x4140),
                     __byte_perm(w0, 0, 0x4342), __byte_perm(w8, 0, 0x4342), xv.x, xv.y);
      }
  }

  // As Q2KB1::run; the super-block is 2-byte aligned (MIS: 2 mod 4);
  // f: 2^24 2^-b_t.
  template <bool MIS>
  __device__ __forceinline__ static void run(uint32_t ra, uint32_t rb, uint32_t xs, uint32_t z,
                                             uint32_t nsx, float inv, float f,
                                             const uint32_t (&real)[8], int t, float2& acc0,
                                             float2& acc8) {
    const uint32_t xl = xs + 8 * t;
    const float d0 = __half2float(__ushort_as_half((unsigned short)lds_u16_nv(ra + 108))) * inv;
    const float d8 = __half2float(__ushort_as_half((unsigned short)lds_u16_nv(rb + 108))) * inv;
    // sub-blocks j = 8h + 2t + (0, 1): low nibbles h of scale bytes 2t, 2t+1;
    // top bits: field 2h + t/2 of bytes 8 + 2(t&1), +1
    const uint32_t l0 = lds_u16_nv(ra + 96 + 2 * t), l8 = lds_u16_nv(rb + 96 + 2 * t);
    const uint32_t u0 = lds_u16_nv(ra + 104 + 2 * (t & 1)), u8 = lds_u16_nv(rb + 104 + 2 * (t & 1));
    const int hs = 2 * (t >> 1);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float D[2][4] = {};
      round<MIS>(ra, rb, h, xl, z, real, t, D);
      const uint32_t v0 = ((l0 >> (4 * h)) & 0x0F0Fu) | (((u0 >> (4 * h + hs)) & 0x0303u) << 4);
      const uint32_t v8 = ((l8 >> (4 * h)) & 0x0F0Fu) | (((u8 >> (4 * h + hs)) & 0x0303u) << 4);
      const float2 sc0 = make_float2((float)((int)(v0 & 63) - 32), (float)((int)(v0 >> 8) - 32));
      const float2 sc8 = make_float2((float)((int)(v8 & 63) - 32), (float)((int)(v8 >> 8) - 32));
      const uint2 nsu = lds_u64_nv(nsx + 4 * (8 * h + 2 * t));
      const float2 ns = make_float2(__uint_as_float(nsu.x), __uint_as_float(nsu.y));
      const float2 c0 = fmul2(sc0, make_float2(d0 * f, d0 * f));
      const float2 c8 = fmul2(sc8, make_float2(d8 * f, d8 * f));
      const float2 k0 = fmul2(sc0, make_float2(4.f * d0, 4.f * d0));
      const float2 k8 = fmul2(sc8, make_float2(4.f * d8, 4.f * d8));
      acc0 = ffma2(ns, k0, ffma2(make_float2(D[0][0], D[1][1]), c0, acc0));
      acc8 = ffma2(ns, k8, ffma2(make_float2(D[0][2], D[1][3]), c8, acc8));
    }
  }
};

// ---------------------------------------------------------------------------
// Q8_0 with one activation column: the block-diagonal core.  The 8 blocks of
// 32 weights of a super-block go to the 8 mma columns.  A holds q + 128 (the
// int8 quant with its sign bit flipped) as exact fp16 subnormals, and each
// block is scaled once in fp32:
//   y_row += d_j (sum_k (q_k + 128) x_k - 128 sum_k x_k)            (j = 0..7)
// Lane (g, t) supplies rows g and g+8 and weights 8t..8t+7 of every block
// (bytes 34j + 2 + 8t ..: 4-byte aligned for odd j, 2 bytes off for even j,
// both known at compile time); its accumulators end with blocks 2t and 2t+1.
// ---------------------------------------------------------------------------
struct Q80B1 {
  // bytes q_{8t..8t+7} of block J of one row (super-block at `row`), as two
  // words with the sign bits flipped
  template <int J>
  __device__ __forceinline__ static uint2 quants(uint32_t row, int t) {
    const uint32_t a = row + 34 * J + 2 + 8 * t;
    uint32_t w0, w1;
    if constexpr (J & 1) {
      w0 = lds_u32_nv(a);
      w1 = lds_u32_nv(a + 4);
    } else {
      const uint32_t p = lds_u32_nv(a - 2), q = lds_u32_nv(a + 2), r = lds_u32_nv(a + 6);
      w0 = __funnelshift_r(p, q, 16);
      w1 = __funnelshift_r(q, r, 16);
    }
    return make_uint2(w0 ^ 0x80808080u, w1 ^ 0x80808080u);
  }

  template <int J>
  __device__ __forceinline__ static void block(uint32_t ra, uint32_t rb, uint32_t xg, uint32_t z,
                                               uint32_t real, int t, float (&D)[4]) {
    const uint2 q0 = quants<J>(ra, t), q8 = quants<J>(rb, t);
    const uint4 xv = lds_u128_nv(z + real * (xg - z));
    // k slots (2t, 2t+1 | 2t+8, 2t+9) = weights (8t, 8t+1 | 8t+2, 8t+3), then +4
    mma_16816_nv(D, __byte_perm(q0.x, 0, 0x4140), __byte_perm(q8.x, 0, 0x4140),
                 __byte_perm(q0.x, 0, 0x4342), __byte_perm(q8.x, 0, 0x4342), xv.x, xv.y);
    mma_16816_nv(D, __byte_perm(q0.y, 0, 0x4140), __byte_perm(q8.y, 0, 0x4140),
                 __byte_perm(q0.y, 0, 0x4342), __byte_perm(q8.y, 0, 0x4342), xv.z, xv.w);
  }

  // ra / rb: shared addresses of the super-block (272 bytes, 16-byte aligned)
  // in rows g / g+8, from order_after_wait() of the stage barrier; xg: this
  // lane's 16 bytes of x (block g, weights 8t..8t+7); ze / zo: 16 zero bytes
  // read in place of x for even / odd blocks; nsx: (-sum x of block 2t,
  // -sum of 2t+1); real[j]: block j is this lane's own (j == g).
  __device__ __forceinline__ static void run(uint32_t ra, uint32_t rb, uint32_t xg, uint32_t ze,
                                             uint32_t zo, uint32_t nsx, float inv,
                                             const uint32_t (&real)[8], int t, float2& acc0,
                                             float2& acc8) {
    float D[4][4] = {};   // four chains: blocks j, j + 4
    block<0>(ra, rb, xg, ze, real[0], t, D[0]);
    block<1>(ra, rb, xg, zo, real[1], t, D[1]);
    block<2>(ra, rb, xg, ze, real[2], t, D[2]);
    block<3>(ra, rb, xg, zo, real[3], t, D[3]);
    block<4>(ra, rb, xg, ze, real[4], t, D[0]);
    block<5>(ra, rb, xg, zo, real[5], t, D[1]);
    block<6>(ra, rb, xg, ze, real[6], t, D[2]);
    block<7>(ra, rb, xg, zo, real[7], t, D[3]);
    // d of blocks 2t, 2t+1 of each row
    const float d0a = __half2float(__ushort_as_half((unsigned short)lds_u16_nv(ra + 68 * t)));
    const float d0b = __half2float(__ushort_as_half((unsigned short)lds_u16_nv(ra + 68 * t + 34)));
    const float d8a = __half2float(__ushort_as_half((unsigned short)lds_u16_nv(rb + 68 * t)));
    const float d8b = __half2float(__ushort_as_half((unsigned short)lds_u16_nv(rb + 68 * t + 34)));
    const uint2 nsu = lds_u64_nv(nsx);
    const float2 ns = make_float2(__uint_as_float(nsu.x), __uint_as_float(nsu.y));
    const float2 dd0 = fmul2(make_float2(d0a, d0b), make_float2(inv, inv));
    const float2 dd8 = fmul2(make_float2(d8a, d8b), make_float2(inv, inv));
    // products in units of 2^-24; the +128 offset against the sums
    const float2 c0 = fmul2(dd0, make_float2(16777216.f, 16777216.f));
    const float2 c8 = fmul2(dd8, make_float2(16777216.f, 16777216.f));
    const float2 k0 = fmul2(dd0, make_float2(128.f, 128.f));
    const float2 k8 = fmul2(dd8, make_float2(128.f, 128.f));
    const float2 s0 = fadd2(fadd2(make_float2(D[0][0], D[0][1]), make_float2(D[1][0], D[1][1])),
                            fadd2(make_float2(D[2][0], D[2][1]), make_float2(D[3][0], D[3][1])));
    const float2 s8 = fadd2(fadd2(make_float2(D[0][2], D[0][3]), make_float2(D[1][2], D[1][3])),
                            fadd2(make_float2(D[2][2], D[2][3]), make_float2(D[3][2], D[3][3])));
    acc0 = ffma2(ns, k0, ffma2(s0, c0, acc0));
    acc8 = ffma2(ns, k8, ffma2(s8, c8, acc8));
  }
};

}  // namespace dqmoe
