// b1.cuh — the pieces of the one-activation-column (block-diagonal) GEMV that
// the plain GEMV kernel (qgemv_b1_kernel) and the MoE layer's one-token
// expert kernel (grouped_b1_kernel) share:
//   * the shared-memory plan of a stage ring (weights, activations, negated
//     sub-block sums, inverse activation scales, 16 zero bytes);
//   * the loader's activation staging: one stage = the 256 activations of
//     one super-block, 8 per loader lane, converted to fp16 (bf16 and fp32
//     inputs with one power-of-two scale per stage), with the negated sum of
//     each sub-block (and, for Q4_K, -x of the odd sub-blocks);
//   * the consumers' per-stage product of the format's block-diagonal core.
#pragma once

#include "qgemv_mma.cuh"

namespace dqmoe {

// stages whose activation loads the loader keeps in flight in registers
constexpr int kB1Prefetch = 4;

struct B1Plan {
  int nstage, off_w, off_x, off_sx, off_inv, off_z, off_red, total;
};

// Per stage: activations (Q4_K: x and -x of the odd sub-blocks; the others:
// x) and the negated sums of its 8 (Q4_K, Q8_0) or 16 (Q6_K, Q2_K, Q3_K)
// sub-blocks.
template <int FMT>
struct B1Fmt {
  static constexpr int kStageX = FMT == DQ_Q4_K ? Q4KB1::kStageX : 512;
  static constexpr int kSubs = (FMT == DQ_Q6_K || FMT == DQ_Q2_K || FMT == DQ_Q3_K) ? 16 : 8;
};

template <int FMT>
__host__ __device__ inline B1Plan b1_plan(int nstage, int ksplit) {
  B1Plan p;
  p.nstage = nstage;
  p.off_w = 1024;                                             // barriers below
  p.off_x = p.off_w + nstage * Layout<FMT>::W_STAGE;          // 128-byte aligned
  p.off_sx = p.off_x + nstage * B1Fmt<FMT>::kStageX;
  p.off_inv = p.off_sx + nstage * 4 * B1Fmt<FMT>::kSubs;
  p.off_z = (p.off_inv + nstage * 4 + 127) / 128 * 128;       // 16 zero bytes at +0
  p.off_red = p.off_z + 128;
  p.total = p.off_red + (ksplit > 1 ? (ksplit - 1) * kConsumerWarps * 32 * 16 : 0);
  return p;
}

// A loader lane's raw activations of one stage: 8 values, 16 bytes of fp16 /
// bf16 or 32 bytes of fp32.
template <int XDT>
struct B1X {
  uint4 v[XDT == DQ_F32 ? 2 : 1];
};

// Values 256 c + 8 lane .. + 7 of the activation row `row`.
template <int XDT>
__device__ __forceinline__ B1X<XDT> b1_load_x(const void* row, int c, int lane) {
  B1X<XDT> r;
  if constexpr (XDT == DQ_F32) {
    const uint4* src = (const uint4*)((const float*)row + (int64_t)c * 256) + 2 * lane;
    r.v[0] = __ldg(src);
    r.v[1] = __ldg(src + 1);
  } else {
    r.v[0] = __ldg((const uint4*)((const uint16_t*)row + (int64_t)c * 256) + lane);
  }
  return r;
}

// Convert and store one stage's activations (the loader warp, every lane):
// xst = the stage's activation area, sx = its negated sub-block sums, inv =
// its inverse scale slot.
template <int FMT, int XDT>
__device__ __forceinline__ void b1_stage_x(const B1X<XDT>& r, uint8_t* xst, float* sx, float* inv,
                                           int lane) {
  constexpr int kSubs = B1Fmt<FMT>::kSubs;
  uint32_t h[4];
  float iv = 1.f;
  if constexpr (XDT == DQ_F16) {
    h[0] = r.v[0].x;
    h[1] = r.v[0].y;
    h[2] = r.v[0].z;
    h[3] = r.v[0].w;
  } else {
    float f[8];
    if constexpr (XDT == DQ_BF16) {
      const uint32_t w[4] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[2 * j] = __uint_as_float(w[j] << 16);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    } else {
      const uint32_t w[8] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w,
                             r.v[1].x, r.v[1].y, r.v[1].z, r.v[1].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(w[j]);
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float scale;
    pow2_scale(amax, scale, iv);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      h[j] = h2_as_u32(__floats2half2_rn(f[2 * j] * scale, f[2 * j + 1] * scale));
  }
  *(uint4*)(xst + 16 * lane) = make_uint4(h[0], h[1], h[2], h[3]);
  if (FMT == DQ_Q4_K && (lane & 4))   // odd sub-block: its negation too
    *(uint4*)(xst + 512 + 16 * lane) = make_uint4(h[0] ^ 0x80008000u, h[1] ^ 0x80008000u,
                                                  h[2] ^ 0x80008000u, h[3] ^ 0x80008000u);
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 v = __half22float2(u32_as_h2(h[j]));
    sum += v.x;
    sum += v.y;
  }
  // sub-blocks of 32 (4 lanes) or 16 (2 lanes) activations
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  if (kSubs == 8) sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  constexpr int lanes_per_sub = 32 / kSubs;
  if ((lane & (lanes_per_sub - 1)) == 0) sx[lane / lanes_per_sub] = -sum;
  if (lane == 0) *inv = iv;
}

// The consumers' side: lane (g, t) of consumer warp cw supplies rows
// `rows_a` + rg and `rows_a` + rg + ROWS_B of every stage (ROWS_B = 8 for a
// plain 64-row tile; 32 where the second row is the matching row of a second
// matrix stacked below the first).
template <int FMT, bool SCALED, int ROWS_B>
struct B1Consumer {
  using L = Layout<FMT>;
  static constexpr int pitch_b = ROWS_B * L::ROW_PITCH;
  static constexpr int kStageX = B1Fmt<FMT>::kStageX, kSubs = B1Fmt<FMT>::kSubs;
  int t, rg;
  uint32_t xlane;   // this lane's 16 activation bytes of a Q4_K / Q8_0 stage: 64 g + 16 t
  float f23;
  Q4KB1::Lane lc;
  uint32_t real6[8];
  uint32_t wrow, xbase, sxb, zb;
  const float* invs;

  // smem: the CTA's dynamic shared memory laid out by `plan`; rows_a: the
  // warp's first row in the stage (its second row is ROWS_B rows further).
  __device__ __forceinline__ B1Consumer(uint8_t* smem, const B1Plan& plan, int rows_a, int lane) {
    const int g = lane >> 2;
    t = lane & 3;
    xlane = 64 * g + 16 * t;
    // Q4_K: mma row g is weight row rg (and rg + rows_b) of the warp's: rows
    // 0,2,4,6 in the first half-warp, 1,3,5,7 in the second, so that the
    // 8-byte quant loads of a half-warp fall on 32 distinct banks (row pitch
    // 144 bytes).  The 4-byte loads of Q6_K, Q2_K and Q3_K (pitches 240, 112,
    // 144: rows 4 banks apart) are conflict-free as is.
    rg = kSubs == 16 ? g : 2 * (g & 3) + (g >> 2);
    // Q2_K / Q3_K: 2^24 times the power of two of run r = t's in-place field
    f23 = FMT == DQ_Q2_K ? 16777216.f / (float)(1 << (2 * t))
                         : 16777216.f / (float)(1 << (t == 3 ? 5 : 2 * t));
    lc = Q4KB1::lane_consts(g, t);
#pragma unroll
    for (int n = 0; n < 8; ++n) real6[n] = n == g ? 1u : 0u;
    wrow = smem_u32(smem + plan.off_w) + (rows_a + rg) * L::ROW_PITCH;
    xbase = smem_u32(smem + plan.off_x);
    sxb = smem_u32(smem + plan.off_sx);
    zb = smem_u32(smem + plan.off_z);
    invs = (const float*)(smem + plan.off_inv);
  }

  // The super-block with index sb (within its row) sitting in stage st; o
  // comes from order_after_wait() of the stage's full barrier.
  __device__ __forceinline__ void stage(int st, int64_t sb, uint32_t o, float2& a0,
                                        float2& a8) const {
    const float inv = SCALED ? invs[st] : 1.f;
    if constexpr (FMT == DQ_Q4_K) {
      Q4KB1::run(wrow + st * L::W_STAGE + o, pitch_b,
                 xbase + kStageX * st + xlane + o, zb,
                 sxb + 4 * kSubs * st + 8 * t + o, inv, lc, a0, a8);
    } else if constexpr (FMT == DQ_Q8_0) {
      const uint32_t ra = wrow + st * L::W_STAGE + o;   // 272-byte super-blocks: aligned
      Q80B1::run(ra, ra + pitch_b, xbase + kStageX * st + xlane + o, zb + 64, zb,
                 sxb + 4 * kSubs * st + 8 * t + o, inv, real6, t, a0, a8);
    } else if constexpr (FMT == DQ_Q2_K) {
      // 84-byte super-blocks: 4-byte aligned
      const uint32_t ra = wrow + st * L::W_STAGE + (int)((sb * L::SBB) & 15) + o;
      Q2KB1::run(ra, ra + pitch_b, xbase + kStageX * st + o, zb, sxb + 4 * kSubs * st + o, inv,
                 f23, real6, t, a0, a8);
    } else if constexpr (FMT == DQ_Q3_K) {
      // 110-byte super-blocks: 2-byte aligned, the offset uniform per stage
      const int delta = (int)((sb * L::SBB) & 15);
      const uint32_t ra = wrow + st * L::W_STAGE + delta + o;
      if (delta & 2)
        Q3KB1::run<true>(ra, ra + pitch_b, xbase + kStageX * st + o, zb,
                         sxb + 4 * kSubs * st + o, inv, f23, real6, t, a0, a8);
      else
        Q3KB1::run<false>(ra, ra + pitch_b, xbase + kStageX * st + o, zb,
                          sxb + 4 * kSubs * st + o, inv, f23, real6, t, a0, a8);
    } else {
      // the 210-byte super-block starts delta bytes into the 16-byte aligned box
      const int delta = (int)((sb * L::SBB) & 15);
      const uint32_t ra = wrow + st * L::W_STAGE + delta + o;
      if (delta & 2)
        Q6KB1::run<true>(ra, ra + pitch_b, xbase + kStageX * st + o, zb,
                         sxb + 4 * kSubs * st + o, inv, real6, t, a0, a8);
      else
        Q6KB1::run<false>(ra, ra + pitch_b, xbase + kStageX * st + o, zb,
                          sxb + 4 * kSubs * st + o, inv, real6, t, a0, a8);
    }
  }
};

// The quad's fixed-order sum: the four lanes of a quad hold sub-blocks 2t,
// 2t+1 (Q6_K: of both halves); after it every lane holds the rows' totals.
__device__ __forceinline__ void b1_quad_sum(float& acc0, float& acc8) {
  acc0 += __shfl_xor_sync(0xffffffffu, acc0, 1);
  acc8 += __shfl_xor_sync(0xffffffffu, acc8, 1);
  acc0 += __shfl_xor_sync(0xffffffffu, acc0, 2);
  acc8 += __shfl_xor_sync(0xffffffffu, acc8, 2);
}

}  // namespace dqmoe
