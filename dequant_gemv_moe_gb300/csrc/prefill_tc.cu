// prefill_tc.cu — the grouped expert GEMM for wide groups (prefill chunks:
// more than 32 tokens routed to one expert, e.g. the shared expert of a
// 256-token chunk), on the 5th-generation tensor core.
//
// One CTA computes D[128 rows][N <= 128 tokens] = W_tile . X^T for one
// 128-row tile of one expert matrix and one unit of <= 128 tokens:
//   * warp 0 (one lane) streams the packed super-blocks of the tile with 2-D
//     TMA (one box of 128 rows per super-block) and the tokens' fp16
//     activations as 64-wide K slabs (TMA, 128-byte swizzle, boxes of 32 rows);
//   * warps 1-8 (two threads per weight row, one per half slab) decode each
//     64-weight slab of their row to fp16 and store it straight into tensor
//     memory (tcgen05.st: row r is TMEM lane r, two fp16 per column), where
//     the MMA reads its A operand: no shared-memory round trip for the
//     decoded weights, whose store and re-read were the largest share of the
//     SM's shared-memory traffic;
//   * warp 9 allocates TMEM (A slab ring and accumulator) and one lane issues
//     tcgen05.mma (A from TMEM, B from shared memory; M=128, N=16..128,
//     K=16) per 16-wide K step; a tcgen05.commit per slab releases the slab;
//   * warps 1-8 then read the accumulator from TMEM (tcgen05.ld) and store
//     out[pos][row] = D * xinv[pos] (xinv undoes the activation scale).
// [KTransformers, §技术原理]: compute-dense work stays on the GPU; here the
// dense part is the prefill chunk's expert GEMM.
#include <algorithm>
#include <cstring>

#include "qgemv_mma.cuh"
#include "tc.cuh"
#include "tmap.h"

namespace dqmoe {

constexpr int kTcRows = 128;      // weight rows per tile (UMMA M)
constexpr int kTcMaxN = 128;      // tokens per unit (UMMA N <= 128 here)
constexpr int kTcWStages = 2;     // packed super-block ring depth
constexpr int kTcSlabs = 4;       // ring of decoded A slabs (TMEM) and activation slabs (smem)
constexpr int kTcDecWarps = 8;    // two threads per weight row: one per half slab
constexpr int kTcThreads = 32 * (kTcDecWarps + 2);   // producer, decoders, MMA
constexpr int kSlabB = kTcMaxN * 128;   // 16 KB: 128 tokens x 64 fp16
// TMEM columns: the A slabs (128 lanes x 64 fp16, two per 32-bit column: 32
// columns each) from column 0, then the fp32 accumulator (N <= 128 columns);
// 256 columns, two CTAs per SM
constexpr int kTmemA = 0;
constexpr int kTmemD = kTcSlabs * 32;
constexpr int kTmemCols = 256;
static_assert(kTmemD + kTcMaxN <= kTmemCols, "TMEM plan");

template <int FMT>
struct TcLayout {
  static constexpr int BOX = Layout<FMT>::BOX;               // bytes per row per super-block
  static constexpr int W_STG = kTcRows * BOX;                // multiple of 1024
  static constexpr int OFF_W = 1024;
  static constexpr int OFF_B = OFF_W + kTcWStages * W_STG;
  static constexpr int TOTAL = OFF_B + kTcSlabs * kSlabB;
  static_assert(W_STG % 1024 == 0, "TMA / swizzle atoms need 1024-byte alignment");
};

// ---------------------------------------------------------------------------
// decode one half of a 64-weight slab (q = 0..3 of the super-block) of one
// row: half h gives chunks 4h..4h+3 of 8 fp16 (weights 64q + 32h + [0, 32),
// natural k order)
// ---------------------------------------------------------------------------
template <int FMT>
struct SlabDecode;

template <>
struct SlabDecode<DQ_Q4_K> {
  // half 0: the low nibbles (sub-block 2q), half 1: the high nibbles (2q+1)
  __device__ __forceinline__ static void run(uint32_t rb, int q, int half, uint4 (&out)[4]) {
    const uint4 hd = lds_u128(rb);
    __half2 slo, olo, shi, ohi;
    SBDot<DQ_Q4_K>::scales_abs(hd, q, slo, olo, shi, ohi);
    const __half2 s = half ? shi : slo, o = half ? ohi : olo;
    const uint32_t mask = half ? 0x00F000F0u : 0x000F000Fu;
    const uint4 qa = lds_u128(rb + 16 + 32 * q), qb = lds_u128(rb + 32 + 32 * q);
    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const __half2 magic = u32_as_h2(0x64006400u);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t p0 = __byte_perm(w[2 * c], 0, 0x3120), p1 = __byte_perm(w[2 * c + 1], 0, 0x3120);
      const uint32_t src[4] = {p0, p0 >> 8, p1, p1 >> 8};
      uint32_t v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[i] = h2_as_u32(__hfma2(__hsub2(u32_as_h2(lop3_and_or(src[i], mask, 0x64006400u)), magic), s, o));
      out[c] = make_uint4(v[0], v[1], v[2], v[3]);
    }
  }
};

template <>
struct SlabDecode<DQ_Q6_K> {
  // half h: run r0 + h of the slab's two 32-weight runs
  __device__ __forceinline__ static void run(uint32_t rb, int q, int half, uint4 (&out)[4]) {
    const int h = q >> 1, r0 = 2 * (q & 1);
    const int r = r0 + half;
    const __half d = __ushort_as_half((unsigned short)lds_u16(rb + 208));
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int l0 = 8 * c;
      const int sidx = 8 * h + 2 * r + (l0 >> 4);
      const int sc = (int)(int8_t)(lds_u32_a2(rb + 192 + (sidx & ~1)) >> (8 * (sidx & 1)));
      const __half2 s2 = __half2half2(__hmul(d, __int2half_rn(sc)));
      uint32_t ch[4];
#pragma unroll
      for (int wv = 0; wv < 2; ++wv) {                 // 4 weights per word
        const uint32_t W = __byte_perm(lds_u32_a2(rb + 64 * h + 32 * half + l0 + 4 * wv), 0, 0x3120);
        const uint32_t H = __byte_perm(lds_u32_a2(rb + 128 + 32 * h + l0 + 4 * wv), 0, 0x3120);
        const uint32_t nlo = (r0 == 2) ? (W >> 4) : W;
        const uint32_t nhi = (r0 == 2) ? (W >> 12) : (W >> 8);
        const uint32_t hs = H >> 8;
        const uint32_t hlo = (r <= 2) ? (H << (4 - 2 * r)) : (H >> (2 * r - 4));
        const uint32_t hhi = (r <= 2) ? (hs << (4 - 2 * r)) : (hs >> (2 * r - 4));
        ch[2 * wv] = h2_as_u32(__hmul2(u32_as_h2(SBDot<DQ_Q6_K>::q6_pair(nlo, hlo)), s2));
        ch[2 * wv + 1] = h2_as_u32(__hmul2(u32_as_h2(SBDot<DQ_Q6_K>::q6_pair(nhi, hhi)), s2));
      }
      out[c] = make_uint4(ch[0], ch[1], ch[2], ch[3]);
    }
  }
};

template <>
struct SlabDecode<DQ_Q8_0> {
  // half h: block 2q + h
  __device__ __forceinline__ static void run(uint32_t rb, int q, int half, uint4 (&out)[4]) {
    const __half2 bias = __float2half2_rn(1152.f);   // 1024 + 128
    const uint32_t blk = rb + 34 * (2 * q + half);
    const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)lds_u16(blk)));
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t o = 2 + 8 * c;
      const uint32_t w0 = lds_u32_a2(blk + o) ^ 0x80808080u, w1 = lds_u32_a2(blk + o + 4) ^ 0x80808080u;
      const uint32_t v[4] = {__byte_perm(w0, 0x64646464u, 0x4140), __byte_perm(w0, 0x64646464u, 0x4342),
                             __byte_perm(w1, 0x64646464u, 0x4140), __byte_perm(w1, 0x64646464u, 0x4342)};
      uint32_t r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) r[i] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(v[i]), bias), d2));
      out[c] = make_uint4(r[0], r[1], r[2], r[3]);
    }
  }
};

// NVFP4: slab q = weights 64q..64q+63 = code bytes 32q..32q+31 of the codes
// and the scales of blocks 4q..4q+3 (half h: blocks 4q + 2h, 4q + 2h + 1);
// exact fp16 weights from the hardware conversions times the block scale.
template <>
struct SlabDecode<DQ_NVFP4> {
  __device__ __forceinline__ static void run(uint32_t rb, int q, int half, uint4 (&out)[4]) {
    const uint32_t sw = lds_u32(rb + 4 * q);
    const __half2 s01 = u32_as_h2(e4m3x2_to_h2((uint16_t)(half ? (sw >> 16) : (sw & 0xFFFF))));
    const __half2 sc[2] = {__low2half2(s01), __high2half2(s01)};
    const uint4 a = lds_u128(rb + 16 + 32 * q + 16 * half);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {                     // weights 64q+32h+8c..+7: block 4q + 2h + c/2
      uint32_t h[4];
      e2m1x8_to_h2x4(w[c], h);
      uint32_t r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) r[i] = h2_as_u32(__hmul2(u32_as_h2(h[i]), sc[c >> 1]));
      out[c] = make_uint4(r[0], r[1], r[2], r[3]);
    }
  }
};

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
struct TcParams {
  CUtensorMap wmap;     // routed experts stacked [E*rows][row_bytes/2], box BOX x 128 rows
  CUtensorMap wmap_sh;  // shared experts stacked
  CUtensorMap xmap;     // activations fp16 [positions][K], box 64 x 32 rows, 128B swizzle
  int rows_per_expert;
  int E;
  int nsb;              // super-blocks along K
  const int4* units;    // (matrix id, first position, tokens <= 128, -)
  const int* n_units;
  const float* xinv;    // per position: 1 / activation scale
  float* out;           // out[pos][row]
  int64_t out_stride;
};

template <int FMT>
__global__ void __launch_bounds__(kTcThreads, 2) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  using TL = TcLayout<FMT>;
  const int unit = blockIdx.y;
  if (unit >= __ldg(p.n_units)) return;            // uniform for the whole CTA
  // swizzle atoms and TMA boxes need a 1024-byte aligned window
  if (smem_u32(smem) & 1023) {
    if (threadIdx.x == 0) report_timeout();
    return;
  }
  const int4 u = __ldg(p.units + unit);
  const bool shared = u.x >= p.E;
  const int mat = shared ? u.x - p.E : u.x;
  const int row0 = blockIdx.x * kTcRows;
  const int grow = mat * p.rows_per_expert + row0;
  const int pos0 = u.y, ncols = u.z;
  const int npad = (ncols + 15) & ~15;
  const int nbox = (ncols + 31) >> 5;
  const int nslab = p.nsb * 4;

  uint64_t* wfull = (uint64_t*)smem;
  uint64_t* wempty = wfull + kTcWStages;
  uint64_t* sfull = wempty + kTcWStages;   // A slab in TMEM and activation slab landed
  uint64_t* sempty = sfull + kTcSlabs;     // the slab's MMAs completed
  uint64_t* accfull = sempty + kTcSlabs;
  uint32_t* tmem_slot = (uint32_t*)(accfull + 1);
  uint8_t* wbuf = smem + TL::OFF_W;
  uint8_t* bbuf = smem + TL::OFF_B;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kMmaWarp = kTcDecWarps + 1;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcWStages; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], kTcDecWarps);
    }
    for (int i = 0; i < kTcSlabs; ++i) {
      mbar_init(&sfull[i], 1 + 32 * kTcDecWarps);   // producer's expect_tx arrival + decoders
      mbar_init(&sempty[i], 1);                     // tcgen05.commit
    }
    mbar_init(accfull, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const CUtensorMap* wm = shared ? &p.wmap_sh : &p.wmap;
      bool ok = true;
      for (int sb = 0; sb < p.nsb && ok; ++sb) {
        const int ws = sb % kTcWStages, wr = sb / kTcWStages;
        if (wr > 0) ok = mbar_wait(&wempty[ws], (wr - 1) & 1);
        if (!ok) break;
        const int64_t a = ((int64_t)sb * Layout<FMT>::SBB) & ~(int64_t)15;
        mbar_arrive_expect_tx(&wfull[ws], TL::W_STG);
        tma_load_2d(wbuf + ws * TL::W_STG, wm, (int)(a >> 1), grow, &wfull[ws], pol);
        for (int q = 0; q < 4 && ok; ++q) {
          const int sl = sb * 4 + q, ss = sl % kTcSlabs, sr = sl / kTcSlabs;
          if (sr > 0) ok = mbar_wait(&sempty[ss], (sr - 1) & 1);
          if (!ok) break;
          mbar_arrive_expect_tx(&sfull[ss], nbox * 32 * 128);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(bbuf + ss * kSlabB + b * 4096, &p.xmap, sl * 64, pos0 + 32 * b, &sfull[ss],
                        pol);
        }
      }
    }
  } else if (warp <= kTcDecWarps) {
    // ---------------------- decoders, then epilogue ----------------------
    // row r of the tile is TMEM lane r; warp w may access lanes 32*(w%4)..;
    // warps 1-4 decode the first half of every slab (TMEM columns 0-15 of
    // the slab), warps 5-8 the second (columns 16-31)
    const int r = 32 * (warp & 3) + lane;
    const int half = (warp - 1) >> 2;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    bool ok = true;
    for (int sb = 0; sb < p.nsb; ++sb) {
      const int ws = sb % kTcWStages;
      ok = ok && mbar_wait(&wfull[ws], (sb / kTcWStages) & 1);
      const uint32_t rb = smem_u32(wbuf + ws * TL::W_STG) + r * TL::BOX +
                          (uint32_t)(((int64_t)sb * Layout<FMT>::SBB) & 15);
      for (int q = 0; q < 4; ++q) {
        const int sl = sb * 4 + q, ss = sl % kTcSlabs, sr = sl / kTcSlabs;
        if (sr > 0) ok = ok && mbar_wait(&sempty[ss], (sr - 1) & 1);
        // tcgen05.st is warp-collective: decide for the whole warp
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc_fence_after();    // the slab's previous MMAs completed before these stores
          uint4 ch[4];
          SlabDecode<FMT>::run(rb, q, half, ch);
          tmem_st16(tmem + lane_base + (uint32_t)(kTmemA + 32 * ss + 16 * half), ch);
          tc_fence_before();   // ... and are ordered before the MMA thread's wait
        }
        mbar_arrive(&sfull[ss]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty[ws]);
    }
    // epilogue: out[pos0 + n][row0 + r] = D[r][n] * xinv[pos0 + n]; the two
    // warps of a lane quarter take half of the columns each
    ok = ok && mbar_wait(accfull, 0);
    tc_fence_after();
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      const int cend = half ? npad : npad / 2;
      for (int c0 = half ? npad / 2 : 0; c0 < cend; c0 += 8) {
        float v[8];
        tmem_ld8(tmem + lane_base + (uint32_t)(kTmemD + c0), v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int n = c0 + i;
          if (n < ncols) {
            const int pos = pos0 + n;
            p.out[(int64_t)pos * p.out_stride + row0 + r] = v[i] * __ldg(p.xinv + pos);
          }
        }
      }
    }
  } else {
    // -------------------------------- MMA --------------------------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(kTcRows, npad);
      bool ok = true;
      for (int sl = 0; sl < nslab && ok; ++sl) {
        const int ss = sl % kTcSlabs;
        ok = mbar_wait(&sfull[ss], (sl / kTcSlabs) & 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t at = tmem + (uint32_t)(kTmemA + 32 * ss);
        const uint64_t bd = sw128_kmajor_desc(smem_u32(bbuf + ss * kSlabB));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)   // K = 16 per instruction: 8 TMEM columns, +32 B in the atom
          tc_mma_f16_tmem_a(tmem + kTmemD, at + 8 * kk, bd + 2 * kk, idesc, (sl | kk) ? 1u : 0u);
        tc_commit(&sempty[ss]);
      }
      tc_commit(accfull);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
template <int FMT>
int launch_tc_fmt(const void* W, const void* Wsh, int E, int n_shared, int rows_per_expert,
                  int K, const int4* units, const int* n_units, int max_units, const __half* X16,
                  int64_t npos, const float* xinv, float* out, int64_t out_stride,
                  cudaStream_t s) {
  using TL = TcLayout<FMT>;
  TcParams p;
  memset(&p, 0, sizeof(p));
  const int qk = FMT == DQ_Q8_0 ? 32 : 256;
  const int bb = Layout<FMT>::SBB * qk / 256;   // bytes per quantisation block
  const uint64_t row_bytes = (uint64_t)(K / qk) * bb;
  if (!make_weight_tmap(&p.wmap, W, (uint64_t)rows_per_expert * E, row_bytes, TL::BOX, kTcRows))
    return DQ_ERR_CUDA;
  if (n_shared > 0 &&
      !make_weight_tmap(&p.wmap_sh, Wsh, (uint64_t)rows_per_expert * n_shared, row_bytes, TL::BOX,
                        kTcRows))
    return DQ_ERR_CUDA;
  if (!make_act_tmap_sw128(&p.xmap, X16, (uint64_t)npos, (uint64_t)K)) return DQ_ERR_CUDA;
  p.rows_per_expert = rows_per_expert;
  p.E = E;
  p.nsb = K / 256;
  p.units = units;
  p.n_units = n_units;
  p.xinv = xinv;
  p.out = out;
  p.out_stride = out_stride;
  static bool attr[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr[dev]) {
    if (cudaFuncSetAttribute(tc_gemm_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TL::TOTAL) != cudaSuccess)
      return DQ_ERR_CUDA;
    if (dev < 64) attr[dev] = true;
  }
  dim3 grid((unsigned)(rows_per_expert / kTcRows), (unsigned)std::max(1, max_units));
  if (launch_pdl(tc_gemm_kernel<FMT>, grid, dim3(kTcThreads), TL::TOTAL, s, 0, p) != cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

int launch_tc_gemm(int fmt, const void* W, const void* Wsh, int E, int n_shared,
                   int rows_per_expert, int K, const int4* units, const int* n_units,
                   int max_units, const __half* X16, int64_t npos, const float* xinv, float* out,
                   int64_t out_stride, cudaStream_t s) {
  if (rows_per_expert % kTcRows) return DQ_ERR_UNSUPPORTED;
#define DQ_TC(F)                                                                          \
  if (fmt == F)                                                                           \
    return launch_tc_fmt<F>(W, Wsh, E, n_shared, rows_per_expert, K, units, n_units,      \
                            max_units, X16, npos, xinv, out, out_stride, s);
  DQ_TC(DQ_Q4_K)
  DQ_TC(DQ_Q6_K)
  DQ_TC(DQ_Q8_0)
  DQ_TC(DQ_NVFP4)
#undef DQ_TC
  return DQ_ERR_UNSUPPORTED;
}

}  // namespace dqmoe
