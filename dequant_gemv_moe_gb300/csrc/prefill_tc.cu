// prefill_tc.cu — the grouped expert GEMM for wide groups (prefill chunks:
// more than 32 tokens routed to one expert, e.g. the shared expert of a
// 256-token chunk), on the 5th-generation tensor core.
//
// One CTA computes D[128 rows][N <= 128 tokens] = W_tile . X^T for one
// 128-row tile of one expert matrix and one unit of <= 128 tokens:
//   * warp 0 (one lane) streams the packed super-blocks of the tile with 2-D
//     TMA (one box of 128 rows per super-block) and the tokens' fp16
//     activations as 64-wide K slabs (TMA, 128-byte swizzle, boxes of 32 rows);
//   * warps 1-4 (one thread per weight row) decode each 64-weight slab of
//     their row to fp16 and store it in the 128-byte-swizzled K-major layout
//     the tensor core reads (the same layout TMA writes for the activations);
//   * warp 5 allocates the TMEM accumulator and one lane issues
//     tcgen05.mma (M=128, N=16..128, K=16) per 16-wide K step; a
//     tcgen05.commit per slab releases the slab's buffers;
//   * warps 1-4 then read the accumulator from TMEM (tcgen05.ld) and store
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
// Slab ring depth (a kernel parameter, SLABS): two slabs keep the shared
// memory at ~103 KB (Q4_K / NVFP4 rows), so that two CTAs share an SM and
// their decoder warps hide each other's latency.  Calls whose routed experts
// are expected above the 32-token threshold (prefill chunks: many units) take
// two (DeepSeek-V3 expert shapes, 32 experts of ~64 tokens, Q4_K: 0.81 ->
// 0.68 ms against four); calls where only the shared experts reach this
// kernel (a few units of 16 row tiles each, fewer CTAs than SMs) keep four:
// a deeper ring per CTA.
constexpr int kTcWStages = 2;     // packed super-block ring depth
constexpr int kTcThreads = 192;   // 6 warps
constexpr int kSlabA = kTcRows * 128;   // 16 KB: 128 rows x 64 fp16
constexpr int kSlabB = kTcMaxN * 128;   // 16 KB: 128 tokens x 64 fp16

template <int FMT, int SLABS>
struct TcLayout {
  static constexpr int BOX = Layout<FMT>::BOX;               // bytes per row per super-block
  static constexpr int W_STG = kTcRows * BOX;                // multiple of 1024
  static constexpr int OFF_W = 1024;
  static constexpr int OFF_A = OFF_W + kTcWStages * W_STG;
  static constexpr int OFF_B = OFF_A + SLABS * kSlabA;
  static constexpr int TOTAL = OFF_B + SLABS * kSlabB;
  static_assert(W_STG % 1024 == 0, "TMA / swizzle atoms need 1024-byte alignment");
};

// ---------------------------------------------------------------------------
// decode one 64-weight slab (q = 0..3 of the super-block) of one row into 8
// chunks of 8 fp16 (natural k order)
// ---------------------------------------------------------------------------
template <int FMT>
struct SlabDecode;

template <>
struct SlabDecode<DQ_Q4_K> {
  __device__ __forceinline__ static void run(uint32_t rb, int q, uint4 (&out)[8]) {
    const uint4 hd = lds_u128(rb);
    __half2 slo, olo, shi, ohi;
    SBDot<DQ_Q4_K>::scales_abs(hd, q, slo, olo, shi, ohi);   // sub-blocks 2q (low), 2q+1 (high)
    const uint4 qa = lds_u128(rb + 16 + 32 * q), qb = lds_u128(rb + 32 + 32 * q);
    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const __half2 magic = u32_as_h2(0x64006400u);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t p0 = __byte_perm(w[2 * c], 0, 0x3120), p1 = __byte_perm(w[2 * c + 1], 0, 0x3120);
      const uint32_t src[4] = {p0, p0 >> 8, p1, p1 >> 8};
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        lo[i] = h2_as_u32(__hfma2(__hsub2(u32_as_h2(lop3_and_or(src[i], 0x000F000Fu, 0x64006400u)), magic), slo, olo));
        hi[i] = h2_as_u32(__hfma2(__hsub2(u32_as_h2(lop3_and_or(src[i], 0x00F000F0u, 0x64006400u)), magic), shi, ohi));
      }
      out[c] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      out[c + 4] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    }
  }
};

template <>
struct SlabDecode<DQ_Q6_K> {
  __device__ __forceinline__ static void run(uint32_t rb, int q, uint4 (&out)[8]) {
    const int h = q >> 1, r0 = 2 * (q & 1);
    const __half d = __ushort_as_half((unsigned short)lds_u16(rb + 208));
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int l0 = 8 * c;
      uint32_t ch[2][4];
#pragma unroll
      for (int part = 0; part < 2; ++part) {          // part 0: run r0, part 1: run r0 + 1
        const int r = r0 + part;
        const int sidx = 8 * h + 2 * r + (l0 >> 4);
        const int sc = (int)(int8_t)(lds_u32_a2(rb + 192 + (sidx & ~1)) >> (8 * (sidx & 1)));
        const __half2 s2 = __half2half2(__hmul(d, __int2half_rn(sc)));
#pragma unroll
        for (int wv = 0; wv < 2; ++wv) {               // 4 weights per word
          const uint32_t W = __byte_perm(lds_u32_a2(rb + 64 * h + 32 * part + l0 + 4 * wv), 0, 0x3120);
          const uint32_t H = __byte_perm(lds_u32_a2(rb + 128 + 32 * h + l0 + 4 * wv), 0, 0x3120);
          const uint32_t nlo = (r0 == 2) ? (W >> 4) : W;
          const uint32_t nhi = (r0 == 2) ? (W >> 12) : (W >> 8);
          const uint32_t hs = H >> 8;
          const uint32_t hlo = (r <= 2) ? (H << (4 - 2 * r)) : (H >> (2 * r - 4));
          const uint32_t hhi = (r <= 2) ? (hs << (4 - 2 * r)) : (hs >> (2 * r - 4));
          ch[part][2 * wv] = h2_as_u32(__hmul2(u32_as_h2(SBDot<DQ_Q6_K>::q6_pair(nlo, hlo)), s2));
          ch[part][2 * wv + 1] = h2_as_u32(__hmul2(u32_as_h2(SBDot<DQ_Q6_K>::q6_pair(nhi, hhi)), s2));
        }
      }
      out[c] = make_uint4(ch[0][0], ch[0][1], ch[0][2], ch[0][3]);
      out[c + 4] = make_uint4(ch[1][0], ch[1][1], ch[1][2], ch[1][3]);
    }
  }
};

template <>
struct SlabDecode<DQ_Q8_0> {
  __device__ __forceinline__ static void run(uint32_t rb, int q, uint4 (&out)[8]) {
    const __half2 bias = __float2half2_rn(1152.f);   // 1024 + 128
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t blk = rb + 34 * (2 * q + (c >> 2));
      const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)lds_u16(blk)));
      const uint32_t o = 2 + 8 * (c & 3);
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
// and the scales of blocks 4q..4q+3; exact fp16 weights from the hardware
// conversions times the block scale.
template <>
struct SlabDecode<DQ_NVFP4> {
  __device__ __forceinline__ static void run(uint32_t rb, int q, uint4 (&out)[8]) {
    const uint32_t sw = lds_u32(rb + 4 * q);
    const __half2 s01 = u32_as_h2(e4m3x2_to_h2((uint16_t)(sw & 0xFFFF)));
    const __half2 s23 = u32_as_h2(e4m3x2_to_h2((uint16_t)(sw >> 16)));
    const __half2 sc[4] = {__low2half2(s01), __high2half2(s01), __low2half2(s23),
                           __high2half2(s23)};
    const uint4 a = lds_u128(rb + 16 + 32 * q), b = lds_u128(rb + 32 + 32 * q);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) {                     // weights 64q+8c..+7: block 4q + c/2
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

template <int FMT, int SLABS>
__global__ void __launch_bounds__(kTcThreads, SLABS == 2 ? 2 : 1)
    tc_gemm_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  using TL = TcLayout<FMT, SLABS>;
  constexpr int kTcSlabs = SLABS;
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
  uint64_t* sfull = wempty + kTcWStages;
  uint64_t* sempty = sfull + kTcSlabs;
  uint64_t* accfull = sempty + kTcSlabs;
  uint32_t* tmem_slot = (uint32_t*)(accfull + 1);
  uint8_t* wbuf = smem + TL::OFF_W;
  uint8_t* abuf = smem + TL::OFF_A;
  uint8_t* bbuf = smem + TL::OFF_B;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcWStages; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], 4);
    }
    for (int i = 0; i < kTcSlabs; ++i) {
      mbar_init(&sfull[i], 1 + kTcRows);   // producer's expect_tx arrival + 128 decoders
      mbar_init(&sempty[i], 1);            // tcgen05.commit
    }
    mbar_init(accfull, 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, kTcMaxN);
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
  } else if (warp <= 4) {
    // ---------------------- decoders, then epilogue ----------------------
    // row r of the tile is TMEM lane r; warp w may read lanes 32*(w%4)..
    const int r = 32 * (warp & 3) + lane;
    bool ok = true;
    for (int sb = 0; sb < p.nsb; ++sb) {
      const int ws = sb % kTcWStages;
      ok = ok && mbar_wait(&wfull[ws], (sb / kTcWStages) & 1);
      const uint32_t rb = smem_u32(wbuf + ws * TL::W_STG) + r * TL::BOX +
                          (uint32_t)(((int64_t)sb * Layout<FMT>::SBB) & 15);
      for (int q = 0; q < 4; ++q) {
        const int sl = sb * 4 + q, ss = sl % kTcSlabs, sr = sl / kTcSlabs;
        if (sr > 0) ok = ok && mbar_wait(&sempty[ss], (sr - 1) & 1);
        if (ok) {
          uint4 ch[8];
          SlabDecode<FMT>::run(rb, q, ch);
          uint8_t* at = abuf + ss * kSlabA;
#pragma unroll
          for (int c = 0; c < 8; ++c) *(uint4*)(at + sw128_offset(r, c)) = ch[c];
          fence_proxy_async_smem();
        }
        mbar_arrive(&sfull[ss]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty[ws]);
    }
    // epilogue: out[pos0 + n][row0 + r] = D[r][n] * xinv[pos0 + n]
    ok = ok && mbar_wait(accfull, 0);
    tc_fence_after();
    // tcgen05.ld is warp-collective: decide for the whole warp
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
      for (int c0 = 0; c0 < npad; c0 += 8) {
        float v[8];
        tmem_ld8(tmem + lane_base + (uint32_t)c0, v);
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
        const uint64_t ad = sw128_kmajor_desc(smem_u32(abuf + ss * kSlabA));
        const uint64_t bd = sw128_kmajor_desc(smem_u32(bbuf + ss * kSlabB));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)   // K = 16 per instruction: +32 bytes in the atom
          tc_mma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (sl | kk) ? 1u : 0u);
        tc_commit(&sempty[ss]);
      }
      tc_commit(accfull);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcMaxN);
  }
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------
template <int FMT, int SLABS>
int launch_tc_fmt(const void* W, const void* Wsh, int E, int n_shared, int rows_per_expert,
                  int K, const int4* units, const int* n_units, int max_units, const __half* X16,
                  int64_t npos, const float* xinv, float* out, int64_t out_stride,
                  cudaStream_t s) {
  using TL = TcLayout<FMT, SLABS>;
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
    if (cudaFuncSetAttribute(tc_gemm_kernel<FMT, SLABS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, TL::TOTAL) != cudaSuccess)
      return DQ_ERR_CUDA;
    if (dev < 64) attr[dev] = true;
  }
  dim3 grid((unsigned)(rows_per_expert / kTcRows), (unsigned)std::max(1, max_units));
  if (launch_pdl(tc_gemm_kernel<FMT, SLABS>, grid, dim3(kTcThreads), TL::TOTAL, s, 0, p) !=
      cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

// many_units: routed experts are expected above the 32-token threshold (two
// slabs, two CTAs per SM); otherwise four slabs, one CTA per SM.
int launch_tc_gemm(int fmt, const void* W, const void* Wsh, int E, int n_shared,
                   int rows_per_expert, int K, const int4* units, const int* n_units,
                   int max_units, const __half* X16, int64_t npos, const float* xinv, float* out,
                   int64_t out_stride, bool many_units, cudaStream_t s) {
  if (rows_per_expert % kTcRows) return DQ_ERR_UNSUPPORTED;
  const bool deep = !many_units;
#define DQ_TC(F)                                                                               \
  if (fmt == F)                                                                                \
    return deep ? launch_tc_fmt<F, 4>(W, Wsh, E, n_shared, rows_per_expert, K, units, n_units, \
                                      max_units, X16, npos, xinv, out, out_stride, s)          \
                : launch_tc_fmt<F, 2>(W, Wsh, E, n_shared, rows_per_expert, K, units, n_units, \
                                      max_units, X16, npos, xinv, out, out_stride, s);
  DQ_TC(DQ_Q4_K)
  DQ_TC(DQ_Q6_K)
  DQ_TC(DQ_Q8_0)
  DQ_TC(DQ_NVFP4)
#undef DQ_TC
  return DQ_ERR_UNSUPPORTED;
}

}  // namespace dqmoe
