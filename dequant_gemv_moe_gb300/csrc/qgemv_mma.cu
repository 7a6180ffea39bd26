// qgemv_mma.cu — dq_qgemv for 16-bit activations (and the scaled path for
// bf16): the streaming GEMV of qgemv_mma.cuh over a grid of 64-row tiles,
// optionally split along K over a thread-block cluster whose partial sums are
// reduced through distributed shared memory (split-K for small N, without a
// second pass and without scratch memory).
#include <algorithm>

#include "b1.cuh"
#include "qgemv_mma.cuh"
#include "tmap.h"

namespace dqmoe {

// stages of a CTA's weights prefetched into L2 before the wait when its K
// range exceeds its ring (see early_weights)
constexpr int kL2PrefetchStages = 2;

struct GemvParams {
  CUtensorMap tmap;  // W as [N rows][row_bytes/2] 16-bit elements, box BOX x 64 rows
  const uint8_t* W;
  int64_t row_bytes;
  int N;
  int nsb;          // super-blocks (256 weights) per row
  XSrc x;           // [batch][K]
  int batch;
  float* y;         // [batch][N]
  int nstage;
  int w_early;      // 1: issue the first stages' weight copies before pdl_wait
};

// bf16 activations of one stage for up to 8 columns: this loader lane's 8
// values of each column (16 bytes) into registers.
__device__ __forceinline__ void bf16_stage_load(const XSrc& xs, int ncols, int64_t k0, int lane,
                                                uint4 (&r)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < ncols)
      r[j] = __ldg((const uint4*)((const uint16_t*)xs.base + (int64_t)j * xs.col_stride + k0) +
                   lane);
}

// ... converted to fp16 with one power-of-two scale per column (as stage_x
// does for bf16: the same values and scales) and stored; arrives on `full`
// like stage_x (two arrivals per lane).
template <int FMT>
__device__ __forceinline__ void bf16_stage_store(const uint4 (&r)[8], int ncols, uint8_t* xdst,
                                                 float* xinv, int lane, uint64_t* full) {
  float amax[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    amax[j] = 0.f;
    if (j < ncols) {
      const uint32_t w[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax[j] = fmaxf(amax[j], fabsf(__uint_as_float(w[i] << 16)));
        amax[j] = fmaxf(amax[j], fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int j = 0; j < 8; ++j) amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], o));
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < ncols) {
      float sc, inv;
      pow2_scale(amax[j], sc, inv);
      const uint32_t w[4] = {r[j].x, r[j].y, r[j].z, r[j].w};
      uint32_t h[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        h[i] = h2_as_u32(__floats2half2_rn(__uint_as_float(w[i] << 16) * sc,
                                           __uint_as_float(w[i] & 0xFFFF0000u) * sc));
      *(uint4*)(xdst + j * Layout<FMT>::XCOL + 2 * xoff(8 * lane)) =
          make_uint4(h[0], h[1], h[2], h[3]);
      if (lane == 0) xinv[j] = inv;
    }
  }
  cp_async_arrive_noinc(full);
  mbar_arrive(full);
}

// PAIR: each consumer iteration takes two stages (more independent work per
// warp and more registers: for grids of at most three CTAs per SM).
// BF16X: bf16 activations at batch >= 4 (Q4_K and Q6_K: >= 2), whose next
// stage the loader holds in registers while it converts the current one (its
// global load latency hidden behind a stage); a separate instance, so that the
// extra registers stay out of the fp16 kernels.  Capped at four CTAs per SM
// (96 registers) except for Q6_K, whose decode measured faster uncapped at
// three.  Measured on the 70B shapes (gate / down / q, us): batch 8 Q4_K
// 103.5 / 99.5 / 29.8 -> 56.0 / 54.4 / 18.2, Q6_K 104.7 / 135.6 / 41.1 -> 64.7 /
// 76.4 / 24.8, Q8_0 107.7 / 126.9 / 40.2 -> 63.3 / 74.0 / 24.4; batch 2 Q4_K
// 47.4 / 50.9 / 17.0 -> 46.8 / 45.2 / 16.1, Q6_K 64.1 / 80.5 / 25.7 -> 55.6 /
// 66.0 / 21.8, Q8_0 slower (61.7 -> 74.3 us on down).
template <int FMT, bool PAIR, bool BF16X>
__global__ void __launch_bounds__(kThreads, PAIR ? 3 : ((BF16X && FMT != DQ_Q6_K) ? 4 : 1))
    qgemv_mma_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using L = Layout<FMT>;
  const int ksplit = (int)cluster_nctarank();
  const int rank = (int)cluster_ctarank();
  const SmemPlan plan = make_plan<FMT>(p.nstage, p.batch, ksplit);
  uint64_t* full = (uint64_t*)(smem + plan.off_bar);
  uint64_t* empty = full + plan.nstage;
  uint64_t* red_full = empty + plan.nstage;
  uint8_t* wbuf = smem + plan.off_w;
  uint8_t* xbuf = smem + plan.off_x;
  float* xinv = (float*)(smem + plan.off_xinv);
  float* red = (float*)(smem + plan.off_red);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.y;
  const int row0 = tile * kTileRows;

  // this CTA's super-block range [sb0, sb1)
  const int sb0 = (int)((int64_t)p.nsb * rank / ksplit);
  const int sb1 = (int)((int64_t)p.nsb * (rank + 1) / ksplit);
  const int nchunk = sb1 - sb0;   // one super-block per stage

  if (threadIdx.x == 0) {
    for (int s = 0; s < plan.nstage; ++s) {
      mbar_init(&full[s], full_arrivals(p.x.dtype));
      mbar_init(&empty[s], kConsumerWarps);    // one per consumer warp
    }
    if (ksplit > 1) mbar_init(red_full, (ksplit - 1) * kConsumerWarps * 32);
    fence_barrier_init();
  }
  init_xinv(xinv, plan.nstage * 8, p.x.dtype);
  if (ksplit > 1) cluster_sync_all();
  else __syncthreads();

  pdl_trigger();

  if (warp == 0) {
    // ------------------------------ loader ------------------------------
    const uint64_t pol = l2_evict_first_policy();
    if (lane == 0) prefetch_tmap(&p.tmap);
    // weights are read-only inputs: with w_early their first stages stream in
    // while the previous kernel in the stream finishes
    const int early = p.w_early == 1 ? min(plan.nstage, nchunk) : 0;
    if (lane == 0) {
      for (int c = 0; c < early; ++c) {
        const int64_t a = ((int64_t)(sb0 + c) * L::SBB) & ~(int64_t)15;
        mbar_arrive_expect_tx(&full[c], L::W_STAGE);
        tma_load_2d(wbuf + c * L::W_STAGE, &p.tmap, (int)(a >> 1), row0, &full[c], pol);
      }
      // the range exceeds the ring: only its first stages, into L2
      if (p.w_early == 2)
        for (int c = 0; c < min(nchunk, kL2PrefetchStages); ++c)
          tma_prefetch_l2_2d(&p.tmap, (int)((((int64_t)(sb0 + c) * L::SBB) & ~(int64_t)15) >> 1),
                             row0);
    }
    pdl_wait();
    bool ok = true;
    int s = 0;
    uint32_t ph = 0;            // phase parity of stage s in the current round
    uint4 nxt[8];               // BF16X: the next stage's raw activations
    if (BF16X && nchunk > 0) bf16_stage_load(p.x, p.batch, (int64_t)sb0 * 256, lane, nxt);
    for (int c = 0; c < nchunk && ok; ++c) {
      if (c >= plan.nstage) ok = mbar_wait(&empty[s], ph ^ 1);
      if (!ok) break;
      const int c0 = sb0 + c;
      // box start: the super-block's first byte rounded down to 16 bytes
      // (Q6_K blocks are 210 bytes; row starts are 16-byte aligned)
      const int64_t a = ((int64_t)c0 * L::SBB) & ~(int64_t)15;
      if (lane == 0 && c >= early) {
        mbar_arrive_expect_tx(&full[s], L::W_STAGE);   // rows past N are zero-filled, still counted
        tma_load_2d(wbuf + s * L::W_STAGE, &p.tmap, (int)(a >> 1), row0, &full[s], pol);
      }
      if constexpr (BF16X) {
        uint4 cur[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
        if (c + 1 < nchunk) bf16_stage_load(p.x, p.batch, (int64_t)(c0 + 1) * 256, lane, nxt);
        bf16_stage_store<FMT>(cur, p.batch, xbuf + s * p.batch * L::XCOL, xinv + s * 8, lane,
                              &full[s]);
      } else {
        stage_x<FMT>(p.x, p.batch, (int64_t)c0 * 256, 1, xbuf + s * p.batch * L::XCOL,
                     xinv + s * 8, lane, &full[s]);
      }
      if (++s == plan.nstage) {
        s = 0;
        ph ^= 1;
      }
    }
  } else {
    // ----------------------------- consumers -----------------------------
    pdl_wait();
    const int cw = warp - 1;
    const int g = lane >> 2, t = lane & 3;
    const int xc = g < p.batch ? g : 0;      // this lane's activation column
    const bool f16 = p.x.dtype == DQ_F16;    // fp16 input carries no scale
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float accs[1][2][4] = {};               // fp16 input: one running accumulator pair
    const uint32_t wrow = smem_u32(wbuf) + (16 * cw + g) * L::ROW_PITCH;
    const uint32_t xcol0 = smem_u32(xbuf) + xc * L::XCOL;
    bool ok = true;
    int s = 0;
    uint32_t ph = 0;
    // super-block c of this CTA from stage st into (acc_, accs_)
    auto compute = [&](int st, int c, uint32_t o, float (&acc_)[4], float (&accs_)[1][2][4]) {
      const int c0 = sb0 + c;
      const uint32_t wst = wrow + st * L::W_STAGE + (uint32_t)(((int64_t)c0 * L::SBB) & 15) + o;
      const uint32_t xcol[1] = {xcol0 + st * p.batch * L::XCOL + o};
      if constexpr (SBDot<FMT>::kRowScale) {
        float d[1][2][4] = {};
        float r0, r8;
        SBDot<FMT>::template run<1>(wst, 8 * L::ROW_PITCH, xcol, 0, t, d, r0, r8);
        const float c0s = f16 ? 1.f : xinv[st * 8 + ((2 * t) & 7)];
        const float c1s = f16 ? 1.f : xinv[st * 8 + ((2 * t + 1) & 7)];
        fold_tile(acc_, d[0], r0, r8, c0s, c1s);
      } else if (f16) {
        SBDot<FMT>::template run<1>(wst, 8 * L::ROW_PITCH, xcol, 0, t, accs_);
      } else {
        float pt[1][2][4] = {};
        SBDot<FMT>::template run<1>(wst, 8 * L::ROW_PITCH, xcol, 0, t, pt);
        const float inv0 = xinv[st * 8 + ((2 * t) & 7)], inv1 = xinv[st * 8 + ((2 * t + 1) & 7)];
        fold_tile(acc_, pt[0], 1.f, 1.f, inv0, inv1);
      }
    };
    auto advance = [&]() {
      if (++s == plan.nstage) {
        s = 0;
        ph ^= 1;
      }
    };
    float accB[4] = {0.f, 0.f, 0.f, 0.f};
    float accsB[1][2][4] = {};
    int c = 0;
    for (; PAIR && c + 1 < nchunk; c += 2) {
      const int s0 = s;
      const uint32_t p0 = ph;
      advance();
      const int s1 = s;
      const uint32_t p1 = ph;
      advance();
      ok = ok && mbar_wait(&full[s0], p0) && mbar_wait(&full[s1], p1);
      if (!ok) continue;   // after a timed-out wait: walk on without waits or reads
      const uint32_t o = order_after_wait(0u);   // stage reads follow the waits
      compute(s0, c, o, acc, accs);
      compute(s1, c + 1, o, accB, accsB);
      keep_before_release<4>(acc);              // ... and finish before their release
      keep_before_release<8>(&accs[0][0][0]);
      keep_before_release<4>(accB);
      keep_before_release<8>(&accsB[0][0][0]);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_relaxed(&empty[s0]);
        mbar_arrive_relaxed(&empty[s1]);
      }
    }
    for (; c < nchunk; ++c) {
      const int s0 = s;
      const uint32_t p0 = ph;
      advance();
      ok = ok && mbar_wait(&full[s0], p0);
      if (!ok) continue;
      const uint32_t o = order_after_wait(0u);
      compute(s0, c, o, acc, accs);
      keep_before_release<4>(acc);
      keep_before_release<8>(&accs[0][0][0]);
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&empty[s0]);
    }
    for (int i = 0; i < 4; ++i) {
      acc[i] += accB[i];
      accs[0][0][i] += accsB[0][0][i];
      accs[0][1][i] += accsB[0][1][i];
    }
    if (!SBDot<FMT>::kRowScale && f16)
      for (int i = 0; i < 4; ++i) acc[i] = accs[0][0][i] + accs[0][1][i];

    // ------------------------ split-K reduction -------------------------
    if (ksplit > 1) {
      if (rank != 0) {
        float* slot = red + (((rank - 1) * kConsumerWarps + cw) * 32 + lane) * 4;
        st_cluster_f32x4(slot, 0, acc[0], acc[1], acc[2], acc[3]);
        mbar_arrive_cluster(red_full, 0);
      } else {
        if (mbar_wait_cluster(red_full, 0)) {
          for (int r = 1; r < ksplit; ++r) {   // fixed order: deterministic
            const float4 v = *(const float4*)(red + (((r - 1) * kConsumerWarps + cw) * 32 + lane) * 4);
            acc[0] += v.x;
            acc[1] += v.y;
            acc[2] += v.z;
            acc[3] += v.w;
          }
        }
      }
    }
    if (rank == 0) {
      const int ra = row0 + 16 * cw + g, rb = ra + 8;
      const int c0 = 2 * t, c1 = 2 * t + 1;
      if (ra < p.N) {
        if (c0 < p.batch) p.y[(int64_t)c0 * p.N + ra] = acc[0];
        if (c1 < p.batch) p.y[(int64_t)c1 * p.N + ra] = acc[1];
      }
      if (rb < p.N) {
        if (c0 < p.batch) p.y[(int64_t)c0 * p.N + rb] = acc[2];
        if (c1 < p.batch) p.y[(int64_t)c1 * p.N + rb] = acc[3];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Q4_K, one activation column: the block-diagonal core (Q4KB1).  Each stage
// carries one super-block of 64 weight rows (TMA) and its 256 activations,
// staged by the loader warp: fp16 values (bf16 input scaled by a power of two
// per stage), the negated sum of each 32-value sub-block, and the stage's
// inverse scale.  The loader keeps the activation loads of the next
// kB1Prefetch stages in flight in registers.
// ---------------------------------------------------------------------------
struct B1Params {
  CUtensorMap tmap;  // W as [N rows][row_bytes/2] 16-bit elements, box BOX x 64 rows
  int N;
  int nsb;           // super-blocks per row
  const void* x;     // [K], fp16 or bf16
  float* y;          // [N]
  int nstage;
  int w_early;
};

// PAIR: each consumer iteration takes two stages (more independent work per
// warp, more registers: three CTAs per SM instead of four).
template <int FMT, bool BF16, bool PAIR>
__global__ void __launch_bounds__(kThreads, PAIR ? 3 : 4)
    qgemv_b1_kernel(const __grid_constant__ B1Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using L = Layout<FMT>;
  constexpr int kStageX = B1Fmt<FMT>::kStageX, kSubs = B1Fmt<FMT>::kSubs;
  const int ksplit = (int)cluster_nctarank();
  const int rank = (int)cluster_ctarank();
  const B1Plan plan = b1_plan<FMT>(p.nstage, ksplit);
  uint64_t* full = (uint64_t*)smem;
  uint64_t* empty = full + plan.nstage;
  uint64_t* red_full = empty + plan.nstage;
  uint8_t* wbuf = smem + plan.off_w;
  float* red = (float*)(smem + plan.off_red);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.y * kTileRows;
  const int sb0 = (int)((int64_t)p.nsb * rank / ksplit);
  const int sb1 = (int)((int64_t)p.nsb * (rank + 1) / ksplit);
  const int nsbl = sb1 - sb0;

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < plan.nstage; ++s) {
      mbar_init(&full[s], 33);          // TMA bytes + one arrival per loader lane
      mbar_init(&empty[s], kConsumerWarps);
    }
    if (ksplit > 1) mbar_init(red_full, (ksplit - 1) * kConsumerWarps * 32);
    fence_barrier_init();
  }
  if (threadIdx.x < 32) ((uint32_t*)(smem + plan.off_z))[threadIdx.x] = 0u;
  __syncthreads();
  const uint64_t pol = l2_evict_first_policy();
  auto issue = [&](int c, int s) {
    mbar_arrive_expect_tx(&full[s], L::W_STAGE);   // rows past N are zero-filled, still counted
    // box start: the super-block's first byte rounded down to 16 bytes
    tma_load_2d(wbuf + s * L::W_STAGE, &p.tmap,
                (int)((((int64_t)(sb0 + c) * L::SBB) & ~(int64_t)15) >> 1), row0, &full[s], pol);
  };
  const int early = p.w_early == 1 ? min(plan.nstage, nsbl) : 0;
  if (threadIdx.x == 0) {
    prefetch_tmap(&p.tmap);
    // weights are read-only: stream them in while the previous kernel ends
    // (and while the cluster forms)
    for (int c = 0; c < early; ++c) issue(c, c);
    // the range exceeds the ring: only its first stages, into L2
    if (p.w_early == 2)
      for (int c = 0; c < min(nsbl, kL2PrefetchStages); ++c)
        tma_prefetch_l2_2d(&p.tmap, (int)((((int64_t)(sb0 + c) * L::SBB) & ~(int64_t)15) >> 1),
                           row0);
  }
  // the cluster's reduction barrier must be initialised before any peer
  // arrives on it, at the end of the kernel
  if (ksplit > 1) cluster_sync_all();

  if (warp == 0) {
    // ------------------------------- loader --------------------------------
    pdl_wait();
    // lane covers activations 8*lane .. 8*lane+7 of a stage; sub-block = lane/4
    constexpr int XDT = BF16 ? DQ_BF16 : DQ_F16;
    B1X<XDT> xr[kB1Prefetch];
#pragma unroll
    for (int u = 0; u < kB1Prefetch; ++u)
      if (u < nsbl) xr[u] = b1_load_x<XDT>(p.x, sb0 + u, lane);
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int c0 = 0; c0 < nsbl && ok; c0 += kB1Prefetch) {
#pragma unroll
      for (int u = 0; u < kB1Prefetch; ++u) {
        const int c = c0 + u;
        // warp-uniform: every lane leaves together after a timed-out wait
        if (ok && c < nsbl && c >= plan.nstage)
          ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ph ^ 1));
        if (!ok || c >= nsbl) continue;
        if (lane == 0 && c >= early) issue(c, s);
        const B1X<XDT> cur = xr[u];
        if (c + kB1Prefetch < nsbl) xr[u] = b1_load_x<XDT>(p.x, sb0 + c + kB1Prefetch, lane);
        b1_stage_x<FMT, XDT>(cur, smem + plan.off_x + s * kStageX,
                             (float*)(smem + plan.off_sx + s * 4 * kSubs),
                             (float*)(smem + plan.off_inv) + s, lane);
        mbar_arrive(&full[s]);
        if (++s == plan.nstage) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  } else {
    // ------------------------------ consumers ------------------------------
    const int cw = warp - 1;
    const B1Consumer<FMT, BF16, 8> cons(smem, plan, 16 * cw, lane);
    float2 accp0 = make_float2(0.f, 0.f), accp8 = make_float2(0.f, 0.f);
    float2 accq0 = make_float2(0.f, 0.f), accq8 = make_float2(0.f, 0.f);
    int s = 0;
    uint32_t ph = 0;
    // super-block c of this CTA sits in stage st
    auto stage = [&](int st, int c, uint32_t o, float2& a0, float2& a8) {
      cons.stage(st, (int64_t)sb0 + c, o, a0, a8);
    };
    auto advance = [&]() {
      if (++s == plan.nstage) {
        s = 0;
        ph ^= 1;
      }
    };
    // two stages per iteration: independent work for the scheduler to interleave
    int c = 0;
    bool ok = true;
    for (; PAIR && c + 1 < nsbl; c += 2) {
      const int s0 = s;
      if (!mbar_wait(&full[s], ph)) { ok = false; break; }
      advance();
      const int s1 = s;
      if (!mbar_wait(&full[s], ph)) { ok = false; break; }
      advance();
      const uint32_t o = order_after_wait(0u);
      stage(s0, c, o, accp0, accp8);
      stage(s1, c + 1, o, accq0, accq8);
      keep_before_release(accp0.x, accp0.y, accp8.x, accp8.y);
      keep_before_release(accq0.x, accq0.y, accq8.x, accq8.y);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_relaxed(&empty[s0]);
        mbar_arrive_relaxed(&empty[s1]);
      }
    }
    for (; ok && c < nsbl; ++c) {
      if (!mbar_wait(&full[s], ph)) break;
      const uint32_t o = order_after_wait(0u);
      stage(s, c, o, accp0, accp8);
      keep_before_release(accp0.x, accp0.y, accp8.x, accp8.y);
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&empty[s]);
      advance();
    }
    float acc0 = (accp0.x + accp0.y) + (accq0.x + accq0.y);
    float acc8 = (accp8.x + accp8.y) + (accq8.x + accq8.y);
    b1_quad_sum(acc0, acc8);
    if (ksplit > 1) {
      if (rank != 0) {
        float* slot = red + (((rank - 1) * kConsumerWarps + cw) * 32 + lane) * 4;
        st_cluster_f32x4(slot, 0, acc0, acc8, 0.f, 0.f);
        mbar_arrive_cluster(red_full, 0);
      } else if (mbar_wait_cluster(red_full, 0)) {
        for (int r = 1; r < ksplit; ++r) {   // fixed order: deterministic
          const float4 v = *(const float4*)(red + (((r - 1) * kConsumerWarps + cw) * 32 + lane) * 4);
          acc0 += v.x;
          acc8 += v.y;
        }
      }
    }
    if (rank == 0 && cons.t == 0) {
      const int ra = row0 + 16 * cw + cons.rg, rb = ra + 8;
      if (ra < p.N) p.y[ra] = acc0;
      if (rb < p.N) p.y[rb] = acc8;
    }
  }
}

namespace {

int device_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64 && cached[dev]) return cached[dev];
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64) cached[dev] = sms;
  return sms;
}

// Early weight streaming (DQ_QGEMV_WEIGHTS_EARLY).  Where a CTA's whole K
// range fits its ring (mode 1) every stage is copied into shared memory
// before the wait, so all of its weights are in flight when the previous
// kernel completes.  Measured on GB300 (graphs of back-to-back launches of one
// Llama-3-8B linear, batch 1): faster for qkv 6144 x 4096 (4 super-blocks per
// CTA, 5.94 against 6.32 us) and o 4096 x 4096 (2: 4.89 against 5.47 us).
// Where it does not (mode 2) the first kL2PrefetchStages stages are only
// prefetched into L2: copying a partial ring into shared memory early was
// slower (gate/up 28672 x 4096: 14.6 against 13.6 us; down 4096 x 14336: 10.6
// against 9.5 us), as it competes with the previous kernel's last CTAs for
// HBM; an L2 prefetch of 2 stages gives 12.4 / 8.7 us (3 stages 12.3 / 8.8,
// 4: 12.4 / 9.0, 6: 12.6 / 9.4, 8: 13.0 / 9.6, the whole range 15.1 / 9.6;
// the 70B gate 28672 x 8192: 24.0 us without, 22.8 us with 2 stages).
int early_weights(bool w_early, int nsb, int ks, int nstage) {
  if (!w_early) return 0;
  return (nsb + ks - 1) / ks <= nstage ? 1 : 2;
}

// Pick the K-split (cluster size) for `tiles` 64-row tiles when an SM holds
// `per_sm` CTAs of the kernel.  Measured on GB300 (graphs of back-to-back
// launches):
//   * with two or more tiles per SM the unsplit grid is best (28672 x 8192:
//     batch 1 23.8 us unsplit against 29.0 us split in two; batch 8 Q4_K 34.5
//     against 38.3 us, Q8_0 46.6 against 50.6 us, Q6_K even);
//   * with fewer, the split that fills the SMs' CTA slots in one wave:
//     per_sm * sms / tiles, rounded down to 4 or 8 from 4 up.  Q4_K at
//     8192 x 28672 / 8192 x 8192 (4 per SM): split 4 26.9 / 10.5 us, 3 27.8 /
//     11.0, 6 (two waves) 35.1 / 14.9.  Kernels whose shared memory allows
//     three per SM (the batch-8 Q6_K / Q8_0 rings, the batch-1 Q8_0 ring) take
//     3: Q8_0 8192 x 28672 batch 8 54.1 us against 74.4 us at 4 (512 CTAs for
//     456 slots: two waves) and 74.1 at 2; Q8_0 batch 1 45.9 against 56.3 us
//     at 4 on the shallower 4-per-SM ring; Q6_K 8192 x 8192 batch 8 21.7
//     against 24.6 us.
int choose_ksplit(int tiles, int nsb, int sms, int per_sm) {
  if (tiles >= 2 * sms) return 1;
  int s = std::min(8, std::min(nsb, std::max(1, per_sm * sms / tiles)));
  if (s >= 4) s = s >= 8 ? 8 : 4;
  return s;
}

}  // namespace

template <int FMT>
int launch_qgemv_mma_fmt(const void* W, int64_t N, int64_t K, const void* x, int xdt, int batch,
                         float* y, cudaStream_t stream, int force_ksplit, bool w_early) {
  using L = Layout<FMT>;
  GemvParams p;
  p.W = (const uint8_t*)W;
  p.nsb = (int)(K / 256);
  p.row_bytes = (int64_t)p.nsb * L::SBB;
  if (!make_weight_tmap(&p.tmap, W, (uint64_t)N, (uint64_t)p.row_bytes, L::BOX, kTileRows))
    return DQ_ERR_CUDA;
  p.N = (int)N;
  p.x.base = x;
  p.x.dtype = xdt;
  p.x.col_stride = K;
  p.x.rows = nullptr;
  p.batch = batch;
  p.y = y;
  const int tiles = (int)((N + kTileRows - 1) / kTileRows);
  const int sms = device_sms();
  if (sms <= 0) return DQ_ERR_CUDA;
  // shared memory per CTA <= 56 KB so that four CTAs (20 warps) share an SM
  constexpr int kSmemBudget = 56 * 1024;
  const bool bf16x =
      xdt == DQ_BF16 && (batch >= 4 || (batch >= 2 && (FMT == DQ_Q4_K || FMT == DQ_Q6_K)));
  // CTAs per SM: four where a three-stage ring fits the 56 KB budget, else
  // three; three for the uncapped Q6_K bf16 instance
  const int per_sm =
      (!(bf16x && FMT == DQ_Q6_K) && make_plan<FMT>(3, batch, 4).total <= kSmemBudget) ? 4 : 3;
  int ks = force_ksplit > 0 ? force_ksplit : choose_ksplit(tiles, p.nsb, sms, per_sm);
  ks = std::max(1, std::min(ks, std::min(8, p.nsb)));
  // Q4_K grids of at most three CTAs per SM take the paired kernel with
  // deeper rings (28672 x 8192 at batch 8: 34.4 us against 38.2 us split in
  // two); the heavier Q6_K / Q8_0 decodes measured slower paired (64.1 / 54.1
  // us against 56.0 / 50.3 us)
  const bool pair = FMT == DQ_Q4_K && (long)tiles * ks <= 3L * sms;
  const int budget = pair ? 74 * 1024 : kSmemBudget;
  int nstage = 12;
  while (nstage > 3 && make_plan<FMT>(nstage, batch, ks).total > budget) --nstage;
  p.nstage = nstage;
  p.w_early = early_weights(w_early, p.nsb, ks, nstage);
  const SmemPlan plan = make_plan<FMT>(nstage, batch, ks);
  auto kern = pair ? (bf16x ? qgemv_mma_kernel<FMT, true, true> : qgemv_mma_kernel<FMT, true, false>)
                   : (bf16x ? qgemv_mma_kernel<FMT, false, true>
                            : qgemv_mma_kernel<FMT, false, false>);
  static bool attr_set[4][64] = {};
  const int v = (pair ? 1 : 0) + (bf16x ? 2 : 0);
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[v][dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
        cudaSuccess)
      return DQ_ERR_CUDA;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
      return DQ_ERR_CUDA;
    if (dev < 64) attr_set[v][dev] = true;
  }
  if (launch_pdl(kern, dim3((unsigned)ks, (unsigned)tiles, 1), dim3(kThreads), (size_t)plan.total,
                 stream, ks, p) != cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

// One fp16 / bf16 column of Q4_K, Q6_K, Q8_0, Q2_K or Q3_K: the block-diagonal kernel.
template <int FMT>
int launch_qgemv_b1(const void* W, int64_t N, int64_t K, const void* x, int xdt, float* y,
                    cudaStream_t stream, int force_ksplit, bool w_early) {
  using L = Layout<FMT>;
  B1Params p;
  p.nsb = (int)(K / 256);
  const int tiles = (int)((N + kTileRows - 1) / kTileRows);
  const int sms = device_sms();
  if (sms <= 0) return DQ_ERR_CUDA;
  // CTAs per SM: four on the single-stage kernel; Q8_0, whose light decode
  // needs the deeper rings of the paired kernel, three
  const int per_sm = FMT == DQ_Q8_0 ? 3 : 4;
  int ks = force_ksplit > 0 ? force_ksplit : choose_ksplit(tiles, p.nsb, sms, per_sm);
  ks = std::max(1, std::min(ks, std::min(8, p.nsb)));
  // grids that fit three CTAs per SM take the paired kernel with deeper rings
  // (28672 x 8192: 23.8 us against 28.2 us); larger ones four CTAs per SM
  const bool pair = (long)tiles * ks <= 3L * sms;
  const int budget = pair ? 74 * 1024 : 56 * 1024;
  int nstage = 12;
  while (nstage > 3 && b1_plan<FMT>(nstage, ks).total > budget) --nstage;
  const B1Plan plan = b1_plan<FMT>(nstage, ks);
  if (!make_weight_tmap(&p.tmap, W, (uint64_t)N, (uint64_t)p.nsb * L::SBB, L::BOX, kTileRows))
    return DQ_ERR_CUDA;
  p.N = (int)N;
  p.x = x;
  p.y = y;
  p.nstage = nstage;
  p.w_early = early_weights(w_early, p.nsb, ks, nstage);
  auto kern = xdt == DQ_BF16 ? (pair ? qgemv_b1_kernel<FMT, true, true>
                                     : qgemv_b1_kernel<FMT, true, false>)
                             : (pair ? qgemv_b1_kernel<FMT, false, true>
                                     : qgemv_b1_kernel<FMT, false, false>);
  static bool attr_set[4][64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int v = (xdt == DQ_BF16 ? 1 : 0) + (pair ? 2 : 0);
  if (dev >= 64 || !attr_set[v][dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
        cudaSuccess)
      return DQ_ERR_CUDA;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
      return DQ_ERR_CUDA;
    if (dev < 64) attr_set[v][dev] = true;
  }
  if (launch_pdl(kern, dim3((unsigned)ks, (unsigned)tiles, 1), dim3(kThreads), (size_t)plan.total,
                 stream, ks, p) != cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

int launch_qgemv_mma(int fmt, const void* W, int64_t N, int64_t K, const void* x, int xdt,
                     int batch, float* y, cudaStream_t s, int force_ksplit, bool w_early) {
  if (fmt == DQ_Q4_K && batch == 1)
    return launch_qgemv_b1<DQ_Q4_K>(W, N, K, x, xdt, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q6_K && batch == 1)
    return launch_qgemv_b1<DQ_Q6_K>(W, N, K, x, xdt, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q8_0 && batch == 1)
    return launch_qgemv_b1<DQ_Q8_0>(W, N, K, x, xdt, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q2_K && batch == 1)
    return launch_qgemv_b1<DQ_Q2_K>(W, N, K, x, xdt, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q3_K && batch == 1)
    return launch_qgemv_b1<DQ_Q3_K>(W, N, K, x, xdt, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q4_K)
    return launch_qgemv_mma_fmt<DQ_Q4_K>(W, N, K, x, xdt, batch, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q6_K)
    return launch_qgemv_mma_fmt<DQ_Q6_K>(W, N, K, x, xdt, batch, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q8_0)
    return launch_qgemv_mma_fmt<DQ_Q8_0>(W, N, K, x, xdt, batch, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q4_0)
    return launch_qgemv_mma_fmt<DQ_Q4_0>(W, N, K, x, xdt, batch, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q5_K)
    return launch_qgemv_mma_fmt<DQ_Q5_K>(W, N, K, x, xdt, batch, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q2_K)
    return launch_qgemv_mma_fmt<DQ_Q2_K>(W, N, K, x, xdt, batch, y, s, force_ksplit, w_early);
  if (fmt == DQ_Q3_K)
    return launch_qgemv_mma_fmt<DQ_Q3_K>(W, N, K, x, xdt, batch, y, s, force_ksplit, w_early);
  return launch_qgemv_mma_fmt<DQ_NVFP4>(W, N, K, x, xdt, batch, y, s, force_ksplit, w_early);
}

}  // namespace dqmoe
