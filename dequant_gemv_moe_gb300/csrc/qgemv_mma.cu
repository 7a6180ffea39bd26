// qgemv_mma.cu — dq_qgemv for 16-bit activations (and the scaled path for
// bf16): the streaming GEMV of qgemv_mma.cuh over a grid of 64-row tiles,
// optionally split along K over a thread-block cluster whose partial sums are
// reduced through distributed shared memory (split-K for small N, without a
// second pass and without scratch memory).
#include <algorithm>

#include "qgemv_mma.cuh"
#include "tmap.h"

namespace dqmoe {

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

template <int FMT>
__global__ void __launch_bounds__(kThreads) qgemv_mma_kernel(const __grid_constant__ GemvParams p) {
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
    const int early = p.w_early ? min(plan.nstage, nchunk) : 0;
    if (lane == 0)
      for (int c = 0; c < early; ++c) {
        const int64_t a = ((int64_t)(sb0 + c) * L::SBB) & ~(int64_t)15;
        mbar_arrive_expect_tx(&full[c], L::W_STAGE);
        tma_load_2d(wbuf + c * L::W_STAGE, &p.tmap, (int)(a >> 1), row0, &full[c], pol);
      }
    pdl_wait();
    bool ok = true;
    int s = 0;
    uint32_t ph = 0;            // phase parity of stage s in the current round
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
      stage_x<FMT>(p.x, p.batch, (int64_t)c0 * 256, 1, xbuf + s * p.batch * L::XCOL,
                   xinv + s * 8, lane, &full[s]);
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
    for (int c = 0; c < nchunk; ++c) {
      ok = ok && mbar_wait(&full[s], ph);
      if (ok) {
        const int c0 = sb0 + c;
        const uint32_t wst = wrow + s * L::W_STAGE + (uint32_t)(((int64_t)c0 * L::SBB) & 15);
        const uint32_t xcol[1] = {xcol0 + s * p.batch * L::XCOL};
        if constexpr (SBDot<FMT>::kRowScale) {
          float d[1][2][4] = {};
          float r0, r8;
          SBDot<FMT>::template run<1>(wst, 8 * L::ROW_PITCH, xcol, 0, t, d, r0, r8);
          const float c0 = f16 ? 1.f : xinv[s * 8 + ((2 * t) & 7)];
          const float c1 = f16 ? 1.f : xinv[s * 8 + ((2 * t + 1) & 7)];
          fold_tile(acc, d[0], r0, r8, c0, c1);
        } else if (f16) {
          SBDot<FMT>::template run<1>(wst, 8 * L::ROW_PITCH, xcol, 0, t, accs);
        } else {
          float pt[1][2][4] = {};
          SBDot<FMT>::template run<1>(wst, 8 * L::ROW_PITCH, xcol, 0, t, pt);
          const float inv0 = xinv[s * 8 + ((2 * t) & 7)], inv1 = xinv[s * 8 + ((2 * t + 1) & 7)];
          fold_tile(acc, pt[0], 1.f, 1.f, inv0, inv1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&empty[s]);
      }
      if (++s == plan.nstage) {
        s = 0;
        ph ^= 1;
      }
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

// Pick the K-split (cluster size).  Measured on GB300 (graphs of back-to-back
// launches): with two or more 64-row tiles per SM the unsplit grid (or a split
// in two for long rows) is within a few percent of the best; with fewer, the
// best split is the largest power of
// two whose CTAs all fit at once (four per SM, the 56 KB shared-memory
// budget).  Odd cluster sizes (3, 5, 6, 7) measured slower than the
// neighbouring powers of two on every shape tried: a cluster's CTAs share one
// GPC, and odd sizes leave SMs of it idle.
int choose_ksplit(int tiles, int nsb, int sms) {
  // many tiles: unsplit, except long rows (>= 32 super-blocks), where halving
  // each CTA's range measured 6-11% faster (28672 x 8192; at 28672 x 4096 the
  // split gained nothing)
  if (tiles >= 2 * sms) return (nsb >= 32 && (long)tiles * 2 <= 8L * sms) ? 2 : 1;
  int s = 1;
  while (2 * s <= 8 && 2 * s <= nsb && (long)tiles * 2 * s <= 4L * sms) s *= 2;
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
  p.w_early = w_early ? 1 : 0;
  const int tiles = (int)((N + kTileRows - 1) / kTileRows);
  const int sms = device_sms();
  if (sms <= 0) return DQ_ERR_CUDA;
  // shared memory per CTA <= 56 KB so that four CTAs (20 warps) share an SM
  constexpr int kSmemBudget = 56 * 1024;
  int ks = force_ksplit > 0 ? force_ksplit : choose_ksplit(tiles, p.nsb, sms);
  ks = std::max(1, std::min(ks, std::min(8, p.nsb)));
  int nstage = 12;
  while (nstage > 3 && make_plan<FMT>(nstage, batch, ks).total > kSmemBudget) --nstage;
  p.nstage = nstage;
  const SmemPlan plan = make_plan<FMT>(nstage, batch, ks);
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr_set[dev]) {
    if (cudaFuncSetAttribute(qgemv_mma_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             200 * 1024) != cudaSuccess)
      return DQ_ERR_CUDA;
    if (cudaFuncSetAttribute(qgemv_mma_kernel<FMT>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) != cudaSuccess)
      return DQ_ERR_CUDA;
    if (dev < 64) attr_set[dev] = true;
  }
  if (launch_pdl(qgemv_mma_kernel<FMT>, dim3((unsigned)ks, (unsigned)tiles, 1), dim3(kThreads),
                 (size_t)plan.total, stream, ks, p) != cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

int launch_qgemv_mma(int fmt, const void* W, int64_t N, int64_t K, const void* x, int xdt,
                     int batch, float* y, cudaStream_t s, int force_ksplit, bool w_early) {
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
  return launch_qgemv_mma_fmt<DQ_NVFP4>(W, N, K, x, xdt, batch, y, s, force_ksplit, w_early);
}

}  // namespace dqmoe
