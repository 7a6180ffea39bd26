// moe_b1.cu — the MoE layer's expert products for experts that received
// exactly one token in this call, on the one-column (block-diagonal) core of
// the batch-1 GEMV.
//
// A decode step routes each token to top_k of E experts; with few tokens
// (DeepSeek-V3-shaped layer: T = 1, or T = 8 with 64 picks over 256 experts)
// almost every touched expert sees one token, so its three matrices are
// GEMVs with one activation column.  The grouped kernel of moe.cu computes
// such a group on the 8-column mma.sync core with one real column (~362 warp
// instructions per 16 rows x 256 weights); this kernel runs the block-
// diagonal core of the batch-1 GEMV (the 8 mma columns carry the 8 sub-blocks
// of one column, ~238) and reads the activations as they are (fp16, bf16, or
// the fp32 SwiGLU output), converting each 256-value stage to fp16 with one
// power-of-two scale in the loader: no separate conversion launch.
//
// Work: units of (one-token group, row tile).  CTA b takes unit b first, then
// claims further units one at a time from a counter (which balances the work
// across SMs); the loader makes each claim two units ahead and reads its group
// record one unit ahead, so their latency hides behind the current unit's
// stages.  Units are streamed as stages of one
// super-block of 64 rows:
//   gate/up: 32 rows of W_gate and the same 32 rows of W_up (two TMA boxes);
//            consumer warp w holds gate rows 8w + r and the matching up rows,
//            so h = silu(g) * u is formed in the lane that holds both;
//   down   : 64 rows of W_down.
// The loader writes each stage's (unit, super-block, output position) into a
// slot beside the stage, and an empty stage with unit -1 after the last one.
// [Titan Engine, §MoE 专家流式加载]: few experts per token are active, so the
// layer is bound by the bytes of the touched experts.
#include <algorithm>
#include <cstring>

#include "b1.cuh"
#include "moe_plan.h"
#include "tmap.h"

namespace dqmoe {

struct GroupedB1Params {
  // the stacked matrices as [experts * rows][row_bytes / 2] 16-bit elements:
  // routed a (gate or down), routed b (up), shared a, shared b; boxes of BOX
  // bytes x 32 rows (gate/up) or 64 rows (down)
  CUtensorMap map_a, map_b, map_sa, map_sb;
  int rows_per_expert;   // F (gate/up) or H (down)
  int E;
  int nsb;               // super-blocks per row (K / 256)
  int tiles;             // units per group: F / 32 (gate/up) or H / 64 (down)
  const int4* groups;    // one-token groups: (matrix: e < E routed, E + s shared,
                         //  position, activation row, 0)
  const int* n_groups;
  int* claim;            // work counter, zero when the kernel starts (counts the
                         // claims beyond the first unit of every CTA)
  const void* x;         // gate/up: x [T][H] (row = the group's token); down: h [NP][F]
                         // (row = the group's position)
  int64_t xstride;       // elements per activation row
  float* out;            // gate/up: h [NP][F]; down: ypos [NP][H]
  int64_t out_stride;
  int nstage;
};

// shared memory: the b1 ring plus one (unit, super-block, position) slot per
// stage
template <int FMT>
__host__ __device__ inline int grouped_b1_item_off(int nstage) {
  return b1_plan<FMT>(nstage, 1).total;
}
template <int FMT>
__host__ __device__ inline int grouped_b1_smem(int nstage) {
  return grouped_b1_item_off<FMT>(nstage) + 16 * nstage;
}

template <int FMT, bool GATEUP, int XDT>
__global__ void __launch_bounds__(kThreads, 4)
    grouped_b1_kernel(const __grid_constant__ GroupedB1Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using L = Layout<FMT>;
  constexpr int kStageX = B1Fmt<FMT>::kStageX, kSubs = B1Fmt<FMT>::kSubs;
  constexpr int kRows = GATEUP ? 32 : 64;   // weight rows per TMA box
  const B1Plan plan = b1_plan<FMT>(p.nstage, 1);
  uint64_t* full = (uint64_t*)smem;
  uint64_t* empty = full + plan.nstage;
  int4* item = (int4*)(smem + grouped_b1_item_off<FMT>(p.nstage));
  uint8_t* wbuf = smem + plan.off_w;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < plan.nstage; ++s) {
      mbar_init(&full[s], 33);          // TMA bytes + one arrival per loader lane
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  if (threadIdx.x < 32) ((uint32_t*)(smem + plan.off_z))[threadIdx.x] = 0u;
  __syncthreads();
  // the groups, the counter and the activations come from earlier kernels
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------- loader --------------------------------
    const uint64_t pol = l2_evict_first_policy();
    if (lane == 0) {
      prefetch_tmap(&p.map_a);
      prefetch_tmap(&p.map_sa);
      if (GATEUP) {
        prefetch_tmap(&p.map_b);
        prefetch_tmap(&p.map_sb);
      }
    }
    const int total = __ldcg(p.n_groups) * p.tiles;
    constexpr int kXBytes = XDT == DQ_F32 ? 4 : 2;
    // lane 0 holds the next unit u1 with its group record g1 and the unit
    // after it, u2: unit b first, then claims from the counter; each claim is
    // made two units ahead and its group record read one unit ahead, so
    // neither load stalls the loader
    int u1 = (int)blockIdx.x, u2 = 0;
    int4 g1 = make_int4(0, 0, 0, 0);
    if (lane == 0) {
      if (u1 < total) g1 = __ldcg(p.groups + u1 / p.tiles);
      u2 = (int)gridDim.x + atomicAdd(p.claim, 1);
    }
    // the current unit (enqueue side): activation row, first weight row (bit
    // 30: shared expert), output position
    const char* xrow = nullptr;
    int wrow = 0, wpos = 0;
    auto take_next = [&]() -> int {
      const int u = __shfl_sync(0xffffffffu, u1, 0);
      if (u >= total) return -1;
      const int gx = __shfl_sync(0xffffffffu, g1.x, 0);
      const int gy = __shfl_sync(0xffffffffu, g1.y, 0);
      const int gz = __shfl_sync(0xffffffffu, g1.z, 0);
      const int tile = u % p.tiles;
      const bool shared = gx >= p.E;
      // gate/up reads the token's x row, down the position's h row
      xrow = (const char*)p.x + (int64_t)(GATEUP ? gz : gy) * p.xstride * kXBytes;
      wrow = (shared ? (1 << 30) : 0) | ((shared ? gx - p.E : gx) * p.rows_per_expert +
                                         tile * kRows);
      wpos = gy;
      if (lane == 0) {
        u1 = u2;
        if (u1 < total) g1 = __ldcg(p.groups + u1 / p.tiles);
        u2 = (int)gridDim.x + atomicAdd(p.claim, 1);
      }
      return u;
    };
    // the next item to enqueue: unit nu (-1: none left), super-block nc
    int nu = take_next(), nc = 0;
    int qu[kB1Prefetch], qc[kB1Prefetch], qw[kB1Prefetch], qp[kB1Prefetch];
    B1X<XDT> qx[kB1Prefetch];
    auto enqueue = [&](int d) {
      qu[d] = nu;
      qc[d] = nc;
      if (nu < 0) return;
      qw[d] = wrow;
      qp[d] = wpos;
      qx[d] = b1_load_x<XDT>(xrow, nc, lane);
      if (++nc == p.nsb) {
        nc = 0;
        nu = take_next();
      }
    };
#pragma unroll
    for (int d = 0; d < kB1Prefetch; ++d) enqueue(d);
    int s = 0, n = 0;
    uint32_t ph = 0;
    bool ok = true, done = false;
    while (ok && !done) {
#pragma unroll
      for (int d = 0; d < kB1Prefetch; ++d) {
        if (!ok || done) continue;
        // warp-uniform: every lane leaves together after a timed-out wait
        if (n >= plan.nstage) ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ph ^ 1));
        if (!ok) continue;
        const int u = qu[d], c = qc[d];
        if (lane == 0) item[s] = make_int4(u, c, u < 0 ? 0 : qp[d], 0);
        if (u < 0) {
          // no work left: an empty stage with unit -1 ends the consumers' walk
          if (lane == 0) mbar_arrive(&full[s]);
          mbar_arrive(&full[s]);
          done = true;
          continue;
        }
        if (lane == 0) {
          const int x0 = (int)((((int64_t)c * L::SBB) & ~(int64_t)15) >> 1);
          const bool shared = (qw[d] >> 30) & 1;
          const int row = qw[d] & ((1 << 30) - 1);
          uint8_t* wst = wbuf + s * L::W_STAGE;
          mbar_arrive_expect_tx(&full[s], L::W_STAGE);
          tma_load_2d(wst, shared ? &p.map_sa : &p.map_a, x0, row, &full[s], pol);
          if (GATEUP)
            tma_load_2d(wst + 32 * L::ROW_PITCH, shared ? &p.map_sb : &p.map_b, x0, row, &full[s],
                        pol);
        }
        const B1X<XDT> cur = qx[d];
        enqueue(d);   // the item kB1Prefetch further on: its activation loads in flight
        b1_stage_x<FMT, XDT>(cur, smem + plan.off_x + s * kStageX,
                             (float*)(smem + plan.off_sx + s * 4 * kSubs),
                             (float*)(smem + plan.off_inv) + s, lane);
        mbar_arrive(&full[s]);
        ++n;
        if (++s == plan.nstage) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  } else {
    // ------------------------------ consumers ------------------------------
    const int cw = warp - 1;
    // gate/up: gate rows 8cw + rg and the up rows 32 further; down: rows
    // 16cw + rg and 8 further
    const B1Consumer<FMT, XDT != DQ_F16, GATEUP ? 32 : 8> cons(smem, plan,
                                                              GATEUP ? 8 * cw : 16 * cw, lane);
    const uint32_t item0 = smem_u32(item);
    float2 a0 = make_float2(0.f, 0.f), a8 = make_float2(0.f, 0.f);
    int s = 0;
    uint32_t ph = 0;
    for (;;) {
      if (!mbar_wait(&full[s], ph)) break;
      const uint32_t o = order_after_wait(0u);
      const uint4 it = lds_u128_nv(item0 + 16 * s + o);
      const int u = (int)it.x, c = (int)it.y, pos = (int)it.z;
      if (u < 0) break;
      cons.stage(s, c, o, a0, a8);
      keep_before_release(a0.x, a0.y, a8.x, a8.y);
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&empty[s]);
      if (++s == plan.nstage) {
        s = 0;
        ph ^= 1;
      }
      if (c == p.nsb - 1) {
        // the unit's last super-block: its rows are complete
        float acc0 = a0.x + a0.y, acc8 = a8.x + a8.y;
        b1_quad_sum(acc0, acc8);
        a0 = make_float2(0.f, 0.f);
        a8 = make_float2(0.f, 0.f);
        if (cons.t == 0) {
          const int tile = u % p.tiles;
          float* orow = p.out + (int64_t)pos * p.out_stride;
          if (GATEUP) {
            // silu(g) = g / (1 + exp(-g)); for g < -88 exp overflows to inf
            // and the quotient is -0, never NaN
            orow[tile * 32 + 8 * cw + cons.rg] = acc0 / (1.f + expf(-acc0)) * acc8;
          } else {
            const int r = tile * 64 + 16 * cw + cons.rg;
            orow[r] = acc0;
            orow[r + 8] = acc8;
          }
        }
      }
    }
  }
}

namespace {

int sm_count_b1() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

template <int FMT, bool GATEUP, int XDT>
int launch_b1(const GroupedB1Params& gp_in, int units_max, const void* Wa, const void* Wb,
              const void* Sa, const void* Sb, int E, int n_shared, int64_t row_bytes,
              cudaStream_t s) {
  using L = Layout<FMT>;
  GroupedB1Params gp = gp_in;
  const uint32_t box_rows = GATEUP ? 32 : 64;
  const uint64_t rpe = (uint64_t)gp.rows_per_expert;
  if (!make_weight_tmap(&gp.map_a, Wa, rpe * E, row_bytes, L::BOX, box_rows)) return DQ_ERR_CUDA;
  if (GATEUP && !make_weight_tmap(&gp.map_b, Wb, rpe * E, row_bytes, L::BOX, box_rows))
    return DQ_ERR_CUDA;
  if (n_shared > 0) {
    if (!make_weight_tmap(&gp.map_sa, Sa, rpe * n_shared, row_bytes, L::BOX, box_rows))
      return DQ_ERR_CUDA;
    if (GATEUP && !make_weight_tmap(&gp.map_sb, Sb, rpe * n_shared, row_bytes, L::BOX, box_rows))
      return DQ_ERR_CUDA;
  } else {
    // never read (no shared groups): valid maps over the routed matrices
    gp.map_sa = gp.map_a;
    gp.map_sb = GATEUP ? gp.map_b : gp.map_a;
  }
  if (!GATEUP) gp.map_b = gp.map_a;
  int nstage = 12;
  while (nstage > 3 && grouped_b1_smem<FMT>(nstage) > 56 * 1024) --nstage;
  gp.nstage = nstage;
  const int smem = grouped_b1_smem<FMT>(nstage);
  auto kern = grouped_b1_kernel<FMT, GATEUP, XDT>;
  static bool attr[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
        cudaSuccess)
      return DQ_ERR_CUDA;
    if (dev < 64) attr[dev] = true;
  }
  const int sms = sm_count_b1();
  if (sms <= 0) return DQ_ERR_CUDA;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem) != cudaSuccess ||
      occ < 1)
    occ = 1;
  const int grid = std::max(1, std::min(units_max, occ * sms));
  if (launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, 0, gp) != cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}


}  // namespace

bool grouped_b1_supported(int fmt) {
  return fmt == DQ_Q4_K || fmt == DQ_Q6_K || fmt == DQ_Q8_0;
}

// gate/up (gateup) or down for the one-token groups listed in groups1 /
// n_groups1 (at most g1_max of them); x: the activation rows (gate/up: x of
// dtype xdt, fp16 or bf16, row = token; down: fp32 h, row = position).
int launch_grouped_b1(bool gateup, const dq_moe_desc& d, const int4* groups1,
                      const int* n_groups1, int g1_max, int* claim, const void* x, int xdt,
                      int64_t xstride, float* out, int64_t out_stride, cudaStream_t s) {
  const int qk = d.fmt == DQ_Q8_0 ? 32 : 256;
  const int bb = d.fmt == DQ_Q4_K ? 144 : d.fmt == DQ_Q6_K ? 210 : 34;
  GroupedB1Params gp;
  memset(&gp, 0, sizeof(gp));
  gp.E = d.E;
  gp.groups = groups1;
  gp.n_groups = n_groups1;
  gp.claim = claim;
  gp.x = x;
  gp.xstride = xstride;
  gp.out = out;
  gp.out_stride = out_stride;
  int64_t row_bytes;
  if (gateup) {
    gp.rows_per_expert = d.ffn;
    gp.nsb = d.hidden / 256;
    gp.tiles = d.ffn / 32;
    row_bytes = (int64_t)(d.hidden / qk) * bb;
  } else {
    gp.rows_per_expert = d.hidden;
    gp.nsb = d.ffn / 256;
    gp.tiles = d.hidden / 64;
    row_bytes = (int64_t)(d.ffn / qk) * bb;
  }
  const int units_max = std::max(1, g1_max * gp.tiles);
#define DQ_B1(F)                                                                             \
  if (d.fmt == F) {                                                                          \
    if (!gateup)                                                                             \
      return launch_b1<F, false, DQ_F32>(gp, units_max, d.w_down, nullptr, d.sh_down, nullptr, \
                                         d.E, d.n_shared, row_bytes, s);                     \
    if (xdt == DQ_BF16)                                                                      \
      return launch_b1<F, true, DQ_BF16>(gp, units_max, d.w_gate, d.w_up, d.sh_gate, d.sh_up, \
                                         d.E, d.n_shared, row_bytes, s);                     \
    return launch_b1<F, true, DQ_F16>(gp, units_max, d.w_gate, d.w_up, d.sh_gate, d.sh_up,   \
                                      d.E, d.n_shared, row_bytes, s);                        \
  }
  DQ_B1(DQ_Q4_K)
  DQ_B1(DQ_Q6_K)
  DQ_B1(DQ_Q8_0)
#undef DQ_B1
  return DQ_ERR_UNSUPPORTED;
}

}  // namespace dqmoe
