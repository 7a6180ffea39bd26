// moe.cu — the sparse MoE layer on one GPU, as a sequence of launches on one
// stream with no host synchronisation (capturable in one CUDA graph, as
// [KTransformers, §技术原理] runs one graph per decode step):
//   1. router_logits_kernel : logits = x W_r^T, fp32, tiled over (experts,
//      tokens) and split over the hidden dimension into partial sums.
//   2. topk_kernel          : one warp per token sums the partials in a fixed
//      order, picks the top_k logits (lowest index first on ties) and the
//      renormalised softmax gates.
//   3. permute_kernel       : one CTA counts pairs per expert, prefix-sums the
//      counts and scatters the (token, slot) pairs stably by expert; it also
//      emits the work list: (expert, first position, <= 8 columns) groups.
//   4. grouped_kernel<gate/up> : persistent; each unit is 32 rows of W_gate
//      and the same 32 rows of W_up of one expert times that group's tokens
//      (gathered rows of x); epilogue h = silu(g) * u in fp32.
//   5. grouped_kernel<down>    : persistent; 64 rows of W_down times h.
//   6. combine_kernel       : y[t] = sum_i gate[t][i] * y_e(t,i) + shared.
// [Titan Engine, §MoE 专家流式加载]: only a few experts per token are active,
// so only the touched experts' packed weights are streamed from HBM.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "moe_plan.h"
#include "qgemv_mma.cuh"
#include "tmap.h"

namespace dqmoe {

// ===========================================================================
// workspace plan
// ===========================================================================
static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// an expert with more than kWide tokens is computed by the tcgen05 GEMM
constexpr int kWide = 32;

// up to kRouterStreamT tokens the router streams W_r in hidden chunks of
// kRouterChunk (one warp per expert row and chunk), up to kRouterStreamT2 in
// chunks of kRouterChunk2 (the chunk of every token's x stays at 32 KB of
// shared memory); beyond, it tiles
constexpr int kRouterStreamT = 8;
constexpr int kRouterChunk = 1024;
constexpr int kRouterStreamT2 = 32;
constexpr int kRouterChunk2 = 256;

int router_chunk(int T) {
  return T <= kRouterStreamT ? kRouterChunk : T <= kRouterStreamT2 ? kRouterChunk2 : 0;
}

MoePlan moe_plan(const dq_moe_desc& d, int T, bool allow_wide) {
  MoePlan p;
  const int tiles = ((d.E + 63) / 64) * ((T + 31) / 32);
  p.KS = router_chunk(T) ? (d.hidden + router_chunk(T) - 1) / router_chunk(T)
                         : std::max(1, std::min(d.hidden / 256, (320 + tiles - 1) / tiles));
  p.P = (int64_t)T * d.top_k;
  p.NP = p.P + (int64_t)d.n_shared * T;
  // group width from the expected tokens per routed expert (uniform routing):
  // wider groups stream an expert's weights once for more tokens
  const double per_expert = (double)p.P / d.E;
  p.NT = per_expert <= 6.0 ? 1 : per_expert <= 14.0 ? 2 : 4;
  p.GW = 8 * p.NT;
  p.G_max = (int)((p.P + p.GW - 1) / p.GW + std::min<int64_t>(d.E, p.P) +
                  (int64_t)d.n_shared * ((T + p.GW - 1) / p.GW));
  // experts with more than kWide tokens go to the tensor-core GEMM in units of
  // <= 128 tokens: at most P/(kWide+1) such experts
  p.wide = allow_wide && T > kWide;
  // one-token groups on the block-diagonal kernel when most touched experts
  // see one token: every expert at T = 1, and while the picks are at most
  // half the experts (DeepSeek-V3 shapes up to T = 16)
  p.single = allow_wide && grouped_b1_supported(d.fmt) && (T == 1 || 2 * p.P <= d.E);
  p.G1_max = p.single ? (int)std::min<int64_t>(d.E, p.P) + (T == 1 ? d.n_shared : 0) : 0;
  p.U_max = p.wide ? (int)(p.P / 128 + p.P / (kWide + 1) + 1 +
                           (int64_t)d.n_shared * ((T + 127) / 128))
                   : 0;
  // Down products split over K (p.DS parts, summed in order by the combine)
  // when the expected units (64-row tiles of the touched experts) are too few
  // for the persistent grid (~3 CTAs on each of 152 SMs) to come out even:
  // Mixtral shapes at T = 16 have 8 experts x 64 tiles = 512 units for 456
  // CTAs, so 56 CTAs would stream a second unit alone.  Only where every
  // position is produced by the grouped kernels (no one-token or tensor-core
  // groups), each part keeps >= 4 super-blocks.
  p.DS = 1;
  if (allow_wide && !p.wide && !p.single) {
    const int64_t units = (std::min<int64_t>(d.E, p.P) +
                           (int64_t)d.n_shared * ((T + p.GW - 1) / p.GW)) * (d.hidden / 64);
    constexpr int64_t kSlots = 3 * 152;
    while (p.DS < 4 && units * p.DS < 4 * kSlots && d.ffn / 256 >= 8 * p.DS) p.DS *= 2;
  }
  size_t o = 0;
  p.off_part = o;    o = align256(o + (size_t)p.KS * T * d.E * 4);
  p.off_logits = o;  o = align256(o + (size_t)T * d.E * 4);
  p.off_idx = o;     o = align256(o + (size_t)p.P * 4);
  p.off_gate = o;    o = align256(o + (size_t)p.P * 4);
  p.off_offsets = o; o = align256(o + (size_t)(d.E + 1) * 4);
  p.off_sorted = o;  o = align256(o + (size_t)p.P * 4);
  p.off_inv = o;     o = align256(o + (size_t)p.P * 4);
  p.off_tok = o;     o = align256(o + (size_t)p.NP * 4);
  p.off_groups = o;  o = align256(o + (size_t)p.G_max * 16);
  p.off_ngroups = o; o = align256(o + 16);
  p.off_h = o;       o = align256(o + (size_t)p.NP * d.ffn * 4);
  p.off_ypos = o;    o = align256(o + (size_t)p.DS * p.NP * d.hidden * 4);
  p.off_units = o;   o = align256(o + (size_t)std::max(p.U_max, 1) * 16);
  p.off_nunits = o;  o = align256(o + 16);
  // fp16 copies of the activations the streaming kernels read
  p.off_x16t = o;    o = align256(o + (size_t)T * d.hidden * 2);   // per token (bf16/fp32 x)
  p.off_xinvt = o;   o = align256(o + (size_t)T * 4);
  p.off_h16 = o;     o = align256(o + (size_t)p.NP * d.ffn * 2);   // per position
  p.off_hinv = o;    o = align256(o + (size_t)p.NP * 4);
  const size_t npw = p.wide ? (size_t)p.NP : 0;   // wide-path buffers only when possible
  p.off_x16 = o;     o = align256(o + npw * d.hidden * 2);
  p.off_xinv = o;    o = align256(o + npw * 4);
  p.off_g = o;       o = align256(o + npw * d.ffn * 4);
  p.off_u = o;       o = align256(o + npw * d.ffn * 4);
  p.off_g1 = o;      o = align256(o + (size_t)std::max(p.G1_max, 1) * 16);
  p.off_ng1 = o;     o = align256(o + 16);   // count, two work counters
  p.total = o;
  return p;
}

// ===========================================================================
// 1. router logits (fp32 SIMT tile 64 experts x 32 tokens, 4x4 per thread)
// ===========================================================================
// Activation i of x (fp32, bf16 or fp16) as fp32.  The dtype is fixed at
// compile time: loads in an unrolled loop are all issued before the first is
// used (a run-time dtype branch around each load keeps them one at a time).
template <int XDT>
__device__ __forceinline__ float act_t(const void* x, int64_t i) {
  if (XDT == DQ_F32) return __ldg((const float*)x + i);
  const unsigned short u = __ldg((const unsigned short*)x + i);
  if (XDT == DQ_BF16) return __uint_as_float((uint32_t)u << 16);
  return __half2float(__ushort_as_half(u));
}

// 16 bytes of activations (8 fp16 / bf16 or 4 fp32 values) as fp32.
template <int XDT>
__device__ __forceinline__ void act_vec(const uint4& r, float* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
  if (XDT == DQ_F32) {
#pragma unroll
    for (int j = 0; j < 4; ++j) f[j] = __uint_as_float(w[j]);
  } else if (XDT == DQ_BF16) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(w[j] << 16);
      f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 v = __half22float2(u32_as_h2(w[j]));
      f[2 * j] = v.x;
      f[2 * j + 1] = v.y;
    }
  }
}

template <int XDT>
__global__ void __launch_bounds__(128) router_logits_kernel(const float* __restrict__ Wr, int E,
                                                            int H, const void* __restrict__ x,
                                                            int T, int KS,
                                                            float* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  // two buffers: the next chunk's loads are in flight (in registers) while
  // this chunk is multiplied.  Loader mapping: a warp covers 8 consecutive
  // hidden indices of 4 consecutive experts (tokens), so that every global
  // load instruction reads whole 32-byte sectors and the transposed stores
  // hit 32 distinct banks (row pitches 68 and 36: 4 hh + e mod 32).
  __shared__ __align__(16) float Ws[2][32][64 + 4];
  __shared__ __align__(16) float Xs[2][32][32 + 4];
  const int e0 = blockIdx.x * 64, t0 = blockIdx.y * 32, ks = blockIdx.z;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int nch = H / 32;
  const int c_begin = (int)((int64_t)nch * ks / KS), c_end = (int)((int64_t)nch * (ks + 1) / KS);
  float wr[16], xr[8];
  auto load = [&](int c) {
    const int h0 = c * 32;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int i = tid + 128 * r;
      const int hh = (i & 7) | ((i >> 9) << 3), e = (i >> 3) & 63;
      wr[r] = (e0 + e < E) ? __ldg(Wr + (int64_t)(e0 + e) * H + h0 + hh) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = tid + 128 * r;
      const int hh = (i & 7) | ((i >> 8) << 3), t = (i >> 3) & 31;
      xr[r] = (t0 + t < T) ? act_t<XDT>(x, (int64_t)(t0 + t) * H + h0 + hh) : 0.f;
    }
  };
  auto store = [&](int b) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int i = tid + 128 * r;
      Ws[b][(i & 7) | ((i >> 9) << 3)][(i >> 3) & 63] = wr[r];
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int i = tid + 128 * r;
      Xs[b][(i & 7) | ((i >> 8) << 3)][(i >> 3) & 31] = xr[r];
    }
  };
  float acc[4][4] = {};
  if (c_begin < c_end) {
    load(c_begin);
    store(0);
  }
  __syncthreads();
  for (int c = c_begin; c < c_end; ++c) {
    const int b = (c - c_begin) & 1;
    const bool more = c + 1 < c_end;
    if (more) load(c + 1);
#pragma unroll 8
    for (int hh = 0; hh < 32; ++hh) {
      const float4 xv = *(const float4*)&Xs[b][hh][ty * 4];
      const float4 wv = *(const float4*)&Ws[b][hh][tx * 4];
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(xa[a], wa[q], acc[a][q]);
    }
    // the other buffer was last read before the previous barrier
    if (more) store(b ^ 1);
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int t = t0 + ty * 4 + a;
    if (t >= T) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = e0 + tx * 4 + q;
      if (e < E) part[((int64_t)ks * T + t) * E + e] = acc[a][q];
    }
  }
}

// Few tokens (T <= 32): the router is a GEMV over the 7.3 MB of W_r
// (DeepSeek); warp w of CTA (b, ks) streams expert row 8b + w over hidden
// chunk ks with 16-byte loads against the chunk of every token's x, staged
// once per CTA in shared memory, and writes part[ks][t][e] like the tiled
// kernel.  TMAX tokens at most, CHUNK hidden values per chunk.
template <int TMAX, int CHUNK, int XDT>
__global__ void __launch_bounds__(256) router_stream_kernel(const float* __restrict__ Wr, int E,
                                                            int H, const void* __restrict__ x,
                                                            int T, float* __restrict__ part,
                                                            int nc) {
  pdl_wait();
  pdl_trigger();
  // CTA (b, ks) sums hidden chunks ks*nc .. ks*nc + nc - 1 (the layer: one
  // chunk per CTA, partials summed by the top-k; dq_moe_router: every chunk,
  // the partial is the logit)
  __shared__ __align__(16) float xs[TMAX][CHUNK];
  const int ks = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  const bool active = e < E;
  constexpr int kES = XDT == DQ_F32 ? 4 : 2;        // bytes per activation
  constexpr int kVE = 16 / kES;                     // activations per 16-byte load
  constexpr int kVec = TMAX * CHUNK / kVE / 256;
  constexpr int kW = CHUNK / 4 / 32;                // float4 of W_r per lane
  float acc[TMAX] = {};
  for (int ci = 0; ci < nc; ++ci) {
    const int h0 = (ks * nc + ci) * CHUNK;
    if (h0 >= H) break;                             // uniform over the CTA
    const int n = min(CHUNK, H - h0);               // multiple of 32
    // every load of the chunk is issued before any is used: the chunk of x
    // (16-byte loads, at most kVec per thread) and this warp's row of W_r
    const int nv = n / kVE, total = T * nv;
    uint4 xr[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int i = threadIdx.x + 256 * j;
      if (i < total) {
        const int t = i / nv, v = i - t * nv;
        xr[j] = __ldg((const uint4*)((const char*)x + ((int64_t)t * H + h0 + v * kVE) * kES));
      }
    }
    float4 wv[kW];
    if (active) {
      const float4* w = (const float4*)(Wr + (int64_t)e * H + h0);
#pragma unroll
      for (int j = 0; j < kW; ++j)
        wv[j] = lane + 32 * j < n / 4 ? __ldcs(w + lane + 32 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (ci > 0) __syncthreads();                    // the previous chunk's reads of xs
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int i = threadIdx.x + 256 * j;
      if (i < total) {
        const int t = i / nv, v = i - t * nv;
        float f[kVE];
        act_vec<XDT>(xr[j], f);
#pragma unroll
        for (int q = 0; q < kVE; q += 4)
          *(float4*)&xs[t][v * kVE + q] = make_float4(f[q], f[q + 1], f[q + 2], f[q + 3]);
      }
    }
    __syncthreads();
    if (active) {
#pragma unroll
      for (int j = 0; j < kW; ++j) {
        if (lane + 32 * j < n / 4) {
          const float4 w4 = wv[j];
#pragma unroll
          for (int t = 0; t < TMAX; ++t) {
            if (t < T) {
              const float4 xv = *(const float4*)&xs[t][4 * (lane + 32 * j)];
              acc[t] = fmaf(w4.x, xv.x, acc[t]);
              acc[t] = fmaf(w4.y, xv.y, acc[t]);
              acc[t] = fmaf(w4.z, xv.z, acc[t]);
              acc[t] = fmaf(w4.w, xv.w, acc[t]);
            }
          }
        }
      }
    }
  }
  if (!active) return;
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    if (t < T) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) part[((int64_t)ks * T + t) * E + e] = v;
    }
  }
}

// ===========================================================================
// 2. top-k + gates: one warp per token
// ===========================================================================
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}

// A float's bits as an unsigned key with the float's order (not NaN), and
// back.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Compare-exchange of (value, index) pairs a, b into descending order.
__device__ __forceinline__ void cas_desc(float& va, int& ia, float& vb, int& ib) {
  if (better(vb, ib, va, ia)) {
    const float tv = va;
    const int ti = ia;
    va = vb;
    ia = ib;
    vb = tv;
    ib = ti;
  }
}

// Selection of token t by one warp from its logits v (lane holds experts
// lane + 32 j, j < 8; -inf / 0x7fffffff past E): each lane first sorts its 8
// candidates (descending logit, lowest expert index first on ties) with a
// sorting network, then k rounds take the best of the 32 lanes' heads (two
// warp reductions) and advance the winning lane's head.  Lanes i < k compute the gate
// of slot i (softmax over all E renormalised over the selection) and write
// the index and the gate, and the index to sidx (nullable, shared memory).
__device__ __forceinline__ void topk_select(float (&v)[8], int (&id)[8], int k, int t, int lane,
                                            int32_t* __restrict__ idx, float* __restrict__ gate,
                                            int* sidx) {
  // Batcher's odd-even merge sort of 8 (19 compare-exchanges)
#define DQ_CAS(a, b) cas_desc(v[a], id[a], v[b], id[b])
  DQ_CAS(0, 1); DQ_CAS(2, 3); DQ_CAS(4, 5); DQ_CAS(6, 7);
  DQ_CAS(0, 2); DQ_CAS(1, 3); DQ_CAS(4, 6); DQ_CAS(5, 7);
  DQ_CAS(1, 2); DQ_CAS(5, 6);
  DQ_CAS(0, 4); DQ_CAS(1, 5); DQ_CAS(2, 6); DQ_CAS(3, 7);
  DQ_CAS(2, 4); DQ_CAS(3, 5);
  DQ_CAS(1, 2); DQ_CAS(3, 4); DQ_CAS(5, 6);
#undef DQ_CAS
  float my_v = -INFINITY, top = -INFINITY;
  int my_i = 0;
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    if (r >= k) break;
    // the best head: the largest logit (as an order-preserving key), then the
    // lowest expert index among the heads holding it (a lane's equal logits
    // are in index order, so the lowest such index is a head)
    const uint32_t key = order_key(v[0]);
    const uint32_t mk = __reduce_max_sync(0xffffffffu, key);
    const int bi = (int)__reduce_min_sync(0xffffffffu, key == mk ? (uint32_t)id[0] : 0xffffffffu);
    const float bv = order_key_inv(mk);
    if (r == 0) top = bv;
    if (lane == r) {
      my_v = bv;
      my_i = bi;
    }
    if (id[0] == bi) {   // the winning lane's next candidate moves up
#pragma unroll
      for (int j = 0; j < 7; ++j) {
        v[j] = v[j + 1];
        id[j] = id[j + 1];
      }
      v[7] = -INFINITY;
      id[7] = 0x7fffffff;
    }
  }
  // softmax over all E renormalised over the selection
  const float ex = lane < k ? expf(my_v - top) : 0.f;
  float z = ex;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  if (lane < k) {
    idx[(int64_t)t * k + lane] = my_i;
    gate[(int64_t)t * k + lane] = ex / z;
    if (sidx) sidx[t * k + lane] = my_i;
  }
}

// Top-k of token t by one warp (lane: this thread's lane) from the router's
// KS partial sums.
__device__ __forceinline__ void topk_warp(const float* __restrict__ part, int KS, int T, int E,
                                          int k, int t, int lane, float* __restrict__ logits,
                                          int32_t* __restrict__ idx, float* __restrict__ gate) {
  float v[8];
  int id[8];
  // sum the KS partials of this lane's 8 experts in a fixed order (q
  // ascending); the 8 experts' loads of one q are independent and in flight
  // together, so KS rounds of memory latency rather than 8 * KS
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = 0.f;
  for (int q = 0; q < KS; ++q) {
    const float* pq = part + ((int64_t)q * T + t) * E;
    float a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      a[j] = e < E ? __ldg(pq + e) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] += a[j];
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = lane + 32 * j;
    id[j] = e;
    if (e < E) {
      if (logits) logits[(int64_t)t * E + e] = v[j];
    } else {
      v[j] = -INFINITY;
      id[j] = 0x7fffffff;
    }
  }
  topk_select(v, id, k, t, lane, idx, gate, nullptr);
}

__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ part, int KS, int T,
                                                   int E, int k, float* __restrict__ logits,
                                                   int32_t* __restrict__ idx,
                                                   float* __restrict__ gate) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t < T) topk_warp(part, KS, T, E, k, t, threadIdx.x & 31, logits, idx, gate);
}

// ===========================================================================
// 3. stable permute + work groups: one CTA of 1024 threads
// ===========================================================================
// Exclusive scan of v over threads 0..255 of the CTA (warp shuffles, then the
// eight warp totals): returns the sum of v over lower threads; *total gets the
// sum over all 256.  Every thread of the CTA calls it (two barriers).
__device__ __forceinline__ int block_scan256(int v, int* wsum, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int inc = tid < 256 ? v : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (tid < 256 && lane == 31) wsum[warp] = inc;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int c = wsum[w];
    if (w < warp) before += c;
    all += c;
  }
  __syncthreads();   // wsum may be reused by the next call
  *total = all;
  return tid < 256 ? before + inc - v : 0;
}

// The same for three values at once (one pair of barriers).
__device__ __forceinline__ int3 block_scan256x3(int3 v, int3* wsum3, int3* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int3 inc = tid < 256 ? v : make_int3(0, 0, 0);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nx = __shfl_up_sync(0xffffffffu, inc.x, o);
    const int ny = __shfl_up_sync(0xffffffffu, inc.y, o);
    const int nz = __shfl_up_sync(0xffffffffu, inc.z, o);
    if (lane >= o) {
      inc.x += nx;
      inc.y += ny;
      inc.z += nz;
    }
  }
  if (tid < 256 && lane == 31) wsum3[warp] = inc;
  __syncthreads();
  int3 before = make_int3(0, 0, 0), all = make_int3(0, 0, 0);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int3 c = wsum3[w];
    if (w < warp) {
      before.x += c.x;
      before.y += c.y;
      before.z += c.z;
    }
    all.x += c.x;
    all.y += c.y;
    all.z += c.z;
  }
  __syncthreads();   // wsum3 may be reused by the next call
  *total = all;
  if (tid >= 256) return make_int3(0, 0, 0);
  return make_int3(before.x + inc.x - v.x, before.y + inc.y - v.y, before.z + inc.z - v.z);
}

// Few tokens: the permute CTA also converts x to fp16 with a power-of-two
// scale per token (the x16 prep of the expert kernels), saving a launch on
// the decode path.  Rows of at most 8192 values.
template <int XDT>
__device__ __forceinline__ void x16_rows_cta_t(const void* x, int T, int K, __half* out,
                                               float* inv, float* red) {
  for (int row = 0; row < T; ++row) {
    const int64_t base = (int64_t)row * K;
    float v[8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {                  // K <= 8192
      const int k = threadIdx.x + 1024 * i;
      v[i] = k < K ? act_t<XDT>(x, base + k) : 0.f;
      amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = 0.f;
    for (int w = 0; w < 32; ++w) amax = fmaxf(amax, red[w]);
    __syncthreads();
    float sc, iv;
    pow2_scale(amax, sc, iv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int k = threadIdx.x + 1024 * i;
      if (k < K) out[base + k] = __float2half_rn(v[i] * sc);
    }
    if (threadIdx.x == 0) inv[row] = iv;
  }
}
__device__ __forceinline__ void x16_rows_cta(const void* x, int xdt, int T, int K, __half* out,
                                             float* inv, float* red) {
  if (xdt == DQ_F32) x16_rows_cta_t<DQ_F32>(x, T, K, out, inv, red);
  else if (xdt == DQ_BF16) x16_rows_cta_t<DQ_BF16>(x, T, K, out, inv, red);
  else x16_rows_cta_t<DQ_F16>(x, T, K, out, inv, red);
}
// tk (nullable): top-k of the T <= 32 tokens first, one warp each, from the
// router partials (tk->part, tk->KS), writing idx, gate and logits; the
// permute then reads idx back (coherent loads: written by this CTA).
struct TopkIn {
  const float* part;
  int KS;
  float* logits;
  float* gate;
};

__global__ void __launch_bounds__(1024) permute_kernel(int32_t* idx, int T,
                                                       int k, int E, int n_shared, int gw,
                                                       int32_t* __restrict__ offsets,
                                                       int32_t* __restrict__ sorted,
                                                       int32_t* __restrict__ inv,
                                                       int32_t* __restrict__ tok,
                                                       int4* __restrict__ groups,
                                                       int32_t* __restrict__ n_groups,
                                                       int4* __restrict__ units,
                                                       int32_t* __restrict__ n_units,
                                                       const void* __restrict__ cx, int cxdt,
                                                       int cK, __half* __restrict__ cx16,
                                                       float* __restrict__ cxinv, TopkIn tk,
                                                       int4* __restrict__ groups1,
                                                       int32_t* __restrict__ n_groups1) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  __shared__ int wsum[8];
  __shared__ int3 wsum3[8];
  __shared__ int cnt[256];
  __shared__ int off[257];
  __shared__ int run[256];
  __shared__ int cntw[32][256];   // per-warp counts; first the top-k's logits [T][E]
  __shared__ int gsc[257];
  __shared__ int usc[257];
  __shared__ int osc[257];
  __shared__ int sidx[256];       // the top-k's indices (T * k <= 256)
  __shared__ int stok[256];       // the token of an expert's pair, for experts with one pair
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = T * k;
  const bool own = tk.part != nullptr;   // the indices are chosen here: read them from sidx
  if (T == 1 && own && groups1 && !units && !cx16) {
    // one token, every selected expert a one-token group (the decode step):
    // the logits as below (every thread sums the partials of its experts in
    // the same order: bit-identical), then warp 0 alone, no further block
    // barriers; every output the general path writes for this case is
    // written: an expert's position is its rank among the selected experts
    // (expert order), its pair's token 0.
    float* lg = (float*)&cntw[0][0];
    for (int e = tid; e < E; e += 1024) {
      const float* pp = tk.part + e;
      float a = 0.f;
      for (int q0 = 0; q0 < tk.KS; q0 += 8) {
        float b[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] = q0 + j < tk.KS ? __ldcg(pp + (int64_t)(q0 + j) * E) : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (q0 + j < tk.KS) a += b[j];
      }
      lg[e] = a;
      if (tk.logits) tk.logits[e] = a;
    }
    __syncthreads();
    if (warp != 0) return;
    float v[8];
    int id[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = lane + 32 * j;
      v[j] = e < E ? lg[e] : -INFINITY;
      id[j] = e < E ? e : 0x7fffffff;
    }
    topk_select(v, id, k, 0, lane, idx, tk.gate, sidx);
    __syncwarp();
    int sel[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) sel[i] = i < k ? sidx[i] : 0x7fffffff;
    if (lane < k) {
      const int e = sel[lane];
      int rank = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) rank += sel[i] < e ? 1 : 0;
      if (sorted) sorted[rank] = lane;
      if (inv) inv[lane] = rank;
      if (tok) tok[rank] = 0;
      groups1[rank] = make_int4(e, rank, 0, 0);
    }
    for (int sh = lane; sh < n_shared; sh += 32) {
      if (tok) tok[P + sh] = 0;
      groups1[k + sh] = make_int4(E + sh, P + sh, 0, 0);
    }
    if (offsets)
      for (int e = lane; e <= E; e += 32) {
        int c = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) c += sel[i] < e ? 1 : 0;
        offsets[e] = c;
      }
    if (lane == 0) {
      if (groups) *n_groups = 0;
      n_groups1[0] = k + n_shared;
      n_groups1[1] = 0;   // the one-token kernels' work counters
      n_groups1[2] = 0;
    }
    return;
  }
  if (own) {
    // logits of the T <= 32 tokens: every thread sums the KS partials of its
    // (token, expert) entries in a fixed order (q ascending), all loads in
    // flight together; then one warp per token selects from shared memory
    float* lg = (float*)&cntw[0][0];
    const int n = T * E;
    const int64_t qstride = (int64_t)T * E;
    for (int i = tid; i < n; i += 1024) {
      const float* pp = tk.part + i;
      float v = 0.f;
      for (int q0 = 0; q0 < tk.KS; q0 += 8) {
        float a[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          a[j] = q0 + j < tk.KS ? __ldcg(pp + (q0 + j) * qstride) : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (q0 + j < tk.KS) v += a[j];
      }
      lg[i] = v;
      if (tk.logits) tk.logits[i] = v;
    }
    __syncthreads();
    if (warp < T) {
      float v[8];
      int id[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int e = lane + 32 * j;
        id[j] = e < E ? e : 0x7fffffff;
        v[j] = e < E ? lg[warp * E + e] : -INFINITY;
      }
      topk_select(v, id, k, warp, lane, idx, tk.gate, sidx);
    }
    __syncthreads();
  }
  if (cx16) x16_rows_cta(cx, cxdt, T, cK, cx16, cxinv, red);
  if (tid < 256) cnt[tid] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += 1024) atomicAdd(&cnt[own ? sidx[p] : __ldcg(idx + p)], 1);
  __syncthreads();
  // exclusive scan of counts (E <= 256)
  {
    int total;
    const int ex = block_scan256(tid < E ? cnt[tid] : 0, wsum, &total);
    if (tid < 256) off[tid] = ex;
    if (tid == 0) off[256] = total;
    __syncthreads();
  }
  if (tid <= E && offsets) offsets[tid] = off[tid];
  if (tid < E) run[tid] = off[tid];
  __syncthreads();
  // stable scatter, 1024 pairs per round: rank inside the warp by match_any,
  // warps ordered through per-warp counts
  for (int base = 0; base < P; base += 1024) {
    const int nw = min(32, (P - base + 31) >> 5);   // warps holding pairs this round
    for (int i = tid; i < nw * 256; i += 1024) (&cntw[0][0])[i] = 0;
    __syncthreads();
    const int p = base + tid;
    const int e = (p < P) ? (own ? sidx[p] : __ldcg(idx + p)) : 256;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (p < P && rank == 0) cntw[warp][e] = __popc(peers);
    __syncthreads();
    if (tid < E) {
      int s = run[tid];
      for (int w = 0; w < nw; ++w) {
        const int c = cntw[w][tid];
        cntw[w][tid] = s;
        s += c;
      }
      run[tid] = s;
    }
    __syncthreads();
    if (p < P) {
      const int pos = cntw[warp][e] + rank;
      sorted[pos] = p;
      if (inv) inv[p] = pos;
      if (tok) tok[pos] = p / k;
      if (cnt[e] == 1) stok[e] = p / k;
    }
    __syncthreads();
  }
  if (!groups) return;
  // shared-expert positions follow the routed ones: P + s*T + t
  for (int i = tid; i < n_shared * T; i += 1024) tok[P + i] = i % T;
  // narrow groups of <= gw columns per expert (experts with <= kWide tokens),
  // wide units of <= 128 columns (more tokens); experts in order, then the
  // shared experts (all T tokens)
  // with groups1, experts that received exactly one pair form the one-token
  // list instead (expert, position, token), and so do the shared experts at
  // T = 1
  const bool wide_ok = units != nullptr;
  const bool one_ok = groups1 != nullptr;
  {
    const int n = (tid < E) ? cnt[tid] : 0;
    const bool w = wide_ok && n > kWide;
    const bool one = one_ok && n == 1;
    int3 tot;
    const int3 ex = block_scan256x3(
        make_int3((w || one) ? 0 : (n + gw - 1) / gw, w ? (n + 127) / 128 : 0, one ? 1 : 0),
        wsum3, &tot);
    if (tid < 256) {
      gsc[tid] = ex.x;
      usc[tid] = ex.y;
      osc[tid] = ex.z;
    }
    if (tid == 0) {
      gsc[256] = tot.x;
      usc[256] = tot.y;
      osc[256] = tot.z;
    }
    __syncthreads();
  }
  if (tid < E) {
    const int n = cnt[tid];
    if (wide_ok && n > kWide) {
      for (int j = 0; j * 128 < n; ++j)
        units[usc[tid] + j] = make_int4(tid, off[tid] + 128 * j, min(128, n - 128 * j), 0);
    } else if (one_ok && n == 1) {
      // the pair's token (recorded by the scatter above)
      groups1[osc[tid]] = make_int4(tid, off[tid], stok[tid], 0);
    } else {
      for (int j = 0; j * gw < n; ++j)
        groups[gsc[tid] + j] = make_int4(tid, off[tid] + gw * j, min(gw, n - gw * j), 0);
    }
  }
  const int nr = gsc[E], ur = usc[E], orr = osc[E];
  const bool sh_one = one_ok && T == 1;
  const bool sh_wide = wide_ok && T > kWide;
  const int per = sh_wide ? (T + 127) / 128 : (T + gw - 1) / gw;
  const int width = sh_wide ? 128 : gw;
  for (int i = tid; i < n_shared * per; i += 1024) {
    const int s = i / per, j = i % per;
    const int4 g = make_int4(E + s, P + s * T + width * j, min(width, T - width * j), 0);
    if (sh_one) groups1[orr + s] = make_int4(E + s, P + s, 0, 0);
    else if (sh_wide) units[ur + i] = g;
    else groups[nr + i] = g;
  }
  if (tid == 0) {
    *n_groups = nr + ((sh_wide || sh_one) ? 0 : n_shared * per);
    if (wide_ok) *n_units = ur + (sh_wide ? n_shared * per : 0);
    if (one_ok) {
      n_groups1[0] = orr + (sh_one ? n_shared : 0);
      n_groups1[1] = 0;   // the one-token kernels' work counters
      n_groups1[2] = 0;
    }
  }
}

// ===========================================================================
// 4/5. persistent grouped streaming GEMV (gate/up with SwiGLU, or down)
// ===========================================================================
struct GroupedParams {
  // TMA maps over the stacked matrices as [experts*rows][row_bytes/2]:
  // routed a (gate or down), routed b (up), shared a, shared b.  Boxes are
  // BOX x 32 rows (gate/up) or BOX x 64 rows (down).
  CUtensorMap map_a, map_b, map_sa, map_sb;
  int rows_per_expert; // F (gate/up) or H (down)
  const uint8_t* Wa;   // routed: W_gate (gate/up) or W_down (down), E stacked
  const uint8_t* Wb;   // routed: W_up (gate/up only)
  const uint8_t* Sa;   // shared experts, same roles
  const uint8_t* Sb;
  int64_t mat_bytes;   // bytes of one expert matrix
  int64_t row_bytes;
  int nsb;             // super-blocks per row (K / 256)
  int E;
  const int4* groups;
  const int* n_groups;
  const int* tok;      // position -> token (gate/up gather)
  const void* xbase;   // gate/up: x [T][H]; down: h [NP][F]
  int xdt;
  int64_t xstride;     // elements per x / h row
  float* out;          // gate/up: h [NP][F]; down: ypos [NP][H]
  int64_t out_stride;
  const float* colinv; // 1/scale of each column's fp16 activations (nullable: 1)
  const int* coltok;   // colinv index of position pos: coltok[pos] (nullable: pos)
  int tiles;           // tiles per group
  int ksplit;          // down only: K parts per tile, part q written at out + q * part_stride
  int64_t part_stride;
  int nstage;
  // expert streaming (both nullable): routed expert e's matrices sit in slot
  // slot_of[e] of the stacked maps; only units of experts with
  // phase_of[e] == phase run (shared experts run in phase 0)
  const int* slot_of;
  const int8_t* phase_of;
  int phase;
};

// Whether a unit of group grp runs in this launch, and its matrix index in
// the routed or shared maps.
__device__ __forceinline__ bool unit_in_phase(const GroupedParams& p, int4 grp, int& mat) {
  const bool shared = grp.x >= p.E;
  if (shared) {
    mat = grp.x - p.E;
    return p.phase_of == nullptr || p.phase == 0;
  }
  mat = p.slot_of ? __ldg(p.slot_of + grp.x) : grp.x;
  return p.phase_of == nullptr || __ldg(p.phase_of + grp.x) == p.phase;
}

// NT: activation tiles of 8 columns per unit (groups hold <= 8*NT columns).
template <int FMT, bool GATEUP, int NT>
__global__ void __launch_bounds__(kThreads) grouped_kernel(const __grid_constant__ GroupedParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  using L = Layout<FMT>;
  constexpr int NC = 8 * NT;
  const SmemPlan plan = make_plan<FMT>(p.nstage, NC, 1);
  uint64_t* full = (uint64_t*)(smem + plan.off_bar);
  uint64_t* empty = full + plan.nstage;
  uint8_t* wbuf = smem + plan.off_w;
  uint8_t* xbuf = smem + plan.off_x;
  float* xinv = (float*)(smem + plan.off_xinv);
  float* ex = (float*)(smem + plan.off_red);   // [64][NC] gate/up exchange

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_group = p.tiles * p.ksplit;
  const int n_units = __ldg(p.n_groups) * per_group;
  const int nchunk = (p.nsb + L::C - 1) / L::C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < plan.nstage; ++s) {
      mbar_init(&full[s], full_arrivals(p.xdt));
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  init_xinv(xinv, plan.nstage * NC, p.xdt);
  __syncthreads();

  if (warp == 0) {
    // ------------------------------ loader ------------------------------
    const uint64_t pol = l2_evict_first_policy();
    int gc = 0, ls = 0;
    uint32_t lph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const int4 grp = __ldg(p.groups + u / per_group);
      const int tile = (u % per_group) / p.ksplit, part = u % p.ksplit;
      const bool shared = grp.x >= p.E;
      int eid;
      if (!unit_in_phase(p, grp, eid)) continue;
      // first stacked row of the tile: gate/up -> 32 gate rows then the same 32 up rows
      const int grow = eid * p.rows_per_expert + (GATEUP ? tile * 32 : tile * 64);
      const CUtensorMap* ma = shared ? &p.map_sa : &p.map_a;
      const CUtensorMap* mb = shared ? &p.map_sb : &p.map_b;
      XSrc xs;
      xs.dtype = p.xdt;
      xs.col_stride = p.xstride;
      if (GATEUP) {
        xs.base = p.xbase;
        xs.rows = p.tok + grp.y;
      } else {
        xs.base = (const __half*)p.xbase + (int64_t)grp.y * p.xstride;
        xs.rows = nullptr;
      }
      const int c_end = (part + 1) * nchunk / p.ksplit;
      for (int c = part * nchunk / p.ksplit; c < c_end && ok; ++c, ++gc) {
        if (gc >= plan.nstage) ok = mbar_wait(&empty[ls], lph ^ 1);
        if (!ok) break;
        const int s = ls;
        if (++ls == plan.nstage) {
          ls = 0;
          lph ^= 1;
        }
        const int c0 = c * L::C;
        const int ncs = min(L::C, p.nsb - c0);
        const int64_t a = ((int64_t)c0 * L::SBB) & ~(int64_t)15;
        if (lane == 0) {
          uint8_t* wst = wbuf + s * L::W_STAGE;
          mbar_arrive_expect_tx(&full[s], L::W_STAGE);
          if (GATEUP) {
            tma_load_2d(wst, ma, (int)(a >> 1), grow, &full[s], pol);
            tma_load_2d(wst + 32 * L::ROW_PITCH, mb, (int)(a >> 1), grow, &full[s], pol);
          } else {
            tma_load_2d(wst, ma, (int)(a >> 1), grow, &full[s], pol);
          }
        }
        stage_x<FMT>(xs, grp.z, (int64_t)c0 * 256, ncs, xbuf + s * NC * L::XCOL, xinv + s * NC,
                     lane, &full[s]);
      }
    }
  } else {
    // ----------------------------- consumers -----------------------------
    const int cw = warp - 1;
    const int g = lane >> 2, t = lane & 3;
    int cs = 0;
    uint32_t cph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const int4 grp = __ldg(p.groups + u / per_group);
      const int tile = (u % per_group) / p.ksplit, part = u % p.ksplit;
      const int ncols = grp.z;
      int mat_unused;
      if (!unit_in_phase(p, grp, mat_unused)) continue;   // the loader skips it too
      const bool f16 = p.xdt == DQ_F16;      // fp16 input carries no scale
      float acc[NT][4] = {};
      float accs[NT][2][4] = {};             // fp16 input: running accumulator pairs
      const int c_end = (part + 1) * nchunk / p.ksplit;
      for (int c = part * nchunk / p.ksplit; c < c_end; ++c) {
        const int s = cs;
        const uint32_t par = cph;
        if (++cs == plan.nstage) {
          cs = 0;
          cph ^= 1;
        }
        // after a timed-out wait the warp keeps walking the same units (no
        // further waits, no reads) so every warp still meets the barriers
        ok = ok && mbar_wait(&full[s], par);
        if (!ok) continue;
        const uint32_t o = order_after_wait(0u);   // stage reads follow the wait
        const int c0 = c * L::C;
        const int ncs = min(L::C, p.nsb - c0);
        const int delta = (int)(((int64_t)c0 * L::SBB) & 15);
        const uint32_t wst =
            smem_u32(wbuf + s * L::W_STAGE) + (16 * cw + g) * L::ROW_PITCH + delta + o;
        // this lane's activation column in each 8-column tile (column 0 past the group)
        uint32_t xcol[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int col = 8 * nt + g;
          xcol[nt] = smem_u32(xbuf + (s * NC + (col < ncols ? col : 0)) * L::XCOL) + o;
        }
        if constexpr (SBDot<FMT>::kRowScale) {
          for (int j = 0; j < ncs; ++j) {
            float d[NT][2][4] = {};
            float r0, r8;
            SBDot<FMT>::template run<NT, true>(wst + j * L::SBB, 8 * L::ROW_PITCH, xcol, j * 256,
                                               t, d, r0, r8);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float c0 = f16 ? 1.f : xinv[s * NC + 8 * nt + 2 * t];
              const float c1 = f16 ? 1.f : xinv[s * NC + 8 * nt + 2 * t + 1];
              fold_tile(acc[nt], d[nt], r0, r8, c0, c1);
            }
          }
        } else if (f16) {
          for (int j = 0; j < ncs; ++j)
            SBDot<FMT>::template run<NT>(wst + j * L::SBB, 8 * L::ROW_PITCH, xcol, j * 256, t, accs);
        } else {
          float part[NT][2][4] = {};
          for (int j = 0; j < ncs; ++j)
            SBDot<FMT>::template run<NT>(wst + j * L::SBB, 8 * L::ROW_PITCH, xcol, j * 256, t, part);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            fold_tile(acc[nt], part[nt], 1.f, 1.f, xinv[s * NC + 8 * nt + 2 * t],
                      xinv[s * NC + 8 * nt + 2 * t + 1]);
        }
        keep_before_release<NT * 4>(&acc[0][0]);    // ... and finish before its release
        keep_before_release<NT * 8>(&accs[0][0][0]);
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(&empty[s]);
      }
      if (!SBDot<FMT>::kRowScale && f16) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[nt][i] = accs[nt][0][i] + accs[nt][1][i];
      }
      // undo the activation scale of each column
      if (p.colinv) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int c0 = 8 * nt + 2 * t;
          const int p0 = grp.y + min(c0, ncols - 1), p1 = grp.y + min(c0 + 1, ncols - 1);
          const float i0 = __ldg(p.colinv + (p.coltok ? __ldg(p.coltok + p0) : p0));
          const float i1 = __ldg(p.colinv + (p.coltok ? __ldg(p.coltok + p1) : p1));
          acc[nt][0] *= i0;
          acc[nt][1] *= i1;
          acc[nt][2] *= i0;
          acc[nt][3] *= i1;
        }
      }
      if (!GATEUP) {
        const int ra = tile * 64 + 16 * cw + g, rb = ra + 8;
        float* o = p.out + part * p.part_stride + (int64_t)grp.y * p.out_stride;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int c0 = 8 * nt + 2 * t, c1 = c0 + 1;
          if (c0 < ncols) {
            o[(int64_t)c0 * p.out_stride + ra] = acc[nt][0];
            o[(int64_t)c0 * p.out_stride + rb] = acc[nt][2];
          }
          if (c1 < ncols) {
            o[(int64_t)c1 * p.out_stride + ra] = acc[nt][1];
            o[(int64_t)c1 * p.out_stride + rb] = acc[nt][3];
          }
        }
      } else {
        // rows 0..31 hold gate, rows 32..63 the matching up rows
        const int ra = 16 * cw + g, rb = ra + 8;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int c0 = 8 * nt + 2 * t, c1 = c0 + 1;
          ex[ra * NC + c0] = acc[nt][0];
          ex[ra * NC + c1] = acc[nt][1];
          ex[rb * NC + c0] = acc[nt][2];
          ex[rb * NC + c1] = acc[nt][3];
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const int ct = threadIdx.x - 32;
        for (int i = ct; i < 32 * ncols; i += 128) {
          const int r = i & 31, col = i >> 5;
          const float gv = ex[r * NC + col], uv = ex[(32 + r) * NC + col];
          // silu(g) = g / (1 + exp(-g)); for g < -88 exp overflows to inf and
          // the quotient is -0, never NaN
          const float h = gv / (1.f + expf(-gv)) * uv;
          p.out[(int64_t)(grp.y + col) * p.out_stride + tile * 32 + r] = h;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
    }
  }
}

// ===========================================================================
// 6. combine: y[t] = sum_i gate[t][i] * ypos[pos(t,i)] + sum_s ypos[P + sT + t]
// where a position's value is the sum of its `parts` K-split parts (part q at
// ypos + q * part_stride), added in part order.
// ===========================================================================
__device__ __forceinline__ float4 ypos_value(const float* __restrict__ ypos, int64_t pos, int H,
                                             int h4, int parts, int64_t part_stride) {
  float4 v = __ldg((const float4*)(ypos + pos * H) + h4);
  for (int q = 1; q < parts; ++q) {
    const float4 w = __ldg((const float4*)(ypos + q * part_stride + pos * H) + h4);
    v.x += w.x;
    v.y += w.y;
    v.z += w.z;
    v.w += w.w;
  }
  return v;
}

template <bool PARTS>
__device__ __forceinline__ void combine_one(const float* __restrict__ ypos,
                                            const int32_t* __restrict__ inv,
                                            const float* __restrict__ gate, int T, int k, int H,
                                            int n_shared, int parts, int64_t part_stride, int64_t i,
                                            float* __restrict__ y) {
  const int H4 = H / 4;
  const int64_t P = (int64_t)T * k;
  const int t = (int)(i / H4), h4 = (int)(i % H4);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < k; ++s) {
    const int pos = __ldg(inv + (int64_t)t * k + s);
    const float g = __ldg(gate + (int64_t)t * k + s);
    const float4 v = PARTS ? ypos_value(ypos, pos, H, h4, parts, part_stride)
                           : __ldg((const float4*)(ypos + (int64_t)pos * H) + h4);
    acc.x = fmaf(g, v.x, acc.x);
    acc.y = fmaf(g, v.y, acc.y);
    acc.z = fmaf(g, v.z, acc.z);
    acc.w = fmaf(g, v.w, acc.w);
  }
  for (int s = 0; s < n_shared; ++s) {
    const int64_t pos = P + (int64_t)s * T + t;
    const float4 v = PARTS ? ypos_value(ypos, pos, H, h4, parts, part_stride)
                           : __ldg((const float4*)(ypos + pos * H) + h4);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  ((float4*)y)[i] = acc;
}

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ypos,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ gate, int T,
                                                      int k, int H, int n_shared, int parts,
                                                      int64_t part_stride,
                                                      float* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)T * (H / 4);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (parts == 1)
      combine_one<false>(ypos, inv, gate, T, k, H, n_shared, 1, 0, i, y);
    else
      combine_one<true>(ypos, inv, gate, T, k, H, n_shared, parts, part_stride, i, y);
  }
}

// ===========================================================================
// host side
// ===========================================================================
namespace {

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

int qk(int fmt) { return fmt == DQ_Q8_0 ? 32 : 256; }
int blk_bytes(int fmt) {
  return (fmt == DQ_Q4_K || fmt == DQ_NVFP4) ? 144 : fmt == DQ_Q6_K ? 210 : 34;
}

template <int FMT, bool GATEUP, int NT>
int launch_grouped(const GroupedParams& gp_in, int units_max, cudaStream_t s, int E_map,
                   int n_shared) {
  using L = Layout<FMT>;
  GroupedParams gp = gp_in;
  const uint32_t box_rows = GATEUP ? 32 : 64;
  const uint64_t rpe = (uint64_t)gp.rows_per_expert;
  if (!make_weight_tmap(&gp.map_a, gp.Wa, rpe * E_map, gp.row_bytes, L::BOX, box_rows))
    return DQ_ERR_CUDA;
  if (GATEUP && !make_weight_tmap(&gp.map_b, gp.Wb, rpe * E_map, gp.row_bytes, L::BOX, box_rows))
    return DQ_ERR_CUDA;
  if (n_shared > 0) {
    if (!make_weight_tmap(&gp.map_sa, gp.Sa, rpe * n_shared, gp.row_bytes, L::BOX, box_rows))
      return DQ_ERR_CUDA;
    if (GATEUP && !make_weight_tmap(&gp.map_sb, gp.Sb, rpe * n_shared, gp.row_bytes, L::BOX, box_rows))
      return DQ_ERR_CUDA;
  }
  const int ex_bytes = 64 * 8 * NT * 4;
  int nstage = 12;
  while (nstage > 3 && make_plan<FMT>(nstage, 8 * NT, 1).total + ex_bytes > 56 * 1024) --nstage;
  gp.nstage = nstage;
  const int smem = make_plan<FMT>(nstage, 8 * NT, 1).total + ex_bytes;
  static bool attr[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !attr[dev]) {
    if (cudaFuncSetAttribute(grouped_kernel<FMT, GATEUP, NT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
      return DQ_ERR_CUDA;
    if (dev < 64) attr[dev] = true;
  }
  const int sms = sm_count();
  if (sms <= 0) return DQ_ERR_CUDA;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, grouped_kernel<FMT, GATEUP, NT>, kThreads,
                                                    smem) != cudaSuccess || occ < 1)
    occ = 1;
  const int grid = std::max(1, std::min(units_max, occ * sms));
  if (launch_pdl(grouped_kernel<FMT, GATEUP, NT>, dim3(grid), dim3(kThreads), smem, s, 0, gp) !=
      cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

template <bool GATEUP>
int launch_grouped_fmt(int fmt, int nt, const GroupedParams& gp, int units_max, cudaStream_t s,
                       int E, int n_shared) {
#define DQ_GROUPED(F, N) \
  if (fmt == F && nt == N) return launch_grouped<F, GATEUP, N>(gp, units_max, s, E, n_shared);
  DQ_GROUPED(DQ_Q4_K, 1) DQ_GROUPED(DQ_Q4_K, 2) DQ_GROUPED(DQ_Q4_K, 4)
  DQ_GROUPED(DQ_Q6_K, 1) DQ_GROUPED(DQ_Q6_K, 2) DQ_GROUPED(DQ_Q6_K, 4)
  DQ_GROUPED(DQ_Q8_0, 1) DQ_GROUPED(DQ_Q8_0, 2) DQ_GROUPED(DQ_Q8_0, 4)
  DQ_GROUPED(DQ_NVFP4, 1) DQ_GROUPED(DQ_NVFP4, 2) DQ_GROUPED(DQ_NVFP4, 4)
#undef DQ_GROUPED
  return DQ_ERR_UNSUPPORTED;
}

}  // namespace

int launch_tc_gemm(int fmt, const void* W, const void* Wsh, int E, int n_shared,
                   int rows_per_expert, int K, const int4* units, const int* n_units,
                   int max_units, const __half* X16, int64_t npos, const float* xinv, float* out,
                   int64_t out_stride, cudaStream_t s);
int launch_x16_rows(const void* x, int xdt, int rows, int K, __half* out, float* inv,
                    cudaStream_t s);
int launch_gather_x16(const int4* units, const int* n_units, int max_units, const int32_t* tok,
                      const __half* x16, const float* tinv, int K, __half* X16, float* xinv,
                      cudaStream_t s);
int launch_swiglu_wide(const int4* units, const int* n_units, int max_units, const float* G,
                       const float* U, int F, float* h, cudaStream_t s);

int launch_router(const float* Wr, int E, int H, const void* x, int xdt, int T, int top_k,
                  int KS, float* part, float* logits, int32_t* idx, float* gate, cudaStream_t s,
                  bool with_topk) {
  const int chunk = router_chunk(T);
  const int nchunks = chunk ? (H + chunk - 1) / chunk : 0;
  const bool vec_ok = ((uintptr_t)x & 15) == 0 && H % 8 == 0;
  // the streaming kernel: one chunk per CTA (KS partials), or every chunk in
  // each CTA when one partial is asked for (dq_moe_router)
  if (chunk && (KS == nchunks || KS == 1) && ((uintptr_t)Wr & 15) == 0 && H % 4 == 0 &&
      vec_ok) {
    const int nc = KS == 1 ? nchunks : 1;
    const dim3 g((unsigned)((E + 7) / 8), (unsigned)KS);
#define DQ_RS(TM, CH, XD) \
  launch_pdl(router_stream_kernel<TM, CH, XD>, g, dim3(256), 0, s, 0, Wr, E, H, x, T, part, nc)
    if (T <= kRouterStreamT) {
      if (xdt == DQ_F32) DQ_RS(kRouterStreamT, kRouterChunk, DQ_F32);
      else if (xdt == DQ_BF16) DQ_RS(kRouterStreamT, kRouterChunk, DQ_BF16);
      else DQ_RS(kRouterStreamT, kRouterChunk, DQ_F16);
    } else {
      if (xdt == DQ_F32) DQ_RS(kRouterStreamT2, kRouterChunk2, DQ_F32);
      else if (xdt == DQ_BF16) DQ_RS(kRouterStreamT2, kRouterChunk2, DQ_BF16);
      else DQ_RS(kRouterStreamT2, kRouterChunk2, DQ_F16);
    }
#undef DQ_RS
  } else {
    dim3 g1((unsigned)((E + 63) / 64), (unsigned)((T + 31) / 32), (unsigned)KS);
    if (xdt == DQ_F32)
      launch_pdl(router_logits_kernel<DQ_F32>, g1, dim3(128), 0, s, 0, Wr, E, H, x, T, KS, part);
    else if (xdt == DQ_BF16)
      launch_pdl(router_logits_kernel<DQ_BF16>, g1, dim3(128), 0, s, 0, Wr, E, H, x, T, KS, part);
    else
      launch_pdl(router_logits_kernel<DQ_F16>, g1, dim3(128), 0, s, 0, Wr, E, H, x, T, KS, part);
  }
  if (cudaGetLastError() != cudaSuccess) return DQ_ERR_CUDA;
  if (!with_topk) return DQ_OK;
  launch_pdl(topk_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, s, 0, part, KS, T, E, top_k, logits, idx, gate);
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

int launch_permute(const int32_t* idx, int T, int k, int E, int32_t* offsets, int32_t* sorted,
                   cudaStream_t s) {
  launch_pdl(permute_kernel, dim3(1), dim3(1024), 0, s, 0, const_cast<int32_t*>(idx), T, k, E, 0,
             8, offsets, sorted, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0,
             0, nullptr, nullptr, TopkIn{nullptr, 0, nullptr, nullptr}, nullptr, nullptr);
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

namespace {

// A second stream per (device, caller stream), of the device's highest
// priority, for the general expert kernels that run beside the one-token
// ones; forked from and joined back into the caller's stream with events.
// Created on first use outside stream capture and kept until the process
// exits; `mu` orders the fork, the launches and the join of concurrent calls
// on the same caller stream.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
};
std::mutex g_side_mu;
std::map<std::pair<int, cudaStream_t>, SideStream*> g_side;

// The side stream of `s` on the current device, or null (none yet and `s` is
// being captured, or creation failed): the caller then stays on `s`.
SideStream* side_stream(cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(g_side_mu);
  auto it = g_side.find({dev, s});
  if (it != g_side.end()) return it->second;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return nullptr;
  int least = 0, greatest = 0;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
  SideStream* ss = new SideStream;
  if (cudaStreamCreateWithPriority(&ss->s, cudaStreamNonBlocking, greatest) != cudaSuccess ||
      cudaEventCreateWithFlags(&ss->fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ss->join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    delete ss;   // handles created before the failure stay with the process
    return nullptr;
  }
  g_side[{dev, s}] = ss;
  return ss;
}

// Joins the side stream back into the caller's stream when the layer's
// launches are enqueued (also on an early error return), then releases the
// side stream's lock.
struct ForkJoin {
  SideStream* ss = nullptr;
  cudaStream_t main = nullptr;
  std::unique_lock<std::mutex> lock;
  int join() {
    if (!ss) return DQ_OK;
    const bool ok = cudaEventRecord(ss->join, ss->s) == cudaSuccess &&
                    cudaStreamWaitEvent(main, ss->join, 0) == cudaSuccess;
    ss = nullptr;
    if (lock.owns_lock()) lock.unlock();
    return ok ? DQ_OK : DQ_ERR_CUDA;
  }
  ~ForkJoin() { join(); }
};

}  // namespace

// stages: 1 = router and top-k, 2 = the rest (permute, experts, combine), 3 = both.
// ms (nullable): the streamed layer's slot cache and copy/compute phases.
int launch_moe_forward(const dq_moe_desc& d, const void* x, int xdt, int T, float* y, void* ws,
                       int32_t* topk_idx, float* topk_gate, float* logits, cudaStream_t s,
                       const MoeStream* ms, int stages, bool side) {
  const MoePlan pl = moe_plan(d, T, ms == nullptr);
  uint8_t* w = (uint8_t*)ws;
  float* part = (float*)(w + pl.off_part);
  float* lg = logits ? logits : (float*)(w + pl.off_logits);
  int32_t* idx = topk_idx ? topk_idx : (int32_t*)(w + pl.off_idx);
  float* gate = topk_gate ? topk_gate : (float*)(w + pl.off_gate);
  int32_t* offsets = (int32_t*)(w + pl.off_offsets);
  int32_t* sorted = (int32_t*)(w + pl.off_sorted);
  int32_t* inv = (int32_t*)(w + pl.off_inv);
  int32_t* tok = (int32_t*)(w + pl.off_tok);
  int4* groups = (int4*)(w + pl.off_groups);
  int32_t* ngroups = (int32_t*)(w + pl.off_ngroups);
  float* h = (float*)(w + pl.off_h);
  float* ypos = (float*)(w + pl.off_ypos);

  int rc = DQ_OK;
  // up to 32 tokens in one call: the permute CTA takes the top-k too (one
  // warp per token), one launch less on the decode path
  const bool fuse_topk = (stages & 3) == 3 && T <= 32;
  if (stages & 1) {
    rc = launch_router(d.router_W, d.E, d.hidden, x, xdt, T, d.top_k, pl.KS, part, lg, idx, gate,
                       s, !fuse_topk);
    if (rc != DQ_OK) return rc;
  }
  if (!(stages & 2)) return DQ_OK;
  int4* units = (int4*)(w + pl.off_units);
  int32_t* nunits = (int32_t*)(w + pl.off_nunits);
  __half* x16t = (__half*)(w + pl.off_x16t);
  float* xinvt = (float*)(w + pl.off_xinvt);
  // one-token groups (pl.single) go to the block-diagonal kernels, which read
  // x and h as they are; the grouped mma.sync kernels and their fp16 copies
  // of x and h are needed only where a group can hold more tokens (T > 1)
  int4* groups1 = (int4*)(w + pl.off_g1);
  int32_t* ng1 = (int32_t*)(w + pl.off_ng1);
  const bool general = !pl.single || T > 1;
  // one or two tokens of bf16/fp32 x: the permute CTA also makes their fp16
  // copy (measured: one launch less at T=1; at T=8 eight CTAs are faster)
  const bool fuse_x16 = general && xdt != DQ_F16 && T <= 2 && d.hidden <= 8192;
  launch_pdl(permute_kernel, dim3(1), dim3(1024), 0, s, 0, idx, T, d.top_k, d.E, d.n_shared,
             pl.GW, offsets, sorted, inv, tok, groups, ngroups, pl.wide ? units : nullptr, nunits,
             fuse_x16 ? x : nullptr, xdt, d.hidden, fuse_x16 ? x16t : nullptr,
             fuse_x16 ? xinvt : nullptr,
             fuse_topk ? TopkIn{part, pl.KS, lg, gate} : TopkIn{nullptr, 0, nullptr, nullptr},
             pl.single ? groups1 : nullptr, pl.single ? ng1 : nullptr);
  if (cudaGetLastError() != cudaSuccess) return DQ_ERR_CUDA;

  const int q = qk(d.fmt), bb = blk_bytes(d.fmt);
  __half* h16 = (__half*)(w + pl.off_h16);
  float* hinv = (float*)(w + pl.off_hinv);
  __half* x16 = (__half*)(w + pl.off_x16);
  float* xinv = (float*)(w + pl.off_xinv);
  float* G = (float*)(w + pl.off_g);
  float* U = (float*)(w + pl.off_u);

  // fp16 activations for the streaming kernels (fp16 input is used as is)
  const __half* xh = (const __half*)x;
  const float* xh_inv = nullptr;
  if (xdt != DQ_F16 && general) {
    if (!fuse_x16) {
      rc = launch_x16_rows(x, xdt, T, d.hidden, x16t, xinvt, s);
      if (rc != DQ_OK) return rc;
    }
    xh = x16t;
    xh_inv = xinvt;
  }

  // one-token groups beside the general kernels (T > 1): the general and
  // tensor-core kernels run on a side stream of higher priority, so that
  // their CTAs are placed first, concurrently with the one-token kernels on
  // `s` (both read the same inputs and write different positions of h and
  // ypos)
  cudaStream_t sg = s;
  ForkJoin fj;
  if (side && !ms && general && pl.single) {
    SideStream* ss = side_stream(s);
    if (ss) {
      fj.lock = std::unique_lock<std::mutex>(ss->mu);
      if (cudaEventRecord(ss->fork, s) != cudaSuccess ||
          cudaStreamWaitEvent(ss->s, ss->fork, 0) != cudaSuccess)
        return DQ_ERR_CUDA;
      fj.ss = ss;
      fj.main = s;
      sg = ss->s;
    }
  }

  GroupedParams gu;
  memset(&gu, 0, sizeof(gu));
  gu.Wa = (const uint8_t*)d.w_gate;
  gu.Wb = (const uint8_t*)d.w_up;
  gu.Sa = (const uint8_t*)d.sh_gate;
  gu.Sb = (const uint8_t*)d.sh_up;
  gu.row_bytes = (int64_t)(d.hidden / q) * bb;
  gu.mat_bytes = gu.row_bytes * d.ffn;
  gu.nsb = d.hidden / 256;
  gu.E = d.E;
  gu.groups = groups;
  gu.n_groups = ngroups;
  gu.tok = tok;
  gu.xbase = xh;
  gu.xdt = DQ_F16;
  gu.xstride = d.hidden;
  gu.out = h;
  gu.out_stride = d.ffn;
  gu.colinv = xh_inv;
  gu.coltok = tok;
  gu.tiles = d.ffn / 32;
  gu.ksplit = 1;
  gu.rows_per_expert = d.ffn;
  if (!ms) {
    if (general) {
      rc = launch_grouped_fmt<true>(d.fmt, pl.NT, gu, pl.G_max * gu.tiles, sg, d.E, d.n_shared);
      if (rc != DQ_OK) return rc;
    }
    if (pl.single) {
      rc = launch_grouped_b1(true, d, groups1, ng1, pl.G1_max, ng1 + 1, x, xdt, d.hidden, h,
                             d.ffn, s);
      if (rc != DQ_OK) return rc;
    }
  } else {
    // streamed: routed matrices from the slot cache, one launch per phase
    // once that phase's copies have landed
    gu.Wa = (const uint8_t*)ms->slot_gate;
    gu.Wb = (const uint8_t*)ms->slot_up;
    gu.slot_of = ms->slot_of;
    gu.phase_of = ms->phase_of;
    for (int ph = 0; ph < ms->nphase; ++ph) {
      if (ms->gu_ready[ph] && cudaStreamWaitEvent(s, ms->gu_ready[ph], 0) != cudaSuccess)
        return DQ_ERR_CUDA;
      gu.phase = ph;
      rc = launch_grouped_fmt<true>(d.fmt, pl.NT, gu, pl.G_max * gu.tiles, s, ms->slots,
                                    d.n_shared);
      if (rc != DQ_OK) return rc;
    }
  }

  // wide units: gathered fp16 rows, tensor-core gate and up GEMMs, SwiGLU
  if (pl.wide) {
    rc = launch_gather_x16(units, nunits, pl.U_max, tok, xh, xh_inv, d.hidden, x16, xinv, sg);
    if (rc != DQ_OK) return rc;
    rc = launch_tc_gemm(d.fmt, d.w_gate, d.sh_gate, d.E, d.n_shared, d.ffn, d.hidden, units,
                        nunits, pl.U_max, x16, pl.NP, xinv, G, d.ffn, sg);
    if (rc != DQ_OK) return rc;
    rc = launch_tc_gemm(d.fmt, d.w_up, d.sh_up, d.E, d.n_shared, d.ffn, d.hidden, units, nunits,
                        pl.U_max, x16, pl.NP, xinv, U, d.ffn, sg);
    if (rc != DQ_OK) return rc;
    rc = launch_swiglu_wide(units, nunits, pl.U_max, G, U, d.ffn, h, sg);
    if (rc != DQ_OK) return rc;
  }

  // h -> fp16 with a power-of-two scale per position (all positions), for
  // the grouped mma.sync kernels
  if (general) {
    rc = launch_x16_rows(h, DQ_F32, (int)pl.NP, d.ffn, h16, hinv, sg);
    if (rc != DQ_OK) return rc;
  }

  GroupedParams dn;
  memset(&dn, 0, sizeof(dn));
  dn.Wa = (const uint8_t*)d.w_down;
  dn.Sa = (const uint8_t*)d.sh_down;
  dn.row_bytes = (int64_t)(d.ffn / q) * bb;
  dn.mat_bytes = dn.row_bytes * d.hidden;
  dn.nsb = d.ffn / 256;
  dn.E = d.E;
  dn.groups = groups;
  dn.n_groups = ngroups;
  dn.tok = nullptr;
  dn.xbase = h16;
  dn.xdt = DQ_F16;
  dn.xstride = d.ffn;
  dn.out = ypos;
  dn.out_stride = d.hidden;
  dn.colinv = hinv;
  dn.coltok = nullptr;
  dn.tiles = d.hidden / 64;
  dn.ksplit = ms ? 1 : pl.DS;
  dn.part_stride = (int64_t)pl.NP * d.hidden;
  dn.rows_per_expert = d.hidden;
  if (!ms) {
    if (general) {
      rc = launch_grouped_fmt<false>(d.fmt, pl.NT, dn, pl.G_max * dn.tiles * dn.ksplit, sg, d.E,
                                     d.n_shared);
      if (rc != DQ_OK) return rc;
    }
    if (pl.single) {
      rc = launch_grouped_b1(false, d, groups1, ng1, pl.G1_max, ng1 + 2, h, DQ_F32, d.ffn, ypos,
                             d.hidden, s);
      if (rc != DQ_OK) return rc;
    }
  } else {
    dn.Wa = (const uint8_t*)ms->slot_down;
    dn.slot_of = ms->slot_of;
    dn.phase_of = ms->phase_of;
    for (int ph = 0; ph < ms->nphase; ++ph) {
      if (ms->dn_ready[ph] && cudaStreamWaitEvent(s, ms->dn_ready[ph], 0) != cudaSuccess)
        return DQ_ERR_CUDA;
      dn.phase = ph;
      rc = launch_grouped_fmt<false>(d.fmt, pl.NT, dn, pl.G_max * dn.tiles, s, ms->slots,
                                     d.n_shared);
      if (rc != DQ_OK) return rc;
    }
  }
  if (pl.wide) {
    rc = launch_tc_gemm(d.fmt, d.w_down, d.sh_down, d.E, d.n_shared, d.hidden, d.ffn, units,
                        nunits, pl.U_max, h16, pl.NP, hinv, ypos, d.hidden, sg);
    if (rc != DQ_OK) return rc;
  }

  // the join, before the combine reads every position
  rc = fj.join();
  if (rc != DQ_OK) return rc;
  const int64_t n4 = (int64_t)T * d.hidden / 4;
  const int cgrid = (int)std::min<int64_t>((n4 + 255) / 256, 4096);
  launch_pdl(combine_kernel, dim3(cgrid), dim3(256), 0, s, 0, ypos, inv, gate, T, d.top_k,
             d.hidden, d.n_shared, pl.DS, (int64_t)pl.NP * d.hidden, y);
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

}  // namespace dqmoe
