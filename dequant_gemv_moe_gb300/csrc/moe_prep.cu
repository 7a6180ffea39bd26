// moe_prep.cu — activation preparation for the MoE layer's streaming kernels.
//
// The grouped expert kernels read 16-bit activations straight into shared
// memory with asynchronous copies, so every activation they read is fp16:
//   * x16_tokens_kernel : bf16 / fp32 x -> fp16 rows with one power-of-two
//     scale per token (max|x| * scale in [2^14, 2^15): no overflow);
//   * h16_kernel        : the fp32 SwiGLU output h -> fp16 rows with one
//     power-of-two scale per position;
//   * gather_x16_kernel : the wide (tensor-core) units' activation rows,
//     gathered by token into position order for TMA;
//   * swiglu_wide_kernel: h = silu(g) * u for the wide units.
// The kernels consuming these undo the scale on their fp32 results.
#include <algorithm>

#include "qgemv_mma.cuh"

namespace dqmoe {

namespace {
__device__ __forceinline__ float wmax(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// the dtype is a compile-time constant, so that the loads of an unrolled
// loop are all in flight before the first is used
template <int XDT>
__device__ __forceinline__ float act(const void* x, int64_t i) {
  if (XDT == DQ_F32) return __ldg((const float*)x + i);
  if (XDT == DQ_BF16) return __uint_as_float((uint32_t)__ldg((const unsigned short*)x + i) << 16);
  return __half2float(__ldg((const __half*)x + i));
}
}  // namespace

// one CTA per row: out[row][k] = fp16(in[row][k] * 2^e), inv[row] = 2^-e, with
// max|in[row]| * 2^e in [2^14, 2^15).  256 threads, or 1024 for rows longer
// than 256 * R values, so that a row of up to 1024 * R values is read once,
// every load in flight before any is used.
template <int XDT>
__global__ void __launch_bounds__(1024) x16_tokens_kernel(const void* __restrict__ x, int rows,
                                                          int K, __half* __restrict__ out,
                                                          float* __restrict__ inv) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  constexpr int R = 32;                 // values kept in registers per thread
  const int row = blockIdx.x, nt = blockDim.x, nw = nt >> 5;
  const int64_t base = (int64_t)row * K;
  const bool in_regs = K <= nt * R;
  float v[R];
  float amax = 0.f;
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int k = threadIdx.x + nt * i;
      v[i] = k < K ? act<XDT>(x, base + k) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < R; ++i) amax = fmaxf(amax, fabsf(v[i]));
  } else {
    for (int k0 = threadIdx.x; k0 < K; k0 += nt * 8) {
      float a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = k0 + nt * i;
        a[i] = k < K ? act<XDT>(x, base + k) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(a[i]));
    }
  }
  amax = wmax(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
  for (int i = 1; i < nw; ++i) amax = fmaxf(amax, red[i]);
  float sc, iv;
  pow2_scale(amax, sc, iv);
  if (in_regs) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int k = threadIdx.x + nt * i;
      if (k < K) out[base + k] = __float2half_rn(v[i] * sc);
    }
  } else {
    for (int k0 = threadIdx.x; k0 < K; k0 += nt * 8) {
      float a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = k0 + nt * i;
        a[i] = k < K ? act<XDT>(x, base + k) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = k0 + nt * i;
        if (k < K) out[base + k] = __float2half_rn(a[i] * sc);
      }
    }
  }
  if (threadIdx.x == 0) inv[row] = iv;
}

// X16[pos] = x16[tok[pos]], xinv[pos] = tinv[tok[pos]] (tinv null: 1) for the
// positions of the wide units.  Grid (kGatherSplit, units): CTA (j, u) copies
// the rows j * 8 + warp (+ 8 kGatherSplit ...) of unit u, one warp per row.
constexpr int kGatherSplit = 8;

__global__ void __launch_bounds__(256) gather_x16_kernel(const int4* __restrict__ units,
                                                         const int* __restrict__ n_units,
                                                         const int32_t* __restrict__ tok,
                                                         const __half* __restrict__ x16,
                                                         const float* __restrict__ tinv, int K,
                                                         __half* __restrict__ X16,
                                                         float* __restrict__ xinv) {
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.y >= __ldg(n_units)) return;
  const int4 u = __ldg(units + blockIdx.y);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int n = blockIdx.x * 8 + warp; n < u.z; n += 8 * kGatherSplit) {
    const int pos = u.y + n;
    const int t = __ldg(tok + pos);
    const uint4* src = (const uint4*)(x16 + (int64_t)t * K);
    uint4* dst = (uint4*)(X16 + (int64_t)pos * K);
#pragma unroll 4
    for (int k = lane; k < K / 8; k += 32) dst[k] = __ldg(src + k);
    if (lane == 0) xinv[pos] = tinv ? __ldg(tinv + t) : 1.f;
  }
}

// h = silu(G) * U for the wide units' positions; silu(g) = g / (1 + exp(-g))
// (-0 for g < -88: exp overflows to inf, never NaN).  Grid: (chunks, units).
__global__ void __launch_bounds__(256) swiglu_wide_kernel(const int4* __restrict__ units,
                                                          const int* __restrict__ n_units,
                                                          const float* __restrict__ G,
                                                          const float* __restrict__ U, int F,
                                                          float* __restrict__ h) {
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.y >= __ldg(n_units)) return;
  const int4 u = __ldg(units + blockIdx.y);
  const int64_t base = (int64_t)u.y * F, n = (int64_t)u.z * F;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float g = G[base + i];
    h[base + i] = g / (1.f + expf(-g)) * U[base + i];
  }
}

int launch_x16_rows(const void* x, int xdt, int rows, int K, __half* out, float* inv,
                    cudaStream_t s) {
  const int threads = K > 256 * 32 ? 1024 : 256;
  cudaError_t e;
  if (xdt == DQ_F32)
    e = launch_pdl(x16_tokens_kernel<DQ_F32>, dim3(rows), dim3(threads), 0, s, 0, x, rows, K, out,
                   inv);
  else if (xdt == DQ_BF16)
    e = launch_pdl(x16_tokens_kernel<DQ_BF16>, dim3(rows), dim3(threads), 0, s, 0, x, rows, K,
                   out, inv);
  else
    e = launch_pdl(x16_tokens_kernel<DQ_F16>, dim3(rows), dim3(threads), 0, s, 0, x, rows, K, out,
                   inv);
  if (e != cudaSuccess) return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

int launch_gather_x16(const int4* units, const int* n_units, int max_units, const int32_t* tok,
                      const __half* x16, const float* tinv, int K, __half* X16, float* xinv,
                      cudaStream_t s) {
  const dim3 grid((unsigned)kGatherSplit, (unsigned)(max_units > 0 ? max_units : 1));
  if (launch_pdl(gather_x16_kernel, grid, dim3(256), 0, s, 0, units, n_units, tok, x16, tinv,
                 K, X16, xinv) != cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

int launch_swiglu_wide(const int4* units, const int* n_units, int max_units, const float* G,
                       const float* U, int F, float* h, cudaStream_t s) {
  const int chunks = (int)std::min<int64_t>(((int64_t)128 * F + 2047) / 2048, 256);
  const dim3 grid((unsigned)chunks, (unsigned)(max_units > 0 ? max_units : 1));
  if (launch_pdl(swiglu_wide_kernel, grid, dim3(256), 0, s, 0, units, n_units, G, U, F, h) !=
      cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

}  // namespace dqmoe
