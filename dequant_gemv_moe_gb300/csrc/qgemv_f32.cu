// qgemv_f32.cu — y = W x for fp32 activations on the CUDA cores.
//
// Used for x in fp32, where the result must match an exact evaluation to
// ~1e-5 of max|y|: every weight is decoded exactly in fp32 (closed forms of
// dqmoe.h, one rounding) and multiplied-accumulated in fp32.  One warp per
// row; each lane owns 8 weights of every 256-weight super-block; warp-shuffle
// reduction at the end.  The tensor-core path (qgemv_mma.cu) serves the 16-bit
// activations of the decode configurations; this path is for exactness.
#include "common.cuh"

namespace dqmoe {

namespace {

__device__ __forceinline__ float h16g(const uint8_t* p) {
  return __half2float(__ushort_as_half((unsigned short)(p[0] | (p[1] << 8))));
}

// Decode the 8 weights lane `l` owns in one 256-weight unit and return their
// offsets inside the unit.
template <int FMT>
__device__ __forceinline__ void lane_weights(const uint8_t* sb, int l, float (&w)[8], int (&k)[8]);

template <>
__device__ __forceinline__ void lane_weights<DQ_Q4_K>(const uint8_t* b, int l, float (&w)[8],
                                                      int (&k)[8]) {
  const float d = h16g(b), dmin = h16g(b + 2);
  const uint8_t* s = b + 4;
  const int c = l >> 3, o = (l & 7) * 4;       // group c, bytes o..o+3
  int sc[2], m[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = 2 * c + h;
    if (j < 4) {
      sc[h] = s[j] & 63;
      m[h] = s[j + 4] & 63;
    } else {
      sc[h] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
      m[h] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint8_t q = b[16 + 32 * c + o + i];
    w[i] = __fmaf_rn(d * (float)sc[0], (float)(q & 15), -(dmin * (float)m[0]));
    k[i] = 64 * c + o + i;
    w[4 + i] = __fmaf_rn(d * (float)sc[1], (float)(q >> 4), -(dmin * (float)m[1]));
    k[4 + i] = 64 * c + 32 + o + i;
  }
}

template <>
__device__ __forceinline__ void lane_weights<DQ_Q6_K>(const uint8_t* b, int l, float (&w)[8],
                                                      int (&k)[8]) {
  const float d = h16g(b + 208);
  const int h = l >> 4, o = (l & 15) * 2;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int li = o + i;
      const uint8_t qlb = b[64 * h + li + ((r & 1) ? 32 : 0)];
      const uint8_t qhb = b[128 + 32 * h + li];
      const int q = ((r & 2) ? (qlb >> 4) : (qlb & 15)) | (((qhb >> (2 * r)) & 3) << 4);
      const int idx = 128 * h + 32 * r + li;
      const int sc = (int)(int8_t)b[192 + (idx >> 4)];
      w[2 * r + i] = d * (float)sc * (float)(q - 32);
      k[2 * r + i] = idx;
    }
  }
}

template <>
__device__ __forceinline__ void lane_weights<DQ_Q8_0>(const uint8_t* b, int l, float (&w)[8],
                                                      int (&k)[8]) {
  const uint8_t* blk = b + 34 * (l >> 2);
  const float d = h16g(blk);
  const int o = (l & 3) * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    w[i] = d * (float)(int8_t)blk[2 + o + i];
    k[i] = 32 * (l >> 2) + o + i;
  }
}

template <>
__device__ __forceinline__ void lane_weights<DQ_Q4_0>(const uint8_t* b, int l, float (&w)[8],
                                                      int (&k)[8]) {
  // 8 blocks of 18 bytes; lane l: block l/4, bytes 4*(l%4)..+3 (weights j, j+16)
  const uint8_t* blk = b + 18 * (l >> 2);
  const float d = h16g(blk);
  const int o = (l & 3) * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint8_t q = blk[2 + o + i];
    w[i] = d * (float)((q & 15) - 8);
    k[i] = 32 * (l >> 2) + o + i;
    w[4 + i] = d * (float)((q >> 4) - 8);
    k[4 + i] = 32 * (l >> 2) + 16 + o + i;
  }
}

template <>
__device__ __forceinline__ void lane_weights<DQ_Q5_K>(const uint8_t* b, int l, float (&w)[8],
                                                      int (&k)[8]) {
  const float d = h16g(b), dmin = h16g(b + 2);
  const uint8_t* s = b + 4;
  const int c = l >> 3, o = (l & 7) * 4;       // group c, bytes o..o+3
  int sc[2], m[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int j = 2 * c + h;
    if (j < 4) {
      sc[h] = s[j] & 63;
      m[h] = s[j + 4] & 63;
    } else {
      sc[h] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
      m[h] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint8_t q = b[48 + 32 * c + o + i];
    const uint8_t h = b[16 + o + i];
    const int q0 = (q & 15) | (((h >> (2 * c)) & 1) << 4);
    const int q1 = (q >> 4) | (((h >> (2 * c + 1)) & 1) << 4);
    w[i] = __fmaf_rn(d * (float)sc[0], (float)q0, -(dmin * (float)m[0]));
    k[i] = 64 * c + o + i;
    w[4 + i] = __fmaf_rn(d * (float)sc[1], (float)q1, -(dmin * (float)m[1]));
    k[4 + i] = 64 * c + 32 + o + i;
  }
}

// Q2_K / Q3_K: lane l owns bytes 2(l%16), +1 of qs half h = l/16: weights
// 128h + 32r + 2(l%16) + {0, 1} for r = 0..3.
template <>
__device__ __forceinline__ void lane_weights<DQ_Q2_K>(const uint8_t* b, int l, float (&w)[8],
                                                      int (&k)[8]) {
  const float d = h16g(b + 80), dmin = h16g(b + 82);
  const int h = l >> 4, li = 2 * (l & 15);
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = 128 * h + 32 * r + li + i;
      const int q = (b[16 + 32 * h + li + i] >> (2 * r)) & 3;
      const int sm = b[idx >> 4];
      w[2 * r + i] = __fmaf_rn(d * (float)(sm & 15), (float)q, -(dmin * (float)(sm >> 4)));
      k[2 * r + i] = idx;
    }
}

template <>
__device__ __forceinline__ void lane_weights<DQ_Q3_K>(const uint8_t* b, int l, float (&w)[8],
                                                      int (&k)[8]) {
  const float d = h16g(b + 108);
  const int h = l >> 4, li = 2 * (l & 15);
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = 128 * h + 32 * r + li + i;
      const int low = (b[32 + 32 * h + li + i] >> (2 * r)) & 3;
      const int q = low - (((b[li + i] >> (4 * h + r)) & 1) ? 0 : 4);
      const int j = idx >> 4;
      const int sc = ((b[96 + (j & 7)] >> (4 * (j >> 3))) & 15) |
                     (((b[104 + (j & 3)] >> (2 * (j >> 2))) & 3) << 4);
      w[2 * r + i] = d * (float)(sc - 32) * (float)q;
      k[2 * r + i] = idx;
    }
}

template <>
__device__ __forceinline__ void lane_weights<DQ_NVFP4>(const uint8_t* b, int l, float (&w)[8],
                                                       int (&k)[8]) {
  // lane l: weights 8l..8l+7 (code bytes 16+4l..+3), block scale l/2
  const uint32_t word = (uint32_t)b[16 + 4 * l] | ((uint32_t)b[17 + 4 * l] << 8) |
                        ((uint32_t)b[18 + 4 * l] << 16) | ((uint32_t)b[19 + 4 * l] << 24);
  uint32_t h[4];
  e2m1x8_to_h2x4(word, h);
  const float s = __low2float(u32_as_h2(e4m3x2_to_h2((uint16_t)b[l >> 1])));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(u32_as_h2(h[i]));
    w[2 * i] = v.x * s;
    w[2 * i + 1] = v.y * s;
    k[2 * i] = 8 * l + 2 * i;
    k[2 * i + 1] = 8 * l + 2 * i + 1;
  }
}

template <int FMT, int B>
__global__ void __launch_bounds__(256) qgemv_f32_kernel(const uint8_t* __restrict__ W,
                                                        int64_t N, int64_t nsb,
                                                        const float* __restrict__ x,
                                                        int64_t K, float* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= N) return;
  const uint8_t* wr = W + row * nsb * Fmt<FMT>::SB_BYTES;
  float acc[B];
#pragma unroll
  for (int b = 0; b < B; ++b) acc[b] = 0.f;
  for (int64_t j = 0; j < nsb; ++j) {
    float w[8];
    int k[8];
    lane_weights<FMT>(wr + j * Fmt<FMT>::SB_BYTES, lane, w, k);
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const float* xb = x + b * K + j * 256;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[b] = __fmaf_rn(w[i], xb[k[i]], acc[b]);
    }
  }
#pragma unroll
  for (int b = 0; b < B; ++b) {
    float v = acc[b];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) y[b * N + row] = v;
  }
}

template <int FMT>
int launch_f32_fmt(const void* W, int64_t N, int64_t K, const float* x, int batch, float* y,
                   cudaStream_t s) {
  const int64_t nsb = K / 256;
  const unsigned grid = (unsigned)((N + 7) / 8);
  const uint8_t* w = (const uint8_t*)W;
  cudaError_t rc = cudaSuccess;
  switch (batch) {
#define DQ_CASE(BB) \
  case BB:                                                                               \
    rc = launch_pdl(qgemv_f32_kernel<FMT, BB>, dim3(grid), dim3(256), 0, s, 0, w, N, nsb, x, K, y); \
    break;
    DQ_CASE(1) DQ_CASE(2) DQ_CASE(3) DQ_CASE(4) DQ_CASE(5) DQ_CASE(6) DQ_CASE(7) DQ_CASE(8)
#undef DQ_CASE
    default: return DQ_ERR_ARG;
  }
  if (rc != cudaSuccess) return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

}  // namespace

int launch_qgemv_f32(int fmt, const void* W, int64_t N, int64_t K, const float* x, int batch,
                     float* y, cudaStream_t s) {
  if (fmt == DQ_Q4_K) return launch_f32_fmt<DQ_Q4_K>(W, N, K, x, batch, y, s);
  if (fmt == DQ_Q6_K) return launch_f32_fmt<DQ_Q6_K>(W, N, K, x, batch, y, s);
  if (fmt == DQ_Q8_0) return launch_f32_fmt<DQ_Q8_0>(W, N, K, x, batch, y, s);
  if (fmt == DQ_Q4_0) return launch_f32_fmt<DQ_Q4_0>(W, N, K, x, batch, y, s);
  if (fmt == DQ_Q5_K) return launch_f32_fmt<DQ_Q5_K>(W, N, K, x, batch, y, s);
  if (fmt == DQ_Q2_K) return launch_f32_fmt<DQ_Q2_K>(W, N, K, x, batch, y, s);
  if (fmt == DQ_Q3_K) return launch_f32_fmt<DQ_Q3_K>(W, N, K, x, batch, y, s);
  return launch_f32_fmt<DQ_NVFP4>(W, N, K, x, batch, y, s);
}

}  // namespace dqmoe
