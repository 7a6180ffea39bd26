// dequant.cu — step "block decode" on its own: packed blocks -> fp32.
//
// The pages name the formats (Titan Engine §激进量化策略: Q4_K; KTransformers
// §支持的量化格式: Q4_K_M, Q6_K, Q8_0, Q4_0, Q5_K, Q2_K, Q3_K; NTransformer
// §量化支持: Q80, Q6K) but print no layout; the GGUF/llama.cpp layouts
// declared in dqmoe.h are used.  Each output is the exact closed form rounded
// once to fp32: every product below is exact in fp32 and the Q4_K / Q5_K /
// Q2_K differences are formed by one fused multiply-add, so the result is
// bit-identical to any exact evaluation.
//
// One thread per output weight (coalesced fp32 stores); the block's few
// header bytes are re-read by its threads through L1.  Every format also has
// a wide form, taken when the output is 16-byte aligned: a warp per 512
// weights, each lane decoding runs of 4 (the scale fields read once per run,
// the quant bytes as 16-bit loads) into 16-byte stores that cover 512
// contiguous bytes per warp instruction (Q8_0: a thread per 8 weights).  It
// evaluates every weight with the same expression, so both forms give the same
// bits.  The GEMV kernels never materialise W: this is the decode step on its
// own.
#include "common.cuh"

namespace dqmoe {

__device__ __forceinline__ float h16(const uint8_t* p) {
  return __half2float(__ushort_as_half((unsigned short)(p[0] | (p[1] << 8))));
}

__global__ void dequant_q4k_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                   float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t blk = gid >> 8;
  if (blk >= nblk) return;
  const int i = (int)(gid & 255);
  const uint8_t* b = blocks + blk * 144;
  const float d = h16(b), dmin = h16(b + 2);
  const uint8_t* s = b + 4;
  const int j = i >> 5;            // sub-block: 32 weights
  int sc, m;
  if (j < 4) {
    sc = s[j] & 63;
    m = s[j + 4] & 63;
  } else {
    sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
    m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
  }
  const int c = i >> 6, l = i & 31;  // 32-byte group c; low nibble first half
  const uint8_t byte = b[16 + 32 * c + l];
  const int q = (i & 32) ? (byte >> 4) : (byte & 15);
  out[gid] = __fmaf_rn(d * (float)sc, (float)q, -(dmin * (float)m));
}

__global__ void dequant_q6k_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                   float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t blk = gid >> 8;
  if (blk >= nblk) return;
  const int i = (int)(gid & 255);
  const uint8_t* b = blocks + blk * 210;
  const int h = i >> 7, r = (i >> 5) & 3, l = i & 31;   // i = 128h + 32r + l
  const uint8_t qlb = b[64 * h + l + ((r & 1) ? 32 : 0)];
  const uint8_t qhb = b[128 + 32 * h + l];
  const int lo = (r & 2) ? (qlb >> 4) : (qlb & 15);
  const int hi = (qhb >> (2 * r)) & 3;
  const int q = lo | (hi << 4);
  const int sc = (int)(int8_t)b[192 + (i >> 4)];
  const float d = h16(b + 208);
  out[gid] = d * (float)sc * (float)(q - 32);
}

__global__ void dequant_q80_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                   float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t blk = gid >> 5;
  if (blk >= nblk) return;
  const uint8_t* b = blocks + blk * 34;
  out[gid] = h16(b) * (float)(int8_t)b[2 + (gid & 31)];
}

// Four bytes at an even address (blocks are 2-byte aligned) as two 16-bit
// loads, byte 0 in bits 0..7.
__device__ __forceinline__ uint32_t bytes4(const uint8_t* p) {
  return (uint32_t)__ldg((const unsigned short*)p) |
         ((uint32_t)__ldg((const unsigned short*)p + 1) << 16);
}
__device__ __forceinline__ void store4(float* o, float a, float b, float c, float d) {
  *(float4*)o = make_float4(a, b, c, d);
}

// Wide forms: weights i .. i + 3 (i % 4 == 0) of one block at b, each by
// the same expression as the one-weight form (so both give the same bits).
template <int FMT> struct DQW;

template <> struct DQW<DQ_Q4_K> {
  static constexpr int QK = 256, BB = 144;
  __device__ __forceinline__ static void run(const uint8_t* b, int i, float (&v)[4]) {
    const float d = h16(b), dmin = h16(b + 2);
    const uint8_t* s = b + 4;
    const int j = i >> 5;
    int sc, m;
    if (j < 4) {
      sc = s[j] & 63;
      m = s[j + 4] & 63;
    } else {
      sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
      m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
    // byte 16 + 32 (i >> 6) + (i & 31): weight i (low nibble) and i + 32
    uint32_t q = bytes4(b + 16 + 32 * (i >> 6) + (i & 31));
    if (i & 32) q >>= 4;
    const float ds = d * (float)sc, dm = -(dmin * (float)m);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = __fmaf_rn(ds, (float)((q >> (8 * e)) & 15), dm);
  }
};

template <> struct DQW<DQ_Q6_K> {
  static constexpr int QK = 256, BB = 210;
  __device__ __forceinline__ static void run(const uint8_t* b, int i, float (&v)[4]) {
    const int h = i >> 7, r = (i >> 5) & 3, l = i & 31;   // i = 128h + 32r + l
    uint32_t lo = bytes4(b + 64 * h + l + ((r & 1) ? 32 : 0));
    if (r & 2) lo >>= 4;
    const uint32_t hi = bytes4(b + 128 + 32 * h + l) >> (2 * r);
    const float ds = h16(b + 208) * (float)(int)(int8_t)b[192 + (i >> 4)];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int q = (int)((lo >> (8 * e)) & 15) | (int)(((hi >> (8 * e)) & 3) << 4);
      v[e] = ds * (float)(q - 32);
    }
  }
};

template <> struct DQW<DQ_Q5_K> {
  static constexpr int QK = 256, BB = 176;
  __device__ __forceinline__ static void run(const uint8_t* b, int i, float (&v)[4]) {
    const float d = h16(b), dmin = h16(b + 2);
    const uint8_t* s = b + 4;
    const int j = i >> 5;
    int sc, m;
    if (j < 4) {
      sc = s[j] & 63;
      m = s[j + 4] & 63;
    } else {
      sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
      m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
    const int c = i >> 6, l = i & 31;
    uint32_t q = bytes4(b + 48 + 32 * c + l);
    if (i & 32) q >>= 4;
    const uint32_t hb = bytes4(b + 16 + l) >> j;   // bit j of qh[l]: bit 4 of q
    const float ds = d * (float)sc, dm = -(dmin * (float)m);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      v[e] = __fmaf_rn(ds, (float)(((q >> (8 * e)) & 15) | (((hb >> (8 * e)) & 1) << 4)), dm);
  }
};

template <> struct DQW<DQ_Q4_0> {
  static constexpr int QK = 32, BB = 18;
  __device__ __forceinline__ static void run(const uint8_t* b, int i, float (&v)[4]) {
    uint32_t q = bytes4(b + 2 + (i & 15));
    if (i & 16) q >>= 4;
    const float d = h16(b);
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = d * (float)((int)((q >> (8 * e)) & 15) - 8);
  }
};

template <> struct DQW<DQ_Q2_K> {
  static constexpr int QK = 256, BB = 84;
  __device__ __forceinline__ static void run(const uint8_t* b, int i, float (&v)[4]) {
    const int h = i >> 7, r = (i >> 5) & 3, l = i & 31;
    const uint32_t q = bytes4(b + 16 + 32 * h + l) >> (2 * r);
    const int sm = b[i >> 4];
    const float ds = h16(b + 80) * (float)(sm & 15), dm = -(h16(b + 82) * (float)(sm >> 4));
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = __fmaf_rn(ds, (float)((q >> (8 * e)) & 3), dm);
  }
};

template <> struct DQW<DQ_Q3_K> {
  static constexpr int QK = 256, BB = 110;
  __device__ __forceinline__ static void run(const uint8_t* b, int i, float (&v)[4]) {
    const int h = i >> 7, r = (i >> 5) & 3, l = i & 31;
    const uint32_t low = bytes4(b + 32 + 32 * h + l) >> (2 * r);
    const uint32_t hm = bytes4(b + l) >> (4 * h + r);
    const int j = i >> 4;
    const int sc = ((b[96 + (j & 7)] >> (4 * (j >> 3))) & 15) |
                   (((b[104 + (j & 3)] >> (2 * (j >> 2))) & 3) << 4);
    const float ds = h16(b + 108) * (float)(sc - 32);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int q = (int)((low >> (8 * e)) & 3) - (((hm >> (8 * e)) & 1) ? 0 : 4);
      v[e] = ds * (float)q;
    }
  }
};

template <> struct DQW<DQ_NVFP4> {
  static constexpr int QK = 256, BB = 144;
  __device__ __forceinline__ static void run(const uint8_t* b, int i, float (&v)[4]) {
    // codes of weights i .. i + 3: bytes 16 + i / 2, + 1 (low nibble first)
    uint32_t h[4];
    e2m1x8_to_h2x4((uint32_t)__ldg((const unsigned short*)(b + 16 + i / 2)), h);
    const float s = __low2float(u32_as_h2(e4m3x2_to_h2((uint16_t)b[i >> 4])));
    const float2 a = __half22float2(u32_as_h2(h[0])), c = __half22float2(u32_as_h2(h[1]));
    v[0] = a.x * s;
    v[1] = a.y * s;
    v[2] = c.x * s;
    v[3] = c.y * s;
  }
};

// Warp w decodes the 512 weights 512 w .. 512 w + 511, 16 per lane in four
// rounds; in round k lane l takes weights 128 k + 4 l .. + 3, so that each
// round's 16-byte stores cover 512 contiguous bytes of the output.
template <int FMT>
__global__ void dequantw_kernel(const uint8_t* __restrict__ blocks, int64_t n,
                                float* __restrict__ out) {
  using D = DQW<FMT>;
  pdl_wait();
  pdl_trigger();
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int l = (int)(g & 31);
  const int64_t w0 = (g >> 5) * 512;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t w = w0 + 128 * k + 4 * l;
    if (w >= n) break;
    float v[4];
    D::run(blocks + (w / D::QK) * D::BB, (int)(w % D::QK), v);
    store4(out + w, v[0], v[1], v[2], v[3]);
  }
}

// Q8_0: thread g decodes weights 8g .. 8g + 7 (a quarter block), two 16-byte
// stores (measured faster for this format than the warp-interleaved form).
__global__ void dequant8_q80_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                    float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t blk = g >> 2;
  if (blk >= nblk) return;
  const uint8_t* b = blocks + blk * 34;
  const int i0 = (int)(g & 3) * 8;
  const uint32_t q0 = bytes4(b + 2 + i0), q1 = bytes4(b + 6 + i0);
  const float d = h16(b);
  store4(out + g * 8, d * (float)(int8_t)(q0 & 0xFF), d * (float)(int8_t)((q0 >> 8) & 0xFF),
         d * (float)(int8_t)((q0 >> 16) & 0xFF), d * (float)(int8_t)(q0 >> 24));
  store4(out + g * 8 + 4, d * (float)(int8_t)(q1 & 0xFF), d * (float)(int8_t)((q1 >> 8) & 0xFF),
         d * (float)(int8_t)((q1 >> 16) & 0xFF), d * (float)(int8_t)(q1 >> 24));
}

// Q4_0: w = d*(q - 8); byte j of qs: weight j (low nibble), j+16 (high).
__global__ void dequant_q40_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                   float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t blk = gid >> 5;
  if (blk >= nblk) return;
  const int i = (int)(gid & 31);
  const uint8_t* b = blocks + blk * 18;
  const uint8_t byte = b[2 + (i & 15)];
  const int q = (i & 16) ? (byte >> 4) : (byte & 15);
  out[gid] = h16(b) * (float)(q - 8);
}

// Q5_K: Q4_K's closed form with a 5-bit q (qh bit 2c or 2c+1 as bit 4).
__global__ void dequant_q5k_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                   float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t blk = gid >> 8;
  if (blk >= nblk) return;
  const int i = (int)(gid & 255);
  const uint8_t* b = blocks + blk * 176;
  const float d = h16(b), dmin = h16(b + 2);
  const uint8_t* s = b + 4;
  const int j = i >> 5;            // sub-block: 32 weights
  int sc, m;
  if (j < 4) {
    sc = s[j] & 63;
    m = s[j + 4] & 63;
  } else {
    sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
    m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
  }
  const int c = i >> 6, l = i & 31;
  const uint8_t byte = b[48 + 32 * c + l];
  const int hb = (b[16 + l] >> j) & 1;   // bit 2c (low half) or 2c+1 (high half) = bit j
  const int q = ((i & 32) ? (byte >> 4) : (byte & 15)) | (hb << 4);
  out[gid] = __fmaf_rn(d * (float)sc, (float)q, -(dmin * (float)m));
}

// Q2_K: weight i = 128h + 32r + l takes bits 2r..2r+1 of qs[32h + l];
// w = d*sc*q - dmin*m of its 16-weight sub-block (both products exact in
// fp32, the difference one fused multiply-add).
__global__ void dequant_q2k_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                   float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t blk = gid >> 8;
  if (blk >= nblk) return;
  const int i = (int)(gid & 255);
  const uint8_t* b = blocks + blk * 84;
  const int h = i >> 7, r = (i >> 5) & 3, l = i & 31;
  const int q = (b[16 + 32 * h + l] >> (2 * r)) & 3;
  const int sm = b[i >> 4];
  out[gid] = __fmaf_rn(h16(b + 80) * (float)(sm & 15), (float)q, -(h16(b + 82) * (float)(sm >> 4)));
}

// Q3_K: low bits 2r..2r+1 of qs[32h + l], high bit 4h + r of hmask[l]
// (clear: q = low - 4); w = d*(s - 32)*q with the 6-bit scale s of the
// 16-weight sub-block.  Every product is exact in fp32.
__global__ void dequant_q3k_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                   float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t blk = gid >> 8;
  if (blk >= nblk) return;
  const int i = (int)(gid & 255);
  const uint8_t* b = blocks + blk * 110;
  const int h = i >> 7, r = (i >> 5) & 3, l = i & 31;
  const int low = (b[32 + 32 * h + l] >> (2 * r)) & 3;
  const int q = low - (((b[l] >> (4 * h + r)) & 1) ? 0 : 4);
  const int j = i >> 4;
  const int sc = ((b[96 + (j & 7)] >> (4 * (j >> 3))) & 15) |
                 (((b[104 + (j & 3)] >> (2 * (j >> 2))) & 3) << 4);
  out[gid] = h16(b + 108) * (float)(sc - 32) * (float)q;
}

// NVFP4: w = e2m1(code) * e4m3(scale of the 16-weight block); both
// conversions by the hardware (exact), the product exact in fp32.  One thread
// per 8 weights (one code word).
__global__ void dequant_nvfp4_kernel(const uint8_t* __restrict__ blocks, int64_t nblk,
                                     float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t blk = gid >> 5;
  if (blk >= nblk) return;
  const int j = (int)(gid & 31);                   // weights 8j..8j+7
  const uint8_t* b = blocks + blk * 144;
  const uint32_t w = (uint32_t)b[16 + 4 * j] | ((uint32_t)b[17 + 4 * j] << 8) |
                     ((uint32_t)b[18 + 4 * j] << 16) | ((uint32_t)b[19 + 4 * j] << 24);
  uint32_t h[4];
  e2m1x8_to_h2x4(w, h);
  const float s = __low2float(u32_as_h2(e4m3x2_to_h2((uint16_t)b[j >> 1])));
  float* o = out + blk * 256 + 8 * j;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(u32_as_h2(h[i]));
    o[2 * i] = v.x * s;
    o[2 * i + 1] = v.y * s;
  }
}

int launch_dequant(int fmt, const void* blocks, int64_t n, float* out, cudaStream_t s) {
  const int threads = 256;
  const int64_t grid = (n + threads - 1) / threads;
  const uint8_t* b = (const uint8_t*)blocks;
  if (((uintptr_t)out & 15) == 0) {
    // the wide forms: one warp per 512 weights (Q8_0: one thread per 8)
    const dim3 gw((unsigned)(((n + 511) / 512 * 32 + threads - 1) / threads));
    if (fmt == DQ_Q4_K) launch_pdl(dequantw_kernel<DQ_Q4_K>, gw, dim3(threads), 0, s, 0, b, n, out);
    else if (fmt == DQ_Q6_K) launch_pdl(dequantw_kernel<DQ_Q6_K>, gw, dim3(threads), 0, s, 0, b, n, out);
    else if (fmt == DQ_Q5_K) launch_pdl(dequantw_kernel<DQ_Q5_K>, gw, dim3(threads), 0, s, 0, b, n, out);
    else if (fmt == DQ_Q4_0) launch_pdl(dequantw_kernel<DQ_Q4_0>, gw, dim3(threads), 0, s, 0, b, n, out);
    else if (fmt == DQ_Q2_K) launch_pdl(dequantw_kernel<DQ_Q2_K>, gw, dim3(threads), 0, s, 0, b, n, out);
    else if (fmt == DQ_Q3_K) launch_pdl(dequantw_kernel<DQ_Q3_K>, gw, dim3(threads), 0, s, 0, b, n, out);
    else if (fmt == DQ_NVFP4) launch_pdl(dequantw_kernel<DQ_NVFP4>, gw, dim3(threads), 0, s, 0, b, n, out);
    else launch_pdl(dequant8_q80_kernel, dim3((unsigned)((n / 8 + threads - 1) / threads)),
                    dim3(threads), 0, s, 0, b, n / 32, out);
    return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
  }
  if (fmt == DQ_Q4_K) launch_pdl(dequant_q4k_kernel, dim3((unsigned)grid), dim3(threads), 0, s, 0, b, n / 256, out);
  else if (fmt == DQ_Q6_K) launch_pdl(dequant_q6k_kernel, dim3((unsigned)grid), dim3(threads), 0, s, 0, b, n / 256, out);
  else if (fmt == DQ_Q8_0) launch_pdl(dequant_q80_kernel, dim3((unsigned)grid), dim3(threads), 0, s, 0, b, n / 32, out);
  else if (fmt == DQ_Q4_0) launch_pdl(dequant_q40_kernel, dim3((unsigned)grid), dim3(threads), 0, s, 0, b, n / 32, out);
  else if (fmt == DQ_Q5_K) launch_pdl(dequant_q5k_kernel, dim3((unsigned)grid), dim3(threads), 0, s, 0, b, n / 256, out);
  else if (fmt == DQ_Q2_K) launch_pdl(dequant_q2k_kernel, dim3((unsigned)grid), dim3(threads), 0, s, 0, b, n / 256, out);
  else if (fmt == DQ_Q3_K) launch_pdl(dequant_q3k_kernel, dim3((unsigned)grid), dim3(threads), 0, s, 0, b, n / 256, out);
  else launch_pdl(dequant_nvfp4_kernel, dim3((unsigned)((n / 8 + threads - 1) / threads)), dim3(threads), 0, s, 0, b, n / 256, out);
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

}  // namespace dqmoe
