// stage.cu — dq_stage: moves a decode step's activations in and its outputs
// out with a kernel launched like every other kernel of the library.
//
// On GB300 the SMs reach page-locked host memory directly over the coherent
// host link, so a copy done by a kernel stays inside the chain of
// programmatic dependent launches: the GEMV after it is scheduled while it
// drains, as after any other kernel here.  A copy-engine copy between two
// kernels (a memcpy node in a CUDA graph) ends that chain and adds the copy
// engine's latency: measured on GB300, the Llama-3-8B decode layer's four
// GEMVs with their activations uploaded and outputs read back took 49.3 us
// per step with two copy-engine copies and 36.8 us with this kernel (32.3 us
// without any copy).
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"

namespace dqmoe {

__global__ void __launch_bounds__(256) stage_kernel(uint4* __restrict__ dst,
                                                    const uint4* __restrict__ src, int64_t n16) {
  // the source may be the previous kernel's output, and the destination its input
  pdl_wait();
  pdl_trigger();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

int launch_stage(void* dst, const void* src, int64_t bytes, cudaStream_t s) {
  const int64_t n16 = bytes / 16;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return DQ_ERR_CUDA;
  // one CTA of 256 threads per 4 KB, at most one per SM (a step's vectors are
  // tens of KB; a grid-stride loop covers larger copies)
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, (n16 + 255) / 256));
  if (launch_pdl(stage_kernel, dim3(grid), dim3(256), 0, s, 0, (uint4*)dst, (const uint4*)src,
                 n16) != cudaSuccess)
    return DQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DQ_OK : DQ_ERR_CUDA;
}

}  // namespace dqmoe

extern "C" int dq_stage(void* dst, const void* src, int64_t bytes, void* stream) {
  if (!dst || !src || bytes <= 0) return DQ_ERR_ARG;
  if (bytes % 16 || ((uintptr_t)dst & 15) || ((uintptr_t)src & 15)) return DQ_ERR_ALIGN;
  const uintptr_t d = (uintptr_t)dst, s = (uintptr_t)src;
  if (d < s + (uintptr_t)bytes && s < d + (uintptr_t)bytes) return DQ_ERR_ARG;   // overlap
  return dqmoe::launch_stage(dst, src, bytes, (cudaStream_t)stream);
}
