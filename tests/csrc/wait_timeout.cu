// wait_timeout.cu — test build of the library's bounded mbarrier waits with a
// short limit (DQ_WAIT_LIMIT_CYCLES on the nvcc command line).  One CTA waits
// on a barrier nothing arrives on: the wait must give up, record
// DQ_ERR_DEVICE_TIMEOUT in the status word and let the kernel return.  No
// bulk copy is in flight, so the kernel leaves nothing behind.
#include "../../dequant_gemv_moe_gb300/csrc/common.cuh"

namespace dqmoe {
__device__ int g_device_status = 0;
}

using namespace dqmoe;

__global__ void wait_nobody_kernel(int* out) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);            // one arrival expected, none ever made
    fence_barrier_init();
  }
  __syncthreads();
  const bool done = mbar_wait(&bar, 0);
  out[threadIdx.x] = done ? 1 : 2;
}

// Same, with the cluster-scope wait of the split-K reduction.
__global__ void __cluster_dims__(2, 1, 1) wait_nobody_cluster_kernel(int* out) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  cluster_sync_all();
  const bool done = mbar_wait_cluster(&bar, 0);
  out[blockIdx.x * blockDim.x + threadIdx.x] = done ? 1 : 2;
  cluster_sync_all();
}

extern "C" int wt_run(int cluster, int* out_host, int n) {
  int* d = nullptr;
  if (cudaMalloc(&d, n * sizeof(int)) != cudaSuccess) return -1;
  cudaMemset(d, 0, n * sizeof(int));
  if (cluster) wait_nobody_cluster_kernel<<<2, n / 2>>>(d);
  else wait_nobody_kernel<<<1, n>>>(d);
  const cudaError_t e = cudaDeviceSynchronize();
  cudaMemcpy(out_host, d, n * sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(d);
  return e == cudaSuccess ? 0 : -2;
}

extern "C" int wt_status(int* st) {
  if (cudaMemcpyFromSymbol(st, g_device_status, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) == cudaSuccess ? 0 : -1;
}
