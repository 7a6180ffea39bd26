// noalloc.cu — dq_moe_forward_noalloc: the MoE layer for callers that cannot
// allocate device memory, with its scratch in a fixed array inside the library.
//
// Who needs it: code that runs under a host framework which owns all device
// memory and offers no workspace hook (plugins, custom-op shims), and decode
// loops that must not allocate on the hot path (no cudaMalloc latency, no
// fragmentation, no allocator call between captured or replayed steps).  They
// cannot size and pass the `ws` buffer dq_moe_forward expects.
//
// The scratch is one file-scope __device__ array of DQ_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads this library holds that much device memory until the
// process exits.  Host code cannot use the array's name as a device address,
// so the device address is fetched with cudaGetSymbolAddress once per device,
// on the first call made with that device current.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "moe_plan.h"

namespace dqmoe {

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The address is
// looked up once per device; the lookup is a runtime call that must not run
// while `stream` is being captured, so a first call under capture is refused
// (DQ_ERR_UNSUPPORTED) instead of calling into the runtime mid-capture.
int scratch_on_current_device(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return DQ_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return DQ_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return DQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DQ_OK;
}

}  // namespace

}  // namespace dqmoe

extern "C" int dq_moe_forward_noalloc(const dq_moe_desc* desc, const void* x, int x_dtype, int T,
                                      float* y, int32_t* topk_idx, float* topk_gate,
                                      float* logits, void* stream) {
  using namespace dqmoe;
  size_t need = 0;
  const int rc = dq_moe_workspace_size(desc, T, &need);
  if (rc != DQ_OK) return rc;
  if (need > (size_t)DQ_NOALLOC_SCRATCH_BYTES) return DQ_ERR_WORKSPACE;
  void* ws = nullptr;
  const int src = scratch_on_current_device((cudaStream_t)stream, &ws);
  if (src != DQ_OK) return src;
  // one stream only: the layer's second stream would be created on first use
  return moe_forward_checked(desc, x, x_dtype, T, y, ws, (size_t)DQ_NOALLOC_SCRATCH_BYTES,
                             topk_idx, topk_gate, logits, stream, false);
}
