// api.cu — the C ABI of dqmoe.h: argument validation (before any launch),
// dispatch on format / activation dtype, status strings, device status word.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>

#include "common.cuh"
#include "moe_plan.h"
#include "stream_cache.h"

namespace dqmoe {
__device__ int g_device_status = 0;

int launch_dequant(int fmt, const void* blocks, int64_t n, float* out, cudaStream_t s);
int launch_qgemv_f32(int fmt, const void* W, int64_t N, int64_t K, const float* x, int batch,
                     float* y, cudaStream_t s);
int launch_qgemv_mma(int fmt, const void* W, int64_t N, int64_t K, const void* x, int xdt,
                     int batch, float* y, cudaStream_t s, int force_ksplit, bool w_early);
int launch_router(const float* Wr, int E, int H, const void* x, int xdt, int T, int top_k,
                  int KS, float* part, float* logits, int32_t* idx, float* gate, cudaStream_t s,
                  bool with_topk = true);
int launch_permute(const int32_t* idx, int T, int k, int E, int32_t* offsets, int32_t* sorted,
                   cudaStream_t s);

}  // namespace dqmoe

using namespace dqmoe;

namespace {

bool fmt_ok(int fmt) { return fmt >= DQ_Q4_K && fmt <= DQ_Q3_K; }
// formats of the MoE layer's expert matrices
bool moe_fmt_ok(int fmt) {
  return fmt == DQ_Q4_K || fmt == DQ_Q6_K || fmt == DQ_Q8_0 || fmt == DQ_NVFP4;
}
bool dtype_ok(int dt) { return dt == DQ_F32 || dt == DQ_F16 || dt == DQ_BF16; }
bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

int qk_of(int fmt) { return (fmt == DQ_Q8_0 || fmt == DQ_Q4_0) ? DQ_QK8_0 : DQ_QK_K; }

int block_bytes(int fmt) {
  switch (fmt) {
    case DQ_Q4_K: return DQ_Q4_K_BYTES;
    case DQ_Q6_K: return DQ_Q6_K_BYTES;
    case DQ_Q8_0: return DQ_Q8_0_BYTES;
    case DQ_Q4_0: return DQ_Q4_0_BYTES;
    case DQ_Q5_K: return DQ_Q5_K_BYTES;
    case DQ_Q2_K: return DQ_Q2_K_BYTES;
    case DQ_Q3_K: return DQ_Q3_K_BYTES;
    default: return DQ_NVFP4_BYTES;
  }
}

int check_qgemv(int fmt, const void* W, int64_t N, int64_t K, const void* x, int xdt, int batch,
                const float* y) {
  if (!fmt_ok(fmt) || !dtype_ok(xdt)) return DQ_ERR_ARG;
  if (!W || !x || !y) return DQ_ERR_ARG;
  if (N <= 0 || K <= 0 || N > (1LL << 31) - 1 || K > (1LL << 30)) return DQ_ERR_ARG;
  if (batch < 1 || batch > DQ_MAX_BATCH) return DQ_ERR_ARG;
  // all kernels stream 256-weight super-block units
  if (K % 256) return DQ_ERR_ARG;
  // rows 16-B aligned: 210- and 110-byte blocks in eights, 84-byte ones in fours
  if ((fmt == DQ_Q6_K || fmt == DQ_Q3_K) && K % 2048) return DQ_ERR_ALIGN;
  if (fmt == DQ_Q2_K && K % 1024) return DQ_ERR_ALIGN;
  if (!aligned(W, 16) || !aligned(x, 16) || !aligned(y, 4)) return DQ_ERR_ALIGN;
  if ((int64_t)((N + 63) / 64) > 65535) return DQ_ERR_UNSUPPORTED;
  return DQ_OK;
}

int check_desc(const dq_moe_desc* d, int T) {
  if (!d || T <= 0) return DQ_ERR_ARG;
  if (!fmt_ok(d->fmt)) return DQ_ERR_ARG;
  if (!moe_fmt_ok(d->fmt)) return DQ_ERR_UNSUPPORTED;
  if (d->E <= 0 || d->top_k <= 0 || d->top_k > d->E || d->hidden <= 0 || d->ffn <= 0 ||
      d->n_shared < 0)
    return DQ_ERR_ARG;
  if (d->E > 256 || d->top_k > 8 || d->n_shared > 4) return DQ_ERR_UNSUPPORTED;
  if (T > 65536 || (int64_t)T * d->top_k > 524288) return DQ_ERR_UNSUPPORTED;
  if (d->hidden % 256 || d->ffn % 256) return DQ_ERR_ARG;
  if (d->fmt == DQ_Q6_K && (d->hidden % 2048 || d->ffn % 2048)) return DQ_ERR_ALIGN;
  if (!d->router_W || !d->w_gate || !d->w_up || !d->w_down) return DQ_ERR_ARG;
  if (d->n_shared > 0 && (!d->sh_gate || !d->sh_up || !d->sh_down)) return DQ_ERR_ARG;
  if (!aligned(d->router_W, 4) || !aligned(d->w_gate, 16) || !aligned(d->w_up, 16) ||
      !aligned(d->w_down, 16))
    return DQ_ERR_ALIGN;
  if (d->n_shared > 0 &&
      (!aligned(d->sh_gate, 16) || !aligned(d->sh_up, 16) || !aligned(d->sh_down, 16)))
    return DQ_ERR_ALIGN;
  return DQ_OK;
}

}  // namespace

int dqmoe::moe_forward_checked(const dq_moe_desc* desc, const void* x, int x_dtype, int T,
                               float* y, void* ws, size_t ws_bytes, int32_t* topk_idx,
                               float* topk_gate, float* logits, void* stream, bool side) {
  int rc = check_desc(desc, T);
  if (rc != DQ_OK) return rc;
  if (!x || !y || !dtype_ok(x_dtype)) return DQ_ERR_ARG;
  // the experts run on 16-bit tensor-core operands: fp32 activations would
  // be held to a bar (1e-5) that path cannot meet, so they are refused
  if (x_dtype == DQ_F32) return DQ_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(y, 16)) return DQ_ERR_ALIGN;
  if ((topk_idx && !aligned(topk_idx, 4)) || (topk_gate && !aligned(topk_gate, 4)) ||
      (logits && !aligned(logits, 4)))
    return DQ_ERR_ALIGN;
  if (!ws) return DQ_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return DQ_ERR_ALIGN;
  if (ws_bytes < moe_plan(*desc, T).total) return DQ_ERR_WORKSPACE;
  return launch_moe_forward(*desc, x, x_dtype, T, y, ws, topk_idx, topk_gate, logits,
                            (cudaStream_t)stream, nullptr, 3, side);
}

extern "C" {

int dq_block_geometry(int fmt, int* weights_per_block, int* bytes_per_block) {
  if (!weights_per_block || !bytes_per_block || !fmt_ok(fmt)) return DQ_ERR_ARG;
  *weights_per_block = qk_of(fmt);
  *bytes_per_block = block_bytes(fmt);
  return DQ_OK;
}

int dq_dequant(int fmt, const void* blocks, int64_t n_weights, float* out, void* stream) {
  if (!fmt_ok(fmt) || !blocks || !out || n_weights <= 0) return DQ_ERR_ARG;
  if (n_weights % qk_of(fmt)) return DQ_ERR_ARG;
  if (n_weights > (1LL << 40)) return DQ_ERR_UNSUPPORTED;
  if (!aligned(blocks, 2) || !aligned(out, 4)) return DQ_ERR_ALIGN;
  return launch_dequant(fmt, blocks, n_weights, out, (cudaStream_t)stream);
}

int dq_qgemv(int fmt, const void* W, int64_t N, int64_t K, const void* x, int x_dtype, int batch,
             float* y, void* stream) {
  return dq_qgemv_ksplit(fmt, W, N, K, x, x_dtype, batch, y, 0, stream);
}

int dq_qgemv_ksplit(int fmt, const void* W, int64_t N, int64_t K, const void* x, int x_dtype,
                    int batch, float* y, int ksplit, void* stream) {
  return dq_qgemv_ex(fmt, W, N, K, x, x_dtype, batch, y, ksplit, 0u, stream);
}

int dq_qgemv_ex(int fmt, const void* W, int64_t N, int64_t K, const void* x, int x_dtype,
                int batch, float* y, int ksplit, unsigned flags, void* stream) {
  const int rc = check_qgemv(fmt, W, N, K, x, x_dtype, batch, y);
  if (rc != DQ_OK) return rc;
  if (ksplit < 0 || ksplit > 8) return DQ_ERR_ARG;
  if (flags & ~DQ_QGEMV_WEIGHTS_EARLY) return DQ_ERR_ARG;
  if (x_dtype == DQ_F32)
    return launch_qgemv_f32(fmt, W, N, K, (const float*)x, batch, y, (cudaStream_t)stream);
  return launch_qgemv_mma(fmt, W, N, K, x, x_dtype, batch, y, (cudaStream_t)stream, ksplit,
                          (flags & DQ_QGEMV_WEIGHTS_EARLY) != 0);
}

int dq_moe_workspace_size(const dq_moe_desc* desc, int T, size_t* bytes) {
  if (!bytes) return DQ_ERR_ARG;
  const int rc = check_desc(desc, T);
  if (rc != DQ_OK) return rc;
  *bytes = moe_plan(*desc, T).total;
  return DQ_OK;
}

int dq_moe_router(const float* router_W, int E, int H, const void* x, int x_dtype, int T,
                  int top_k, float* logits, int32_t* topk_idx, float* topk_gate, void* stream) {
  if (!router_W || !x || !logits || !topk_idx || !topk_gate || !dtype_ok(x_dtype)) return DQ_ERR_ARG;
  if (E <= 0 || H <= 0 || T <= 0 || top_k <= 0 || top_k > E || H % 32) return DQ_ERR_ARG;
  if (E > 256 || top_k > 8 || T > 65536) return DQ_ERR_UNSUPPORTED;
  if (!aligned(router_W, 4) || !aligned(x, 4) || !aligned(logits, 4) || !aligned(topk_idx, 4) ||
      !aligned(topk_gate, 4))
    return DQ_ERR_ALIGN;
  // one hidden-dimension slice: the logits buffer holds the single partial sum
  return launch_router(router_W, E, H, x, x_dtype, T, top_k, 1, logits, logits, topk_idx,
                       topk_gate, (cudaStream_t)stream);
}

int dq_moe_permute(const int32_t* topk_idx, int T, int top_k, int E, int32_t* offsets,
                   int32_t* sorted, void* stream) {
  if (!topk_idx || !offsets || !sorted || T <= 0 || top_k <= 0 || E <= 0) return DQ_ERR_ARG;
  if (E > 256 || (int64_t)T * top_k > 65536) return DQ_ERR_UNSUPPORTED;
  return launch_permute(topk_idx, T, top_k, E, offsets, sorted, (cudaStream_t)stream);
}

int dq_moe_forward(const dq_moe_desc* desc, const void* x, int x_dtype, int T, float* y, void* ws,
                   size_t ws_bytes, int32_t* topk_idx, float* topk_gate, float* logits,
                   void* stream) {
  return dqmoe::moe_forward_checked(desc, x, x_dtype, T, y, ws, ws_bytes, topk_idx, topk_gate,
                                    logits, stream, true);
}


int dq_expert_cache_create(const dq_moe_desc* d, int slots, void* slot_gate, void* slot_up,
                           void* slot_down, int max_tokens, int phases, dq_expert_cache** cache) {
  if (!cache) return DQ_ERR_ARG;
  *cache = nullptr;
  if (max_tokens <= 0) return DQ_ERR_ARG;
  const int rc = check_desc(d, max_tokens);
  if (rc != DQ_OK) return rc;
  if (phases < 1 || phases > dqmoe::kMaxStreamPhases) return DQ_ERR_ARG;
  const long long need = std::min<long long>(d->E, (long long)max_tokens * d->top_k);
  if (slots < need || slots > d->E) return DQ_ERR_ARG;
  if (!slot_gate || !slot_up || !slot_down) return DQ_ERR_ARG;
  if (!aligned(slot_gate, 16) || !aligned(slot_up, 16) || !aligned(slot_down, 16))
    return DQ_ERR_ALIGN;
  // the routed experts must be page-locked host memory (asynchronous copies)
  const void* hp[3] = {d->w_gate, d->w_up, d->w_down};
  for (const void* ptr : hp) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
      cudaGetLastError();
      return DQ_ERR_ARG;
    }
    if (a.type != cudaMemoryTypeHost) return DQ_ERR_ARG;
  }
  const int q = qk_of(d->fmt), bb = block_bytes(d->fmt);
  const int64_t gu_bytes = (int64_t)d->ffn * (d->hidden / q) * bb;
  const int64_t dn_bytes = (int64_t)d->hidden * (d->ffn / q) * bb;
  dq_expert_cache* c = new (std::nothrow) dq_expert_cache;
  if (!c) return DQ_ERR_CUDA;
  const int irc = dqmoe::stream_cache_init(c, *d, slots, slot_gate, slot_up, slot_down,
                                           max_tokens, phases, gu_bytes, dn_bytes);
  if (irc != DQ_OK) {
    dqmoe::stream_cache_release(c);
    delete c;
    return irc;
  }
  *cache = c;
  return DQ_OK;
}

int dq_expert_cache_workspace_size(const dq_expert_cache* cache, int T, size_t* bytes) {
  if (!cache || !bytes || T <= 0 || T > cache->max_tokens) return DQ_ERR_ARG;
  size_t a, b;
  *bytes = dqmoe::stream_workspace(*cache, T, &a, &b);
  return DQ_OK;
}

int dq_moe_forward_streamed(dq_expert_cache* cache, const void* x, int x_dtype, int T, float* y,
                            void* ws, size_t ws_bytes, void* stream, void* copy_stream) {
  if (!cache || !x || !y || !dtype_ok(x_dtype) || T <= 0 || T > cache->max_tokens)
    return DQ_ERR_ARG;
  if (x_dtype == DQ_F32) return DQ_ERR_UNSUPPORTED;   // as dq_moe_forward
  if (stream == copy_stream) return DQ_ERR_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return DQ_ERR_ALIGN;
  if (!ws) return DQ_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return DQ_ERR_ALIGN;
  size_t a, b;
  if (ws_bytes < dqmoe::stream_workspace(*cache, T, &a, &b)) return DQ_ERR_WORKSPACE;
  return dqmoe::stream_forward(cache, x, x_dtype, T, y, ws, (cudaStream_t)stream,
                               (cudaStream_t)copy_stream);
}

int dq_expert_cache_stats(const dq_expert_cache* cache, long long* hits, long long* misses,
                          long long* bytes_copied) {
  if (!cache || !hits || !misses || !bytes_copied) return DQ_ERR_ARG;
  *hits = cache->hits;
  *misses = cache->misses;
  *bytes_copied = cache->bytes_copied;
  return DQ_OK;
}

int dq_expert_cache_destroy(dq_expert_cache* cache) {
  if (!cache) return DQ_ERR_ARG;
  dqmoe::stream_cache_release(cache);
  delete cache;
  return DQ_OK;
}

const char* dq_status_string(int status) {
  switch (status) {
    case DQ_OK: return "ok";
    case DQ_ERR_ARG: return "invalid argument";
    case DQ_ERR_ALIGN: return "misaligned pointer or row stride";
    case DQ_ERR_UNSUPPORTED: return "unsupported format, dtype or shape";
    case DQ_ERR_WORKSPACE: return "workspace missing or too small";
    case DQ_ERR_CUDA: return "CUDA runtime or launch error";
    case DQ_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait timed out";
    default: return "unknown status";
  }
}

int dq_device_status(int* status) {
  if (!status) return DQ_ERR_ARG;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return DQ_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return DQ_ERR_CUDA;
  *status = v;
  return DQ_OK;
}

}  // extern "C"
