// stream.cu — the streamed MoE layer: routed experts in page-locked host
// memory, a device cache of expert slots kept least-recently-used, and the
// missing experts copied in chunks on a copy stream while the grouped
// kernels of the chunks already in place run ([Titan Engine, §MoE
// 专家流式加载]: on-demand expert loading, an LRU cache of hot experts,
// asynchronous loads that hide the transfer; [NTransformer, §核心技术] SLEP:
// a double-buffered pipeline overlapping transfers with GPU compute).
//
// Per call: router and top-k on the device, the routing read back (one host
// synchronisation of the compute stream), host-side cache bookkeeping, one
// cudaMemcpyAsync per missing expert matrix on the copy stream (an event
// after each chunk), then the grouped kernels phase by phase, each after its
// chunk's event.  Phase 0 holds the cached experts and the shared experts.
#include <algorithm>
#include <cstring>
#include <vector>

#include "stream_cache.h"


namespace dqmoe {

namespace {
size_t align256(size_t v) { return (v + 255) / 256 * 256; }
}  // namespace

// device tables after the layer's own workspace
size_t stream_workspace(const dq_expert_cache& c, int T, size_t* off_slot, size_t* off_phase) {
  const size_t base = moe_plan(c.d, T, false).total;
  *off_slot = base;
  *off_phase = align256(base + (size_t)c.d.E * 4);
  return align256(*off_phase + (size_t)c.d.E);
}

int stream_cache_init(dq_expert_cache* c, const dq_moe_desc& d, int slots, void* sg, void* su,
                      void* sd, int max_tokens, int phases, int64_t gu_bytes, int64_t dn_bytes) {
  c->d = d;
  c->slots = slots;
  c->max_tokens = max_tokens;
  c->phases = phases;
  c->slot_gate = sg;
  c->slot_up = su;
  c->slot_down = sd;
  c->gu_bytes = gu_bytes;
  c->dn_bytes = dn_bytes;
  c->slot_expert.assign(slots, -1);
  c->expert_slot.assign(d.E, -1);
  c->last_use.assign(slots, -1);
  c->calls = 0;
  c->hits = c->misses = c->bytes_copied = 0;
  c->h_idx = nullptr;
  c->h_slot = nullptr;
  c->h_phase = nullptr;
  for (int i = 0; i < kMaxStreamPhases; ++i) c->gu_ready[i] = c->dn_ready[i] = nullptr;
  if (cudaHostAlloc((void**)&c->h_idx, (size_t)max_tokens * d.top_k * 4, cudaHostAllocDefault) !=
          cudaSuccess ||
      cudaHostAlloc((void**)&c->h_slot, (size_t)d.E * 4, cudaHostAllocDefault) != cudaSuccess ||
      cudaHostAlloc((void**)&c->h_phase, (size_t)d.E, cudaHostAllocDefault) != cudaSuccess)
    return DQ_ERR_CUDA;
  for (int i = 0; i < kMaxStreamPhases; ++i)
    if (cudaEventCreateWithFlags(&c->gu_ready[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->dn_ready[i], cudaEventDisableTiming) != cudaSuccess)
      return DQ_ERR_CUDA;
  return DQ_OK;
}

void stream_cache_release(dq_expert_cache* c) {
  if (c->h_idx) cudaFreeHost(c->h_idx);
  if (c->h_slot) cudaFreeHost(c->h_slot);
  if (c->h_phase) cudaFreeHost(c->h_phase);
  for (int i = 0; i < kMaxStreamPhases; ++i) {
    if (c->gu_ready[i]) cudaEventDestroy(c->gu_ready[i]);
    if (c->dn_ready[i]) cudaEventDestroy(c->dn_ready[i]);
  }
}

int stream_forward(dq_expert_cache* c, const void* x, int xdt, int T, float* y, void* ws,
                   cudaStream_t s, cudaStream_t cs) {
  const dq_moe_desc& d = c->d;
  const MoePlan pl = moe_plan(d, T, false);
  size_t off_slot, off_phase;
  stream_workspace(*c, T, &off_slot, &off_phase);
  uint8_t* w = (uint8_t*)ws;
  MoeStream ms;
  memset(&ms, 0, sizeof(ms));
  ms.slot_of = (const int*)(w + off_slot);
  ms.phase_of = (const int8_t*)(w + off_phase);
  ms.slot_gate = c->slot_gate;
  ms.slot_up = c->slot_up;
  ms.slot_down = c->slot_down;
  ms.slots = c->slots;

  // 1. routing on the device, read back
  int rc = launch_moe_forward(d, x, xdt, T, y, ws, nullptr, nullptr, nullptr, s, &ms, 1);
  if (rc != DQ_OK) return rc;
  const int P = T * d.top_k;
  if (cudaMemcpyAsync(c->h_idx, w + pl.off_idx, (size_t)P * 4, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return DQ_ERR_CUDA;

  // 2. cache bookkeeping: experts of this call in order of first use
  const long long now = ++c->calls;
  std::vector<int> need, miss;
  std::vector<char> seen(d.E, 0);
  for (int i = 0; i < P; ++i) {
    const int e = c->h_idx[i];
    if (e < 0 || e >= d.E) return DQ_ERR_CUDA;   // routing outside [0, E): not ours to stream
    if (!seen[e]) {
      seen[e] = 1;
      need.push_back(e);
    }
  }
  for (int e : need) {
    const int sl = c->expert_slot[e];
    if (sl >= 0) c->last_use[sl] = now;
    else miss.push_back(e);
  }
  for (int e : miss) {
    // a free slot, else the least recently used one not needed by this call
    int best = -1;
    for (int sl = 0; sl < c->slots; ++sl) {
      if (c->last_use[sl] == now) continue;
      if (best < 0 || c->last_use[sl] < c->last_use[best]) best = sl;
    }
    if (best < 0) return DQ_ERR_UNSUPPORTED;   // more experts than slots (checked at creation)
    if (c->slot_expert[best] >= 0) c->expert_slot[c->slot_expert[best]] = -1;
    c->slot_expert[best] = e;
    c->expert_slot[e] = best;
    c->last_use[best] = now;
  }
  c->hits += (long long)(need.size() - miss.size());
  c->misses += (long long)miss.size();

  // 3. phases: 0 = cached experts (and the shared ones); the missing experts
  // split in order into up to phases-1 chunks (all in phase 0 with phases = 1)
  const int nm = (int)miss.size();
  const int chunks = c->phases == 1 ? (nm > 0 ? 1 : 0) : std::min(c->phases - 1, nm);
  ms.nphase = c->phases == 1 ? 1 : 1 + chunks;
  memset(c->h_phase, -1, (size_t)d.E);
  for (int e : need) c->h_phase[e] = 0;
  for (int e = 0; e < d.E; ++e) c->h_slot[e] = c->expert_slot[e] < 0 ? 0 : c->expert_slot[e];
  std::vector<int> chunk_of(nm);
  for (int i = 0; i < nm; ++i) {
    const int ch = chunks ? (int)((int64_t)i * chunks / nm) : 0;
    chunk_of[i] = ch;
    c->h_phase[miss[i]] = (int8_t)(c->phases == 1 ? 0 : 1 + ch);
  }

  // 4. copies: every chunk's gate and up first (needed first), then its down
  const uint8_t* hg = (const uint8_t*)d.w_gate;
  const uint8_t* hu = (const uint8_t*)d.w_up;
  const uint8_t* hd = (const uint8_t*)d.w_down;
  for (int ch = 0; ch < chunks; ++ch) {
    for (int i = 0; i < nm; ++i) {
      if (chunk_of[i] != ch) continue;
      const int e = miss[i], sl = c->expert_slot[e];
      if (cudaMemcpyAsync((uint8_t*)c->slot_gate + (int64_t)sl * c->gu_bytes,
                          hg + (int64_t)e * c->gu_bytes, (size_t)c->gu_bytes,
                          cudaMemcpyHostToDevice, cs) != cudaSuccess ||
          cudaMemcpyAsync((uint8_t*)c->slot_up + (int64_t)sl * c->gu_bytes,
                          hu + (int64_t)e * c->gu_bytes, (size_t)c->gu_bytes,
                          cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return DQ_ERR_CUDA;
      c->bytes_copied += 2 * c->gu_bytes;
    }
    const int ph = c->phases == 1 ? 0 : 1 + ch;
    if (cudaEventRecord(c->gu_ready[ph], cs) != cudaSuccess) return DQ_ERR_CUDA;
    ms.gu_ready[ph] = c->gu_ready[ph];
  }
  for (int ch = 0; ch < chunks; ++ch) {
    for (int i = 0; i < nm; ++i) {
      if (chunk_of[i] != ch) continue;
      const int e = miss[i], sl = c->expert_slot[e];
      if (cudaMemcpyAsync((uint8_t*)c->slot_down + (int64_t)sl * c->dn_bytes,
                          hd + (int64_t)e * c->dn_bytes, (size_t)c->dn_bytes,
                          cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return DQ_ERR_CUDA;
      c->bytes_copied += c->dn_bytes;
    }
    const int ph = c->phases == 1 ? 0 : 1 + ch;
    if (cudaEventRecord(c->dn_ready[ph], cs) != cudaSuccess) return DQ_ERR_CUDA;
    ms.dn_ready[ph] = c->dn_ready[ph];
  }

  // 5. the tables, then permute, the experts phase by phase, combine
  if (cudaMemcpyAsync(w + off_slot, c->h_slot, (size_t)d.E * 4, cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaMemcpyAsync(w + off_phase, c->h_phase, (size_t)d.E, cudaMemcpyHostToDevice, s) !=
          cudaSuccess)
    return DQ_ERR_CUDA;
  return launch_moe_forward(d, x, xdt, T, y, ws, nullptr, nullptr, nullptr, s, &ms, 2);
}

}  // namespace dqmoe
