// stream_cache.h — state of the streamed MoE layer (one per expert cache):
// the host-resident experts, the device slot buffers, the least-recently-used
// bookkeeping, page-locked staging for the routing read-back and the tables,
// and the copy-completion events of each phase.
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "moe_plan.h"

struct dq_expert_cache {
  dq_moe_desc d;          // w_gate / w_up / w_down: page-locked host memory
  int slots, max_tokens, phases;
  void* slot_gate;
  void* slot_up;
  void* slot_down;
  int64_t gu_bytes;       // one expert's gate (= up) matrix
  int64_t dn_bytes;       // one expert's down matrix
  std::vector<int> slot_expert;     // expert held by each slot, -1: free
  std::vector<int> expert_slot;     // slot of each expert, -1: not cached
  std::vector<long long> last_use;  // per slot: call counter of its last use
  long long calls;
  int32_t* h_idx;         // page-locked [max_tokens * top_k]
  int32_t* h_slot;        // page-locked [E]
  int8_t* h_phase;        // page-locked [E]
  cudaEvent_t gu_ready[dqmoe::kMaxStreamPhases];
  cudaEvent_t dn_ready[dqmoe::kMaxStreamPhases];
  long long hits, misses, bytes_copied;
};
