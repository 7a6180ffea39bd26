// moe_plan.h — workspace layout of dq_moe_forward (host side, shared by the
// C-ABI validation in api.cu and the launch sequence in moe.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dqmoe.h"

namespace dqmoe {

struct MoePlan {
  int KS;           // router hidden-dimension split
  int64_t P;        // routed (token, slot) pairs = T * top_k
  int64_t NP;       // positions: P routed + n_shared * T shared
  int NT;           // 8-column activation tiles per grouped-GEMV unit (1, 2, 4)
  int GW;           // group width = 8 * NT columns
  int G_max;        // upper bound of narrow work groups (<= GW columns, mma.sync path)
  int U_max;        // upper bound of wide units (<= 128 columns, tcgen05 path)
  bool wide;        // wide units are possible (some expert may get > 32 tokens)
  bool single;      // one-token groups run on the block-diagonal kernel (moe_b1.cu)
  int G1_max;       // upper bound of one-token groups
  int DS;           // K parts of the grouped down products (ypos holds DS copies)
  size_t off_part, off_logits, off_idx, off_gate, off_offsets, off_sorted, off_inv, off_tok,
      off_groups, off_ngroups, off_h, off_ypos, off_units, off_nunits, off_x16t, off_xinvt,
      off_x16, off_xinv, off_g, off_u, off_h16, off_hinv, off_g1, off_ng1, total;
};

// allow_wide = false keeps every expert on the grouped mma.sync kernel (the
// streamed layer, whose experts live in a slot cache).
MoePlan moe_plan(const dq_moe_desc& d, int T, bool allow_wide = true);

// The streamed layer's expert cache as the launch sequence sees it: routed
// expert e's gate/up/down sit in slot slot_of[e] of the slot buffers, and its
// units run in copy/compute phase phase_of[e] (both device arrays of E).
constexpr int kMaxStreamPhases = 8;
struct MoeStream {
  const int* slot_of;
  const int8_t* phase_of;
  int nphase;
  cudaEvent_t gu_ready[kMaxStreamPhases];   // gate/up of the phase copied (null: none)
  cudaEvent_t dn_ready[kMaxStreamPhases];   // down of the phase copied (null: none)
  const void* slot_gate;
  const void* slot_up;
  const void* slot_down;
  int slots;
};

// The one-token expert kernels (moe_b1.cu).
bool grouped_b1_supported(int fmt);
int launch_grouped_b1(bool gateup, const dq_moe_desc& d, const int4* groups1,
                      const int* n_groups1, int g1_max, int* claim, const void* x, int xdt,
                      int64_t xstride, float* out, int64_t out_stride, cudaStream_t s);

// side: the general expert kernels may run on a second stream beside the
// one-token ones (created on first use; dq_moe_forward_noalloc passes false).
int launch_moe_forward(const dq_moe_desc& d, const void* x, int xdt, int T, float* y, void* ws,
                       int32_t* topk_idx, float* topk_gate, float* logits, cudaStream_t s,
                       const MoeStream* ms = nullptr, int stages = 3, bool side = true);

// dq_moe_forward's argument checks and launch, with the side-stream choice.
int moe_forward_checked(const dq_moe_desc* desc, const void* x, int x_dtype, int T, float* y,
                        void* ws, size_t ws_bytes, int32_t* topk_idx, float* topk_gate,
                        float* logits, void* stream, bool side);

}  // namespace dqmoe

struct dq_expert_cache;   // the streamed layer's state (csrc/stream.cu)

namespace dqmoe {
size_t stream_workspace(const ::dq_expert_cache& c, int T, size_t* off_slot, size_t* off_phase);
int stream_cache_init(::dq_expert_cache* c, const dq_moe_desc& d, int slots, void* sg, void* su,
                      void* sd, int max_tokens, int phases, int64_t gu_bytes, int64_t dn_bytes);
void stream_cache_release(::dq_expert_cache* c);
int stream_forward(::dq_expert_cache* c, const void* x, int xdt, int T, float* y, void* ws,
                   cudaStream_t s, cudaStream_t cs);
}  // namespace dqmoe
