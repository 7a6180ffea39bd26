// moe_plan.h — workspace layout of dq_moe_forward (host side, shared by the
// C-ABI validation in api.cu and the launch sequence in moe.cu).
#pragma once

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
  size_t off_part, off_logits, off_idx, off_gate, off_offsets, off_sorted, off_inv, off_tok,
      off_groups, off_ngroups, off_h, off_ypos, off_units, off_nunits, off_x16t, off_xinvt,
      off_x16, off_xinv, off_g, off_u, off_h16, off_hinv, total;
};

MoePlan moe_plan(const dq_moe_desc& d, int T);

}  // namespace dqmoe
