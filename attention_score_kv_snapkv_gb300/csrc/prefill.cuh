// Launcher of the prompt self-attention with SnapKV votes (prefill.cu).
#pragma once
#include "kvc_internal.cuh"

namespace kvc {

struct PrefillArgs {
  const void *q;      // [Uq, L, D] bf16, Uq = layers * batch * query heads
  const void *k, *v;  // [Ukv, L, D] bf16, Ukv = Uq / G
  void *o;            // [Uq, L, D] bf16 output
  float *votes;       // [Ukv, L] fp32 or null (zeroed here before the launch)
  float *lse;         // [Uq, L] fp32 or null: each row's log-sum-exp of its causal scores
  int units_q, G, L, D, Wq;
};
cudaError_t launch_prefill(const Ctx &c, const PrefillArgs &a);

}  // namespace kvc
