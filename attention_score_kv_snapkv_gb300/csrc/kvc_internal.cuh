// Internal declarations of libkvcompress: device helpers (inline PTX for mbarrier,
// TMA bulk-tensor copies and tcgen05 tensor-core MMA with TMEM accumulators), bounded
// waits, and the host-side launch functions each kernel file exports to kvc_api.cu.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/kvcompress.h"

namespace kvc {

// ------------------------------------------------------------------------------
// Launch context shared by every kernel launch.
// ------------------------------------------------------------------------------
struct Ctx {
  cudaStream_t stream;
  uint32_t *status;              // device status word (KVC_DEV_* bits)
  unsigned long long timeout_ns; // limit of every device-side wait
  int num_sms;
};

// A named NVTX range around one C-ABI call (shows each entry point on a profiler's
// timeline; costs nothing measurable when no tool is attached).
struct TraceRange {
  explicit TraceRange(const char *name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange &) = delete;
  TraceRange &operator=(const TraceRange &) = delete;
};

// ------------------------------------------------------------------------------
// Small device helpers.
// ------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair (packed in a uint32) -> two floats.  bf16 is the upper half of an fp32.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// packed fp32x2 helpers: a 64-bit register holds two fp32 lanes
__device__ __forceinline__ unsigned long long pk(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 upk(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
// d += a * b, lane-wise on two fp32 values
__device__ __forceinline__ void ffma2(unsigned long long &d, unsigned long long a,
                                      unsigned long long b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
// d = a * b + c, lane-wise
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// d = a + b, lane-wise
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits) {
  atomicOr(status, bits);
}

// ------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits until the phase with parity `parity` of the barrier has completed, for at most
// `limit_ns` nanoseconds (and at most 2^26 polls).  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1; it < (1u << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// A CTA-wide abort flag in shared memory plus the device status word: the first wait
// that runs out raises both; every later wait of the CTA returns false immediately so
// the CTA drains quickly.
struct Abort {
  volatile int *flag;      // shared memory
  uint32_t *status;        // global status word
  unsigned long long limit;

  __device__ __forceinline__ bool raised() const { return *flag != 0; }
  __device__ __forceinline__ void raise() const {
    *flag = 1;
    set_status(status, KVC_DEV_TIMEOUT);
  }
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (*flag) return false;
    if (mbar_wait_bounded(bar, parity, limit)) return true;
    raise();
    return false;
  }
};

// *ctr += v with release semantics at GPU scope: every write that happens before it in
// this thread -- including other threads' writes ordered before it by a CTA barrier --
// is visible to a thread that reads the new count with acquire semantics.
__device__ __forceinline__ void red_release_gpu(int *ctr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ctr), "r"(v) : "memory");
}

// Spin (bounded) until *ctr >= target with acquire semantics at GPU scope.  Gives up early
// if another CTA has already flagged a timeout in the status word.
__device__ __forceinline__ bool spin_count_bounded(const int *ctr, int target,
                                                   const uint32_t *status,
                                                   unsigned long long limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (*(volatile const uint32_t *)status & KVC_DEV_TIMEOUT) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
    __nanosleep(64);
  }
  return false;
}

// ------------------------------------------------------------------------------
// TMA (bulk tensor copy global -> shared, completion counted on an mbarrier)
// ------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// The same with an L2 cache policy (from l2_policy_*): how long L2 should keep the lines.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int32_t x,
                                                 int32_t y, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
// L2 policies: keep the lines ahead of normal ones (data read again soon), or let them go
// first (data read for the last time).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA (kind::f16, bf16 inputs, fp32 accumulator), loads.
// ------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 operand stored as rows of 128
// bytes with the 128-byte swizzle (the layout a TMA load with SWIZZLE_128B writes):
// 8-row core groups 1024 bytes apart (stride byte offset), descriptor version 1,
// layout type 2 = SWIZZLE_128B.  The leading byte offset is unused for this layout.
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A and B bf16, both K-major,
// shape M x N (M = 128; N a multiple of 16 in [16, 256]).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32-bit, 16 consecutive columns: thread i of the warp gets lane
// (warp quarter base + i), columns taddr.col .. +15, into v[0..15].
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Same with 8 consecutive columns into v[0..7].
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float *v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Same with 32 consecutive columns into v[0..31].
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Named barrier among `nthreads` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------------------
// Host-side launchers (one per kernel file).  All return cudaError_t of the launch.
// ------------------------------------------------------------------------------

// window_vote.cu: steps 1-2 of SnapKV (and H2O's prompt scores).
struct WindowVoteArgs {
  const void *q;   // [U * R, D] bf16, R = G * Wq rows per unit
  const void *k;   // [U * L, D] bf16
  int units, L, R, Wq, D;
  float *votes;    // [U, L] fp32 (zeroed here when several row tiles add into it)
  void *ws;        // workspace (statistics exchange), WindowVotePlan::ws_bytes bytes
};
struct WindowVotePlan {
  int single = 0;    // 1: the single-pass kernel (window_vote_tmem.cu), 0: two passes
  int row_tiles, jobs, g, ngroups, min_nkt, max_nkt;
  int qr = 128;      // single pass: query rows per Q tile and per tensor-memory buffer
  size_t ws_bytes;
};
// The single-pass plan when every CTA's share of a job fits its tensor memory, else the
// two-pass plan.
WindowVotePlan plan_window_vote(int units, int L, int R, int Wq, int num_sms);
cudaError_t launch_window_vote(const Ctx &c, const WindowVoteArgs &a);
// window_vote_tmem.cu: false if no group size fits tensor memory.
bool plan_window_vote_tmem(int units, int L, int R, int Wq, int num_sms, WindowVotePlan *pl);
cudaError_t launch_window_vote_tmem(const Ctx &c, const WindowVoteArgs &a,
                                    const WindowVotePlan &pl);

// window_vote_lse.cu: step 2 when each voting row's log-sum-exp is already known.
struct WindowVoteLseArgs {
  const void *q;      // [U * R, D] bf16, R = G * Wq rows per unit
  const void *k;      // [U * L, D] bf16
  const float *lse;   // [U, G, L] fp32 natural-log log-sum-exp of every prompt row
  int units, L, G, Wq, D;
  float *votes;       // [U, L] fp32 (zeroed here when several row tiles add into it)
};
cudaError_t launch_window_vote_lse(const Ctx &c, const WindowVoteLseArgs &a);

// select.cu: steps 3-4 (pool + top-k + gather).
struct SelectArgs {
  const float *votes;   // [U, L]
  const void *k, *v;    // [U, L, D]
  void *k_out, *v_out;  // [U, cap, D]
  int32_t *pos_out;     // [U, cap]
  int32_t *n_valid_out; // [U]
  float *kept_scores;   // [U, cap] or null
  int units, L, D, keep_window, pool_kernel, budget, cap;
  int pool_avg;         // 1: average pool (window sum / P, zeros past the ends), 0: max
  int identity;         // keep every position (budget >= L or W_keep >= L)
  int32_t *sel_ws;      // [U, cap] scratch for the selected positions
};
size_t select_ws_bytes(int units, int L, int keep_window, int cap);
cudaError_t launch_select_gather(const Ctx &c, const SelectArgs &a);

// decode.cu: decode attention over a compact / ring cache (+ optional append).
struct DecodeArgs {
  const void *q;        // [U*G, D]
  const void *k_new, *v_new; // [U, D] or null
  void *k_cache, *v_cache;   // [U, cap, D]
  int32_t *pos;         // [U, cap] or null
  int32_t *n_valid;     // [U] or null
  void *out;            // [U*G, D]
  void *ws;
  int units, G, D, cap, n_uniform, new_pos;
};
size_t decode_ws_bytes(int units, int G, int D, int cap, int num_sms);
// bytes at the start of the workspace holding the per-unit split-K counters
size_t decode_counter_bytes(int units);
cudaError_t launch_decode(const Ctx &c, const DecodeArgs &a);

// h2o.cu: one H2O decode step.
struct H2OArgs {
  const void *q;        // [U*G, D]
  const void *k_new, *v_new; // [U, D]
  void *k, *v;          // [U, S, D]
  float *score;         // [U, S]
  int32_t *pos;         // [U, S]
  int32_t *n_used, *free_slot; // [U]
  void *out;            // [U*G, D]
  int32_t *evicted;     // [U] or null
  int units, G, D, slots, n_recent, t;
  int split;            // 1: the split step (several CTAs per unit) in `scratch`
  void *scratch;        // plan_h2o_split(...).scratch_bytes, zero between calls
};
cudaError_t launch_h2o_step(const Ctx &c, const H2OArgs &a);
// The split step's geometry: CTAs per unit, rows per CTA, scratch bytes; feasible is
// false when a CTA's rows would not fit its shared memory.
struct H2OSplitPlan {
  int nsplit, chunk;
  bool feasible;
  size_t scratch_bytes;
};
H2OSplitPlan plan_h2o_split(long long units, int G, int D, int slots, int num_sms);
// Whether one CTA per unit keeps a unit's logits in shared memory.
bool h2o_single_fits(int G, int D, long long slots);
cudaError_t launch_h2o_init_state(const Ctx &c, int32_t *pos, int32_t *n_used,
                                  int32_t *free_slot, const int32_t *n_valid, int units,
                                  int slots);

// sink.cu: StreamingLLM ring append.
cudaError_t launch_sink_append(const Ctx &c, const void *k_new, const void *v_new, void *k_cache,
                               void *v_cache, int32_t *pos, int units, int D, int rows,
                               int slot, int64_t t);

// selftest.cu
cudaError_t run_selftest_wait(const Ctx &c, int *result);

// kvc_api.cu: tensor-map encoding shared by the TMA kernels.
bool encode_rows_map(CUtensorMap *map, const void *base, uint64_t rows, int D, int box_rows);
// kvc_api.cu: compressed_decode_attn, optionally clearing the workspace's split-K
// counters right before the launch (after every argument check has passed).
kvc_status decode_call(const kvc_decode_params *p, const void *q, const void *k_new,
                       const void *v_new, void *k_cache, void *v_cache, int32_t *pos,
                       int32_t *n_valid, void *out, void *workspace, size_t workspace_bytes,
                       kvc_stream_t stream, bool clear_counters);
// kvc_api.cu: KVC_OK if the current device is supported (sm_103), else its error.
kvc_status device_check(kvc_stream_t stream);
// kvc_api.cu: the causal prefill attention with optional votes and per-row log-sum-exp.
kvc_status prefill_call(const kvc_snapkv_params *p, const void *q, const void *k, const void *v,
                        void *o_out, float *votes_out, float *lse_out, kvc_stream_t stream);

}  // namespace kvc
