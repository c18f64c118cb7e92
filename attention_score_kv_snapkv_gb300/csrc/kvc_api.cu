// C ABI of libkvcompress (declared and documented in include/kvcompress.h): host-side
// argument checks, workspace layout, TMA tensor maps and kernel launches.  Nothing here
// allocates or frees device memory; the caller owns every buffer and the stream.
#include <math.h>
#include <string.h>

#include <cudaTypedefs.h>

#include <mutex>

#include "kvc_internal.cuh"
#include "prefill.cuh"

namespace kvc {

namespace {

__device__ uint32_t g_status;  // per-device status word (KVC_DEV_* bits)

struct DevInfo {
  bool init = false;
  bool supported = false;
  int num_sms = 0;
  uint32_t *status = nullptr;
};

constexpr int MAX_DEV = 64;
DevInfo g_dev[MAX_DEV];
std::mutex g_mu;
unsigned long long g_timeout_ns = 1000000000ull;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Context of the current device; KVC_ERR_UNSUPPORTED unless it is an sm_103 GPU.
kvc_status get_ctx(kvc_stream_t stream, Ctx *c) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEV) return KVC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo &d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return KVC_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.num_sms = sms;
    if (d.supported) {
      void *addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_status) != cudaSuccess) return KVC_ERR_CUDA;
      d.status = reinterpret_cast<uint32_t *>(addr);
    }
    d.init = true;
  }
  if (!d.supported) return KVC_ERR_UNSUPPORTED;
  c->stream = reinterpret_cast<cudaStream_t>(stream);
  c->status = d.status;
  c->timeout_ns = g_timeout_ns;
  c->num_sms = d.num_sms;
  return KVC_OK;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }
inline kvc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA; }

const long long kMaxRows = (1ll << 31) - 1;

bool common_heads_ok(int Ly, int B, int Hq, int Hkv, int D) {
  return Ly >= 1 && B >= 1 && Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0 && (D == 64 || D == 128) &&
         Hq / Hkv <= 4096;
}

// Derived sizes of a snapkv_compress call.
struct SnapPlan {
  long long units;
  int G, R;
  bool identity, need_votes;
  int n_keep;
  size_t wv_bytes, votes_bytes, sel_bytes, total;
};

kvc_status plan_snapkv(const kvc_snapkv_params *p, bool want_scores, int num_sms, SnapPlan *s) {
  if (!p) return KVC_ERR_NULL;
  if (!common_heads_ok(p->n_layers, p->batch, p->n_q_heads, p->n_kv_heads, p->head_dim))
    return KVC_ERR_SHAPE;
  if (p->prompt_len < 1 || p->n_query < 1 || p->n_query > p->prompt_len || p->keep_window < 0 ||
      p->pool_kernel < 1 || (p->pool_kernel & 1) == 0 || p->budget < 1 || p->cap < 1 ||
      (p->pool_avg != 0 && p->pool_avg != 1))
    return KVC_ERR_SHAPE;
  s->units = (long long)p->n_layers * p->batch * p->n_kv_heads;
  s->G = p->n_q_heads / p->n_kv_heads;
  if ((long long)s->G * p->n_query > kMaxRows) return KVC_ERR_SHAPE;
  s->R = s->G * p->n_query;
  if (s->units * p->prompt_len > kMaxRows || s->units * s->R > kMaxRows ||
      s->units * p->cap > kMaxRows || p->cap > 65535 * 32)  // the gather's grid: cap / 32 <= 65535
    return KVC_ERR_SHAPE;
  s->identity = p->budget >= p->prompt_len || p->keep_window >= p->prompt_len;
  if (!s->identity && p->budget < p->keep_window) return KVC_ERR_BUDGET;
  s->n_keep = s->identity ? p->prompt_len : p->budget;
  if (p->cap < s->n_keep) return KVC_ERR_BUDGET;
  s->need_votes = !s->identity || want_scores;
  const int nsm = num_sms > 0 ? num_sms : 1;
  s->wv_bytes = s->need_votes
                    ? plan_window_vote((int)s->units, p->prompt_len, s->R, p->n_query, nsm).ws_bytes
                    : 0;
  s->votes_bytes = align256((size_t)s->units * p->prompt_len * sizeof(float));
  s->sel_bytes = select_ws_bytes((int)s->units, p->prompt_len, p->keep_window, p->cap);
  s->total = align256(s->wv_bytes) + s->votes_bytes + s->sel_bytes;
  return KVC_OK;
}

// SM count of the current device for sizing queries, or 160 without a usable device (a
// failed lookup's error is cleared so that the caller's own error checks do not see it).
int sms_for_sizing() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 160;
  }
  return sms > 0 ? sms : 160;
}

// votes_in: votes computed elsewhere (the prefill attention); then q_win is not read and
// the window vote does not run.
kvc_status run_snapkv(const kvc_snapkv_params *p, const void *q_win, const void *k, const void *v,
                      void *k_out, void *v_out, int32_t *pos_out, int32_t *n_valid_out,
                      float *votes_out, float *kept_scores_out, void *workspace,
                      size_t workspace_bytes, kvc_stream_t stream, const float *votes_in = nullptr) {
  Ctx c;
  kvc_status st = get_ctx(stream, &c);
  if (st != KVC_OK) return st;
  SnapPlan s;
  st = plan_snapkv(p, kept_scores_out != nullptr || votes_out != nullptr, c.num_sms, &s);
  if (st != KVC_OK) return st;
  if ((!q_win && !votes_in) || !k || !v || !k_out || !v_out || !pos_out || !n_valid_out)
    return KVC_ERR_NULL;
  if ((q_win && !aligned16(q_win)) || (votes_in && !aligned4(votes_in)) || !aligned16(k) || !aligned16(v) || !aligned16(k_out) ||
      !aligned16(v_out) || !aligned4(pos_out) || !aligned4(n_valid_out) ||
      (votes_out && !aligned4(votes_out)) || (kept_scores_out && !aligned4(kept_scores_out)))
    return KVC_ERR_ALIGN;
  if (!workspace || workspace_bytes < s.total) return KVC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KVC_ERR_ALIGN;
  if (!g_encode) return KVC_ERR_CUDA;
  // v may be page-locked host memory mapped for the device: the gather reads it there
  cudaPointerAttributes va;
  if (cudaPointerGetAttributes(&va, v) != cudaSuccess) {
    (void)cudaGetLastError();
    return KVC_ERR_UNSUPPORTED;
  }
  if (va.type == cudaMemoryTypeHost) {
    if (!va.devicePointer || !aligned16(va.devicePointer)) return KVC_ERR_UNSUPPORTED;
    v = va.devicePointer;
  } else if (va.type != cudaMemoryTypeDevice && va.type != cudaMemoryTypeManaged) {
    return KVC_ERR_UNSUPPORTED;
  }

  uint8_t *w = reinterpret_cast<uint8_t *>(workspace);
  void *wv_ws = w;
  float *votes = votes_out ? votes_out : reinterpret_cast<float *>(w + align256(s.wv_bytes));
  int32_t *sel_ws = reinterpret_cast<int32_t *>(w + align256(s.wv_bytes) + s.votes_bytes);
  if (votes_in) {
    if (votes_out && votes_out != votes_in)
      if (cudaMemcpyAsync(votes_out, votes_in, (size_t)s.units * p->prompt_len * sizeof(float),
                          cudaMemcpyDeviceToDevice, c.stream) != cudaSuccess)
        return KVC_ERR_CUDA;
    votes = const_cast<float *>(votes_in);
  }

  if (s.need_votes && !votes_in) {
    WindowVoteArgs a;
    a.q = q_win;
    a.k = k;
    a.units = (int)s.units;
    a.L = p->prompt_len;
    a.R = s.R;
    a.Wq = p->n_query;
    a.D = p->head_dim;
    a.votes = votes;
    a.ws = wv_ws;
    st = cuda_status(launch_window_vote(c, a));
    if (st != KVC_OK) return st;
  }
  SelectArgs sa;
  sa.votes = votes;
  sa.k = k;
  sa.v = v;
  sa.k_out = k_out;
  sa.v_out = v_out;
  sa.pos_out = pos_out;
  sa.n_valid_out = n_valid_out;
  sa.kept_scores = kept_scores_out;
  sa.units = (int)s.units;
  sa.L = p->prompt_len;
  sa.D = p->head_dim;
  sa.keep_window = p->keep_window;
  sa.pool_kernel = p->pool_kernel;
  sa.pool_avg = p->pool_avg;
  sa.budget = p->budget;
  sa.cap = p->cap;
  sa.identity = s.identity ? 1 : 0;
  sa.sel_ws = sel_ws;
  return cuda_status(launch_select_gather(c, sa));
}

}  // namespace

bool encode_rows_map(CUtensorMap *map, const void *base, uint64_t rows, int D, int box_rows) {
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace kvc

using namespace kvc;

namespace {
void ensure_encode() { std::call_once(g_encode_once, load_encode); }
}  // namespace

namespace kvc {

// compressed_decode_attn with an option to clear the split-K counters of the workspace
// first (after every argument check has passed, right before the launch).
kvc_status decode_call(const kvc_decode_params *p, const void *q, const void *k_new,
                       const void *v_new, void *k_cache, void *v_cache, int32_t *pos,
                       int32_t *n_valid, void *out, void *workspace, size_t workspace_bytes,
                       kvc_stream_t stream, bool clear_counters) {
  ensure_encode();
  Ctx c;
  kvc_status st = get_ctx(stream, &c);
  if (st != KVC_OK) return st;
  if (!p) return KVC_ERR_NULL;
  if (!common_heads_ok(p->n_layers, p->batch, p->n_q_heads, p->n_kv_heads, p->head_dim) ||
      p->cap < 1)
    return KVC_ERR_SHAPE;
  const int G = p->n_q_heads / p->n_kv_heads;
  if (G > 8) return KVC_ERR_SHAPE;  // query heads per KV head: 1..8
  const long long units = (long long)p->n_layers * p->batch * p->n_kv_heads;
  if (units * p->cap > kMaxRows || units > 65535ll * 32768ll) return KVC_ERR_SHAPE;
  if (p->n_uniform < 0 || p->n_uniform > p->cap) return KVC_ERR_SHAPE;
  if (!q || !k_cache || !v_cache || !out) return KVC_ERR_NULL;
  if ((k_new == nullptr) != (v_new == nullptr)) return KVC_ERR_NULL;
  if (k_new && !n_valid) return KVC_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (k_new && (!aligned16(k_new) || !aligned16(v_new))) || (pos && !aligned4(pos)) ||
      (n_valid && !aligned4(n_valid)))
    return KVC_ERR_ALIGN;
  const size_t need = decode_ws_bytes((int)units, G, p->head_dim, p->cap, c.num_sms);
  if (!workspace || workspace_bytes < need) return KVC_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVC_ERR_ALIGN;
  if (!g_encode) return KVC_ERR_CUDA;
  if (units > KVC_DECODE_MAX_UNITS) return KVC_ERR_SHAPE;  // one split-K counter per unit
  DecodeArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.pos = pos;
  a.n_valid = n_valid;
  a.out = out;
  a.ws = workspace;
  a.units = (int)units;
  a.G = G;
  a.D = p->head_dim;
  a.cap = p->cap;
  a.n_uniform = p->n_uniform;
  a.new_pos = p->new_pos;
  if (clear_counters &&
      cudaMemsetAsync(workspace, 0, decode_counter_bytes((int)units), c.stream) != cudaSuccess)
    return KVC_ERR_CUDA;
  return cuda_status(launch_decode(c, a));
}

kvc_status device_check(kvc_stream_t stream) {
  Ctx c;
  return get_ctx(stream, &c);
}

// The causal prefill attention with optional votes of the last n_query rows and optional
// per-row log-sum-exp.
kvc_status prefill_call(const kvc_snapkv_params *p, const void *q, const void *k, const void *v,
                        void *o_out, float *votes_out, float *lse_out, kvc_stream_t stream) {
  ensure_encode();
  Ctx c;
  kvc_status st = get_ctx(stream, &c);
  if (st != KVC_OK) return st;
  if (!p) return KVC_ERR_NULL;
  if (!common_heads_ok(p->n_layers, p->batch, p->n_q_heads, p->n_kv_heads, p->head_dim) ||
      p->prompt_len < 1 || (votes_out && (p->n_query < 1 || p->n_query > p->prompt_len)))
    return KVC_ERR_SHAPE;
  const long long uq = (long long)p->n_layers * p->batch * p->n_q_heads;
  if (uq * p->prompt_len > kMaxRows) return KVC_ERR_SHAPE;
  if (!q || !k || !v || !o_out) return KVC_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_out) ||
      (votes_out && !aligned4(votes_out)) || (lse_out && !aligned4(lse_out)))
    return KVC_ERR_ALIGN;
  if (!g_encode) return KVC_ERR_CUDA;
  PrefillArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o_out;
  a.votes = votes_out;
  a.lse = lse_out;
  a.units_q = (int)uq;
  a.G = p->n_q_heads / p->n_kv_heads;
  a.L = p->prompt_len;
  a.D = p->head_dim;
  a.Wq = votes_out ? p->n_query : 1;
  return cuda_status(launch_prefill(c, a));
}


// h2o_prefill from the prompt's queries (q) or from column sums computed elsewhere (votes).
kvc_status h2o_prefill_call(const kvc_h2o_params *p, int32_t prompt_len, const void *q,
                            const float *votes, const void *k, const void *v,
                            const kvc_h2o_state *st, void *workspace, size_t workspace_bytes,
                            kvc_stream_t stream) {
  ensure_encode();
  if (!p || !st) return KVC_ERR_NULL;
  if (p->n_heavy < 0 || p->n_recent < 1) return KVC_ERR_SHAPE;
  if (!st->k || !st->v || !st->score || !st->pos || !st->n_used || !st->free_slot)
    return KVC_ERR_NULL;
  if (!aligned4(st->n_used) || !aligned4(st->free_slot)) return KVC_ERR_ALIGN;
  kvc_snapkv_params s;
  s.n_layers = p->n_layers;
  s.batch = p->batch;
  s.n_q_heads = p->n_q_heads;
  s.n_kv_heads = p->n_kv_heads;
  s.head_dim = p->head_dim;
  s.prompt_len = prompt_len;
  s.n_query = prompt_len;
  s.keep_window = p->n_recent;
  s.pool_kernel = 1;
  s.pool_avg = 0;
  s.budget = p->n_heavy + p->n_recent;
  s.cap = p->n_heavy + p->n_recent + 1;
  kvc_status r = run_snapkv(&s, q, k, v, st->k, st->v, st->pos, st->n_used, nullptr, st->score,
                            workspace, workspace_bytes, stream, votes);
  if (r != KVC_OK) return r;
  Ctx c;
  r = get_ctx(stream, &c);
  if (r != KVC_OK) return r;
  const long long units = (long long)p->n_layers * p->batch * p->n_kv_heads;
  return cuda_status(
      launch_h2o_init_state(c, st->pos, st->n_used, st->free_slot, st->n_used, (int)units, s.cap));
}

// Step 2 of SnapKV (or H2O's column sums with n_query = L) from the rows' log-sum-exp.
kvc_status votes_from_lse_call(const kvc_snapkv_params *p, const void *q_win, const void *k,
                               const float *lse, float *votes_out, kvc_stream_t stream) {
  ensure_encode();
  Ctx c;
  kvc_status st = get_ctx(stream, &c);
  if (st != KVC_OK) return st;
  if (!p) return KVC_ERR_NULL;
  if (!common_heads_ok(p->n_layers, p->batch, p->n_q_heads, p->n_kv_heads, p->head_dim) ||
      p->prompt_len < 1 || p->n_query < 1 || p->n_query > p->prompt_len)
    return KVC_ERR_SHAPE;
  const long long units = (long long)p->n_layers * p->batch * p->n_kv_heads;
  const int G = p->n_q_heads / p->n_kv_heads;
  if ((long long)G * p->n_query > kMaxRows || units * G * p->n_query > kMaxRows ||
      units * G * p->prompt_len > kMaxRows)
    return KVC_ERR_SHAPE;
  if (!q_win || !k || !lse || !votes_out) return KVC_ERR_NULL;
  if (!aligned16(q_win) || !aligned16(k) || !aligned4(lse) || !aligned4(votes_out))
    return KVC_ERR_ALIGN;
  if (!g_encode) return KVC_ERR_CUDA;
  WindowVoteLseArgs a;
  a.q = q_win;
  a.k = k;
  a.lse = lse;
  a.units = (int)units;
  a.L = p->prompt_len;
  a.G = G;
  a.Wq = p->n_query;
  a.D = p->head_dim;
  a.votes = votes_out;
  return cuda_status(launch_window_vote_lse(c, a));
}

}  // namespace kvc

extern "C" {

const char *kvc_status_string(kvc_status s) {
  switch (s) {
    case KVC_OK: return "KVC_OK";
    case KVC_ERR_NULL: return "KVC_ERR_NULL: a required pointer is NULL";
    case KVC_ERR_SHAPE: return "KVC_ERR_SHAPE: a size is out of range or inconsistent";
    case KVC_ERR_ALIGN: return "KVC_ERR_ALIGN: a tensor base is not aligned";
    case KVC_ERR_BUDGET: return "KVC_ERR_BUDGET: budget or capacity inconsistent";
    case KVC_ERR_CUDA: return "KVC_ERR_CUDA: a CUDA call or kernel launch failed";
    case KVC_ERR_TIMEOUT: return "KVC_ERR_TIMEOUT: a device-side bounded wait ran out";
    case KVC_ERR_WORKSPACE: return "KVC_ERR_WORKSPACE: workspace missing or too small";
    case KVC_ERR_UNSUPPORTED: return "KVC_ERR_UNSUPPORTED: needs an sm_103 (GB300) device";
  }
  return "unknown kvc_status";
}

int kvc_version(void) { return 100; }

void kvc_set_wait_timeout_ns(uint64_t ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timeout_ns = ns > 0 ? ns : 1;
}

kvc_status kvc_device_status(uint32_t *flags_out, int clear, kvc_stream_t stream) {
  const TraceRange trace_range("kvc_device_status");
  Ctx c;
  kvc_status st = get_ctx(stream, &c);
  if (st != KVC_OK) return st;
  if (!flags_out) return KVC_ERR_NULL;
  if (cudaStreamSynchronize(c.stream) != cudaSuccess) return KVC_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, c.status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return KVC_ERR_CUDA;
  if (clear && cudaMemset(c.status, 0, sizeof(uint32_t)) != cudaSuccess) return KVC_ERR_CUDA;
  *flags_out = v;
  return (v & KVC_DEV_TIMEOUT) ? KVC_ERR_TIMEOUT : KVC_OK;
}

kvc_status kvc_selftest_wait_timeout(uint32_t timeout_us, kvc_stream_t stream) {
  const TraceRange trace_range("kvc_selftest_wait_timeout");
  Ctx c;
  kvc_status st = get_ctx(stream, &c);
  if (st != KVC_OK) return st;
  if (cudaStreamSynchronize(c.stream) != cudaSuccess) return KVC_ERR_CUDA;
  if (cudaMemset(c.status, 0, sizeof(uint32_t)) != cudaSuccess) return KVC_ERR_CUDA;
  c.timeout_ns = (unsigned long long)timeout_us * 1000ull;
  int result = 0;
  if (run_selftest_wait(c, &result) != cudaSuccess) return KVC_ERR_CUDA;
  uint32_t flags = 0;
  if (cudaMemcpy(&flags, c.status, sizeof(flags), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KVC_ERR_CUDA;
  return (result == 3 && (flags & KVC_DEV_TIMEOUT)) ? KVC_ERR_TIMEOUT : KVC_OK;
}

size_t snapkv_workspace_bytes(const kvc_snapkv_params *p) {
  SnapPlan s;
  if (plan_snapkv(p, true, sms_for_sizing(), &s) != KVC_OK) return 256;
  return s.total > 0 ? s.total : 256;
}

kvc_status snapkv_vote_plan(const kvc_snapkv_params *p, int32_t num_sms, int64_t *out) {
  if (!p || !out) return KVC_ERR_NULL;
  const int sms = num_sms > 0 ? num_sms : sms_for_sizing();
  SnapPlan s;
  const kvc_status st = plan_snapkv(p, true, sms, &s);
  if (st != KVC_OK) return st;
  const WindowVotePlan pl = plan_window_vote((int)s.units, p->prompt_len, s.R, p->n_query, sms);
  out[0] = pl.single;
  out[1] = pl.g;
  out[2] = pl.ngroups;
  out[3] = pl.row_tiles;
  out[4] = pl.qr;
  out[5] = (int64_t)pl.ws_bytes;
  return KVC_OK;
}

kvc_status snapkv_compress(const kvc_snapkv_params *p, const void *q_win, const void *k,
                           const void *v, void *k_out, void *v_out, int32_t *pos_out,
                           int32_t *n_valid_out, float *votes_out, float *kept_scores_out,
                           void *workspace, size_t workspace_bytes, kvc_stream_t stream) {
  const TraceRange trace_range("snapkv_compress");
  ensure_encode();
  return run_snapkv(p, q_win, k, v, k_out, v_out, pos_out, n_valid_out, votes_out,
                    kept_scores_out, workspace, workspace_bytes, stream);
}

kvc_status snapkv_select(const kvc_snapkv_params *p, const float *votes, const void *k,
                         const void *v, void *k_out, void *v_out, int32_t *pos_out,
                         int32_t *n_valid_out, float *kept_scores_out, void *workspace,
                         size_t workspace_bytes, kvc_stream_t stream) {
  const TraceRange trace_range("snapkv_select");
  ensure_encode();
  if (!votes) return KVC_ERR_NULL;
  return run_snapkv(p, nullptr, k, v, k_out, v_out, pos_out, n_valid_out, nullptr,
                    kept_scores_out, workspace, workspace_bytes, stream, votes);
}

kvc_status snapkv_prefill_attention(const kvc_snapkv_params *p, const void *q, const void *k,
                                    const void *v, void *o_out, float *votes_out,
                                    kvc_stream_t stream) {
  const TraceRange trace_range("snapkv_prefill_attention");
  return kvc::prefill_call(p, q, k, v, o_out, votes_out, nullptr, stream);
}

kvc_status prefill_attention_lse(const kvc_snapkv_params *p, const void *q, const void *k,
                                 const void *v, void *o_out, float *lse_out, kvc_stream_t stream) {
  const TraceRange trace_range("prefill_attention_lse");
  if (!lse_out) return KVC_ERR_NULL;
  return kvc::prefill_call(p, q, k, v, o_out, nullptr, lse_out, stream);
}

kvc_status snapkv_votes_from_lse(const kvc_snapkv_params *p, const void *q_win, const void *k,
                                 const float *lse, float *votes_out, kvc_stream_t stream) {
  const TraceRange trace_range("snapkv_votes_from_lse");
  return kvc::votes_from_lse_call(p, q_win, k, lse, votes_out, stream);
}

size_t compressed_decode_attn_workspace_bytes(const kvc_decode_params *p) {
  if (!p || !common_heads_ok(p->n_layers, p->batch, p->n_q_heads, p->n_kv_heads, p->head_dim) ||
      p->cap < 1)
    return 256;
  const long long units = (long long)p->n_layers * p->batch * p->n_kv_heads;
  return decode_ws_bytes((int)units, p->n_q_heads / p->n_kv_heads, p->head_dim, p->cap,
                         sms_for_sizing());
}

kvc_status compressed_decode_attn(const kvc_decode_params *p, const void *q, const void *k_new,
                                  const void *v_new, void *k_cache, void *v_cache, int32_t *pos,
                                  int32_t *n_valid, void *out, void *workspace,
                                  size_t workspace_bytes, kvc_stream_t stream) {
  const TraceRange trace_range("compressed_decode_attn");
  return kvc::decode_call(p, q, k_new, v_new, k_cache, v_cache, pos, n_valid, out, workspace,
                          workspace_bytes, stream, false);
}

size_t h2o_step_scratch_bytes(const kvc_h2o_params *p) {
  if (!p || !common_heads_ok(p->n_layers, p->batch, p->n_q_heads, p->n_kv_heads, p->head_dim) ||
      p->n_heavy < 0 || p->n_recent < 1)
    return 256;
  const long long slots = (long long)p->n_heavy + p->n_recent + 1;
  if (slots > (1 << 20)) return 256;
  const long long units = (long long)p->n_layers * p->batch * p->n_kv_heads;
  return plan_h2o_split(units, p->n_q_heads / p->n_kv_heads, p->head_dim, (int)slots,
                        sms_for_sizing())
      .scratch_bytes;
}

int32_t h2o_step_ctas_per_unit(const kvc_h2o_params *p) {
  if (!p || !common_heads_ok(p->n_layers, p->batch, p->n_q_heads, p->n_kv_heads, p->head_dim) ||
      p->n_heavy < 0 || p->n_recent < 1 || p->n_q_heads / p->n_kv_heads > 8)
    return 0;
  const long long slots = (long long)p->n_heavy + p->n_recent + 1;
  if (slots > (1 << 20)) return 0;
  const long long units = (long long)p->n_layers * p->batch * p->n_kv_heads;
  const int G = p->n_q_heads / p->n_kv_heads;
  const H2OSplitPlan sp = plan_h2o_split(units, G, p->head_dim, (int)slots, sms_for_sizing());
  const bool fits1 = h2o_single_fits(G, p->head_dim, slots);
  if (sp.feasible && (sp.nsplit > 1 || !fits1)) return sp.nsplit;
  return fits1 ? 1 : 0;
}

size_t h2o_prefill_workspace_bytes(const kvc_h2o_params *p, int32_t prompt_len) {
  if (!p) return 256;
  kvc_snapkv_params s;
  s.n_layers = p->n_layers;
  s.batch = p->batch;
  s.n_q_heads = p->n_q_heads;
  s.n_kv_heads = p->n_kv_heads;
  s.head_dim = p->head_dim;
  s.prompt_len = prompt_len;
  s.n_query = prompt_len;
  s.keep_window = p->n_recent;
  s.pool_kernel = 1;
  s.pool_avg = 0;
  s.budget = p->n_heavy + p->n_recent;
  s.cap = p->n_heavy + p->n_recent + 1;
  return snapkv_workspace_bytes(&s);
}

kvc_status h2o_prefill(const kvc_h2o_params *p, int32_t prompt_len, const void *q, const void *k,
                       const void *v, const kvc_h2o_state *st, void *workspace,
                       size_t workspace_bytes, kvc_stream_t stream) {
  const TraceRange trace_range("h2o_prefill");
  if (!q) return KVC_ERR_NULL;
  return kvc::h2o_prefill_call(p, prompt_len, q, nullptr, k, v, st, workspace, workspace_bytes,
                               stream);
}

kvc_status h2o_prefill_from_votes(const kvc_h2o_params *p, int32_t prompt_len,
                                  const float *votes, const void *k, const void *v,
                                  const kvc_h2o_state *st, void *workspace,
                                  size_t workspace_bytes, kvc_stream_t stream) {
  const TraceRange trace_range("h2o_prefill_from_votes");
  if (!votes) return KVC_ERR_NULL;
  return kvc::h2o_prefill_call(p, prompt_len, nullptr, votes, k, v, st, workspace,
                               workspace_bytes, stream);
}

kvc_status h2o_decode_step(const kvc_h2o_params *p, const void *q, const void *k_new,
                           const void *v_new, const kvc_h2o_state *st, int32_t t, void *out,
                           int32_t *evicted_pos_out, kvc_stream_t stream) {
  const TraceRange trace_range("h2o_decode_step");
  Ctx c;
  kvc_status r = get_ctx(stream, &c);
  if (r != KVC_OK) return r;
  if (!p || !st) return KVC_ERR_NULL;
  if (!common_heads_ok(p->n_layers, p->batch, p->n_q_heads, p->n_kv_heads, p->head_dim) ||
      p->n_heavy < 0 || p->n_recent < 1 || t < 0)
    return KVC_ERR_SHAPE;
  const int G = p->n_q_heads / p->n_kv_heads;
  if (G > 8) return KVC_ERR_SHAPE;  // query heads per KV head: 1..8
  const long long slots = (long long)p->n_heavy + p->n_recent + 1;
  const long long units = (long long)p->n_layers * p->batch * p->n_kv_heads;
  if (slots > (1 << 20) || units * slots > kMaxRows || units > (1ll << 31) - 1)
    return KVC_ERR_SHAPE;
  // one CTA per unit, or the unit's cache split over several CTAs
  const H2OSplitPlan sp = plan_h2o_split(units, G, p->head_dim, (int)slots, c.num_sms);
  const bool fits1 = h2o_single_fits(G, p->head_dim, slots);
  const bool have_scratch = st->scratch && st->scratch_bytes >= sp.scratch_bytes;
  const bool split = sp.feasible && have_scratch && (sp.nsplit > 1 || !fits1);
  if (!split && !fits1) return sp.feasible ? KVC_ERR_WORKSPACE : KVC_ERR_SHAPE;
  if (split && (reinterpret_cast<uintptr_t>(st->scratch) & 255u) != 0) return KVC_ERR_ALIGN;
  if (!q || !k_new || !v_new || !out || !st->k || !st->v || !st->score || !st->pos ||
      !st->n_used || !st->free_slot)
    return KVC_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out) ||
      !aligned16(st->k) || !aligned16(st->v) || !aligned4(st->score) || !aligned4(st->pos) ||
      !aligned4(st->n_used) || !aligned4(st->free_slot) ||
      (evicted_pos_out && !aligned4(evicted_pos_out)))
    return KVC_ERR_ALIGN;
  H2OArgs a;
  a.q = q;
  a.k_new = k_new;
  a.v_new = v_new;
  a.k = st->k;
  a.v = st->v;
  a.score = st->score;
  a.pos = st->pos;
  a.n_used = st->n_used;
  a.free_slot = st->free_slot;
  a.out = out;
  a.evicted = evicted_pos_out;
  a.units = (int)units;
  a.G = G;
  a.D = p->head_dim;
  a.slots = (int)slots;
  a.n_recent = p->n_recent;
  a.t = t;
  a.split = split ? 1 : 0;
  a.scratch = st->scratch;
  return cuda_status(launch_h2o_step(c, a));
}

kvc_status sink_window_append(const kvc_sink_params *p, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, int32_t *pos, int64_t t,
                              kvc_stream_t stream) {
  const TraceRange trace_range("sink_window_append");
  Ctx c;
  kvc_status r = get_ctx(stream, &c);
  if (r != KVC_OK) return r;
  if (!p) return KVC_ERR_NULL;
  if (p->n_layers < 1 || p->batch < 1 || p->n_kv_heads < 1 ||
      (p->head_dim != 64 && p->head_dim != 128) || p->n_sink < 0 || p->n_recent < 1 || t < 0 ||
      t > 2147483647ll)
    return KVC_ERR_SHAPE;
  const long long units = (long long)p->n_layers * p->batch * p->n_kv_heads;
  const long long rows = (long long)p->n_sink + p->n_recent;
  if (units * rows > kMaxRows || units > (1ll << 31) - 1) return KVC_ERR_SHAPE;
  if (!k_new || !v_new || !k_cache || !v_cache) return KVC_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (pos && !aligned4(pos)))
    return KVC_ERR_ALIGN;
  const long long slot = t < p->n_sink ? t : p->n_sink + (t - p->n_sink) % p->n_recent;
  return cuda_status(launch_sink_append(c, k_new, v_new, k_cache, v_cache, pos, (int)units,
                                        p->head_dim, (int)rows, (int)slot, t));
}

}  // extern "C"
