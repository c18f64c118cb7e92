/*
 * kvcompress.h -- C ABI of the GB300 (sm_103a) attention-score KV-cache compression
 * library (libkvcompress.so): SnapKV prompt compression, decode attention over the
 * compact cache, H2O heavy-hitter eviction and the StreamingLLM sink + ring cache.
 *
 * Sources of the operations (abeam.tech article summaries):
 *   [SnapKV]       "SnapKV: LLM Knows What You are Looking for Before Generation"
 *                  (2026-07-18), sections 処理の流れ (processing flow) steps 1-4 and
 *                  推論方法 (inference).
 *   [H2O]          "H2O: Heavy-Hitter Oracle for Efficient Generative Inference of
 *                  Large Language Models" (2026-06-24), sections 何を残すのか
 *                  (what is kept) and 処理の流れ (processing flow).
 *   [StreamingLLM] "Efficient Streaming Language Models with Attention Sinks"
 *                  (2026-07-02), sections キャッシュ構造 (cache structure) and
 *                  推論の流れ (inference flow).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Plain C: pointers, integers and a CUDA stream handle (kvc_stream_t is a
 *   cudaStream_t; NULL is the legacy default stream).  No library allocates, frees
 *   or synchronises device memory: the caller owns every buffer and the stream.  The
 *   only calls that synchronise are kvc_device_status() and the self-test.
 * - Device pointers ("dev") must point to memory of the current CUDA device.  Tensors
 *   are dense, row-major, 16-byte aligned at their base, bf16 ("bf16") unless stated.
 *   Shapes use: Ly layers, B batch, Hq query heads, Hkv KV heads (Hq % Hkv == 0,
 *   G = Hq / Hkv query heads share KV head h = q_head / G), D head dim (64 or 128),
 *   U = Ly * B * Hkv independent (layer, batch, KV-head) units.
 * - Attention everywhere is softmax(q . k / sqrt(D)) . v with fp32 accumulation; a
 *   bf16 output is rounded once at the end.
 * - Every argument check runs on the host before anything is launched; on an error
 *   nothing is launched and the error code is returned.  A failed launch returns
 *   KVC_ERR_CUDA.  Conditions only the device can see (a wait that ran out, a full
 *   cache) set bits of a per-device status word read with kvc_device_status().
 * - Calls are asynchronous on `stream`.  Two calls that share a workspace, a cache or
 *   a state must be ordered (same stream, or events).
 * - The library needs an sm_103 GPU (GB300); elsewhere every call returns
 *   KVC_ERR_UNSUPPORTED.
 */
#ifndef KVCOMPRESS_H
#define KVCOMPRESS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void *kvc_stream_t;

typedef enum {
  KVC_OK = 0,
  KVC_ERR_NULL = 1,        /* a required pointer is NULL */
  KVC_ERR_SHAPE = 2,       /* a size is out of range or inconsistent */
  KVC_ERR_ALIGN = 3,       /* a tensor base is not 16-byte aligned */
  KVC_ERR_BUDGET = 4,      /* budget / capacity inconsistent (e.g. budget < kept window) */
  KVC_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  KVC_ERR_TIMEOUT = 6,     /* a device-side bounded wait ran out (see kvc_device_status) */
  KVC_ERR_WORKSPACE = 7,   /* workspace missing or smaller than the *_workspace_bytes() size */
  KVC_ERR_UNSUPPORTED = 8  /* no sm_103 device current */
} kvc_status;

/* Device status bits (kvc_device_status). */
#define KVC_DEV_TIMEOUT    0x1u  /* a bounded wait (mbarrier, peer flag) gave up */
#define KVC_DEV_CACHE_FULL 0x2u  /* an append found its cache full; the token was dropped */
#define KVC_DEV_BAD_STATE  0x4u  /* an H2O/decode state was inconsistent (e.g. slot out of range) */

/* Limits of the decode-time entry points (compressed_decode_attn, its _noalloc variant
 * and h2o_decode_step): G = Hq / Hkv query heads per KV head in 1..8; at most
 * KVC_DECODE_MAX_UNITS units (Ly * B * Hkv) per compressed_decode_attn call (one split-K
 * counter per unit in the workspace's fixed header). */
#define KVC_DECODE_MAX_UNITS 131072

/* Human-readable name of a status code (static string, never NULL). */
const char *kvc_status_string(kvc_status s);

/* ABI version of this header (major * 10000 + minor * 100 + patch). */
int kvc_version(void);

/* Waits for `stream`, then copies the current device's status bits to *flags_out
 * (KVC_DEV_* above); with clear != 0 the word is reset to 0 afterwards.  Returns
 * KVC_ERR_TIMEOUT if KVC_DEV_TIMEOUT is set, else KVC_OK (or KVC_ERR_CUDA). */
kvc_status kvc_device_status(uint32_t *flags_out, int clear, kvc_stream_t stream);

/* Limit, in nanoseconds, of every device-side wait in kernels launched after this
 * call by this process (default 1e9 = 1 s).  A wait that runs out sets
 * KVC_DEV_TIMEOUT, abandons the rest of its work and returns. */
void kvc_set_wait_timeout_ns(uint64_t ns);

/* Self-test of the bounded waits: launches one kernel that waits on an mbarrier and on
 * a global flag that nothing ever completes, each with a limit of `timeout_us`
 * microseconds, synchronises, and returns KVC_ERR_TIMEOUT if (as expected) both waits
 * gave up and set KVC_DEV_TIMEOUT, KVC_OK otherwise.  The status word is left set. */
kvc_status kvc_selftest_wait_timeout(uint32_t timeout_us, kvc_stream_t stream);

/* ------------------------------------------------------------------------------ */
/* SnapKV prompt compression ([SnapKV] 処理の流れ steps 1-4; 推論方法: once, right   */
/* after the prompt is processed).                                                  */
/* ------------------------------------------------------------------------------ */
typedef struct {
  int32_t n_layers;    /* Ly >= 1 (all tensors carry this leading dimension) */
  int32_t batch;       /* B >= 1 */
  int32_t n_q_heads;   /* Hq >= 1 */
  int32_t n_kv_heads;  /* Hkv >= 1, Hq % Hkv == 0 */
  int32_t head_dim;    /* D: 64 or 128 */
  int32_t prompt_len;  /* L >= 1 */
  int32_t n_query;     /* Wq, 1 <= Wq <= L: trailing prompt queries that vote.  SnapKV:
                          the observation window W.  H2O prefill: Wq = L. */
  int32_t keep_window; /* W_keep >= 0: trailing prompt positions always kept (SnapKV: W) */
  int32_t pool_kernel; /* odd P >= 1: 1D pooling kernel over the vote (1 = no pooling) */
  int32_t budget;      /* Kb: kept entries including the window; W_keep <= Kb */
  int32_t cap;         /* rows per unit of the output cache; cap >= min(Kb, L),
                          cap <= 2097120 (65535 * 32) */
  int32_t pool_avg;    /* 0: max-pool (the SnapKV default); 1: average pool, the window's sum
                          divided by P with zeros beyond both ends of the candidates */
} kvc_snapkv_params;

/* Bytes of device workspace snapkv_compress needs for *p (0 is never returned). */
size_t snapkv_workspace_bytes(const kvc_snapkv_params *p);

/* The plan of the window votes (SnapKV article, 処理の流れ steps 1-2) that snapkv_compress
 * uses for *p on a GPU with num_sms SMs (num_sms <= 0: the current device's count, or 160
 * without one).  Host-only: no device is needed and nothing is launched; for diagnostics
 * and for callers that check which kernel runs.  On KVC_OK, out (host, 6 entries) holds:
 *   out[0] 1 for the single-pass kernel (each CTA's scores held in tensor memory until the
 *          rows' statistics are known), 0 for the two-pass kernel;
 *   out[1] CTAs per job (the group size g; a job is a unit's tile of query rows);
 *   out[2] groups (num_sms / g; CTAs past the last whole group stay idle);
 *   out[3] row tiles per unit; out[4] query rows per tile;
 *   out[5] bytes of the groups' statistics-exchange records within the workspace.
 * The votes are formed unless the call keeps every position and asks for no votes.
 * Returns KVC_ERR_NULL, KVC_ERR_SHAPE or KVC_ERR_BUDGET where snapkv_compress would reject
 * *p with that code (out untouched), else KVC_OK. */
kvc_status snapkv_vote_plan(const kvc_snapkv_params *p, int32_t num_sms, int64_t *out);

/* For every unit (layer, batch b, KV head h):
 *   1. window scores: each of the Wq trailing queries of the G query heads of h, at
 *      position i = L - Wq + r, takes softmax over the keys 0..i (prefix keys always,
 *      window keys causally) with scale 1/sqrt(D);
 *   2. vote v_j = sum of those probabilities over the G*Wq rows (fp32);
 *   3. u = 1D max-pool of v over the candidates 0..L-W_keep-1 (kernel P, stride 1,
 *      windows cut at both ends), or with pool_avg the window average
 *      u_j = (1/P) sum_{|t-j| <= (P-1)/2, 0 <= t < L-W_keep} v_t;
 *   4. the k = Kb - W_keep candidates with the largest u (equal u: lower position
 *      first), in ascending position order, followed by the W_keep trailing positions;
 *      their K/V rows are gathered into rows 0..n-1 of the unit's compact cache.
 *   If Kb >= L or W_keep >= L, every position is kept (n = L) and steps 1-3 are skipped
 *   unless kept_scores_out is given.
 * Inputs (bf16): q_win [Ly,B,Hq,Wq,D] and k [Ly,B,Hkv,L,D] in device memory; v
 *   [Ly,B,Hkv,L,D] in device memory or in page-locked host memory mapped for the device
 *   (cudaHostAlloc, cudaHostRegister): v is read only at the kept rows, so a prompt's V
 *   can stay on the host and only the kept rows cross the host link.  Other host memory
 *   returns KVC_ERR_UNSUPPORTED.
 * Outputs (dev): k_out, v_out bf16 [Ly,B,Hkv,cap,D] (rows >= n untouched);
 *   pos_out int32 [Ly,B,Hkv,cap] (kept prompt positions in rows 0..n-1, -1 in rows
 *   n..cap-1); n_valid_out int32 [U] (= n);
 *   votes_out fp32 [Ly,B,Hkv,L] or NULL (the raw vote v, every position);
 *   kept_scores_out fp32 [Ly,B,Hkv,cap] or NULL (vote of each kept row, 0 beyond n;
 *   this is H2O's initial cumulative score when Wq = L).
 * workspace: dev, >= snapkv_workspace_bytes(p) bytes, 256-byte aligned; contents need
 *   no initialisation and are scratch after the call.
 * Errors: KVC_ERR_NULL, KVC_ERR_SHAPE, KVC_ERR_ALIGN, KVC_ERR_BUDGET, KVC_ERR_WORKSPACE,
 *   KVC_ERR_CUDA, KVC_ERR_UNSUPPORTED. */
kvc_status snapkv_compress(const kvc_snapkv_params *p, const void *q_win, const void *k,
                           const void *v, void *k_out, void *v_out, int32_t *pos_out,
                           int32_t *n_valid_out, float *votes_out, float *kept_scores_out,
                           void *workspace, size_t workspace_bytes, kvc_stream_t stream);

/* Steps 3-4 of snapkv_compress from votes computed elsewhere (snapkv_prefill_attention):
 * pooling, top-k and the gather exactly as snapkv_compress does them, without its window
 * vote.  votes: dev fp32 [Ly,B,Hkv,L] (read only).  The other arguments, the workspace
 * (snapkv_workspace_bytes(p) bytes suffice) and the errors are those of snapkv_compress;
 * p->n_query is not used. */
kvc_status snapkv_select(const kvc_snapkv_params *p, const float *votes, const void *k,
                         const void *v, void *k_out, void *v_out, int32_t *pos_out,
                         int32_t *n_valid_out, float *kept_scores_out, void *workspace,
                         size_t workspace_bytes, kvc_stream_t stream);

/* The prompt's self-attention with the SnapKV votes as a by-product (SnapKV article,
 * 推論方法: the compression follows the prompt's processing).  For every (layer, batch,
 * query head h): o = softmax(q . k^T / sqrt(D)) . v over the prompt with the causal mask
 * (row i sees positions 0..i; KV head h / G).  With votes_out, the last n_query rows of
 * every query head also add their probabilities per key into votes_out of their KV head:
 * the same votes as snapkv_compress's step 2 (fp32; summed over the G heads with atomic
 * adds, so the order of the additions, and the last bits, can vary between calls).
 * The query tiles that hold window rows are swept twice (row statistics, then output and
 * votes); every other tile once.
 * Uses n_layers, batch, n_q_heads, n_kv_heads, head_dim, prompt_len and n_query of p.
 * Inputs (dev, bf16): q [Ly,B,Hq,L,D], k, v [Ly,B,Hkv,L,D].  Outputs (dev): o_out bf16
 * [Ly,B,Hq,L,D]; votes_out fp32 [Ly,B,Hkv,L] or NULL (then n_query is not used).
 * Needs no workspace.  Errors: KVC_ERR_NULL, KVC_ERR_SHAPE, KVC_ERR_ALIGN, KVC_ERR_CUDA,
 * KVC_ERR_UNSUPPORTED. */
kvc_status snapkv_prefill_attention(const kvc_snapkv_params *p, const void *q, const void *k,
                                    const void *v, void *o_out, float *votes_out,
                                    kvc_stream_t stream);

/* The prompt's causal self-attention (as snapkv_prefill_attention without votes) that also
 * writes each row's log-sum-exp: lse_out[.., i] = ln sum_{j <= i} exp(q_i . k_j / sqrt(D)),
 * the normaliser of the row's softmax (SnapKV article, 処理の流れ step 1, and the H2O
 * article, 処理の流れ: both scores are rows of this softmax).  With it,
 * snapkv_votes_from_lse forms the SnapKV votes, or H2O's initial scores, in one pass over
 * the keys.  Uses n_layers, batch, n_q_heads, n_kv_heads, head_dim and prompt_len of p.
 * Inputs (dev, bf16): q [Ly,B,Hq,L,D], k, v [Ly,B,Hkv,L,D].  Outputs (dev): o_out bf16
 * [Ly,B,Hq,L,D]; lse_out fp32 [Ly,B,Hq,L] (natural logarithm; must not be NULL).
 * Needs no workspace.  Errors: as snapkv_prefill_attention. */
kvc_status prefill_attention_lse(const kvc_snapkv_params *p, const void *q, const void *k,
                                 const void *v, void *o_out, float *lse_out,
                                 kvc_stream_t stream);

/* Step 2 of snapkv_compress (the vote) when every voting row's softmax normaliser is
 * known (prefill_attention_lse): v_j = sum over the G * Wq voting rows i that see key j
 * of exp(q_i . k_j / sqrt(D) - lse_i), fp32, every position j of every unit.  These are
 * snapkv_compress's votes_out up to fp32 rounding when lse is the rows' own log-sum-exp;
 * feed them to snapkv_select (SnapKV) or h2o_prefill_from_votes (n_query = L: H2O's
 * initial cumulative scores).  One pass over the keys, no statistics pass.
 * Uses n_layers, batch, n_q_heads, n_kv_heads, head_dim, prompt_len and n_query of p.
 * Inputs (dev): q_win bf16 [Ly,B,Hq,Wq,D] (the trailing Wq queries of every head);
 * k bf16 [Ly,B,Hkv,L,D]; lse fp32 [Ly,B,Hq,L] (only positions L-Wq..L-1 are read; a
 * non-finite entry makes its row add nothing).  Output: votes_out fp32 [Ly,B,Hkv,L].
 * When G * Wq > 128 several row tiles add into a key's vote with atomic adds, so the
 * order of the additions, and the last bits, can vary between calls.
 * Needs no workspace.  Errors: KVC_ERR_NULL, KVC_ERR_SHAPE, KVC_ERR_ALIGN, KVC_ERR_CUDA,
 * KVC_ERR_UNSUPPORTED. */
kvc_status snapkv_votes_from_lse(const kvc_snapkv_params *p, const void *q_win, const void *k,
                                 const float *lse, float *votes_out, kvc_stream_t stream);

/* ------------------------------------------------------------------------------ */
/* Decode attention over a compact (SnapKV) or ring (StreamingLLM) cache           */
/* ([SnapKV] 推論方法: decoding reads only the compressed cache; [StreamingLLM]       */
/* 推論の流れ: attention reads only sink and recent tokens).                          */
/* ------------------------------------------------------------------------------ */
typedef struct {
  int32_t n_layers, batch, n_q_heads, n_kv_heads, head_dim; /* as above */
  int32_t cap;        /* rows per unit in k_cache / v_cache */
  int32_t n_uniform;  /* n_valid == NULL: entries attended in every unit.  n_valid given:
                         0, or an upper bound on every unit's row count after the append
                         that the work is planned for (rows beyond it are not attended and
                         raise KVC_DEV_BAD_STATE); 0 plans for the full capacity */
  int32_t new_pos;    /* position recorded in pos[] for an appended token */
} kvc_decode_params;

/* Bytes of workspace compressed_decode_attn needs (split-K partials and counters). */
size_t compressed_decode_attn_workspace_bytes(const kvc_decode_params *p);

/* One decode step.  If k_new and v_new are given (dev bf16 [Ly,B,Hkv,D]), each unit
 * first appends them at row n_valid[u] (which must then be non-NULL), records
 * p->new_pos in pos[u][row] (if pos != NULL) and increments n_valid[u]; a full unit
 * (n_valid == cap) drops the token and sets KVC_DEV_CACHE_FULL.  Then for each query
 * head of each unit: out = softmax(q . K_c^T / sqrt(D)) . V_c over the unit's first n
 * rows (n = n_valid[u], or p->n_uniform when n_valid == NULL); n = 0 gives zeros.
 * q and out: dev bf16 [Ly,B,Hq,D].  k_cache, v_cache: dev bf16 [Ly,B,Hkv,cap,D].
 * pos: dev int32 [Ly,B,Hkv,cap] or NULL.  n_valid: dev int32 [U] or NULL.
 * workspace: dev, >= compressed_decode_attn_workspace_bytes(p) bytes; it must be
 *   zero-filled before its first use with this function; every call that returns
 *   normally leaves its counters at zero again (after KVC_DEV_TIMEOUT, zero it again).
 * Limits: G in 1..8 and U <= KVC_DECODE_MAX_UNITS, else KVC_ERR_SHAPE.
 * Errors: as snapkv_compress. */
kvc_status compressed_decode_attn(const kvc_decode_params *p, const void *q, const void *k_new,
                                  const void *v_new, void *k_cache, void *v_cache, int32_t *pos,
                                  int32_t *n_valid, void *out, void *workspace,
                                  size_t workspace_bytes, kvc_stream_t stream);

/* The same decode step for callers that cannot give the library a device workspace:
 * no counterpart in the articles; it exists for serving engines that own all device
 * memory through their own pool and pass only the step's tensors to the attention call
 * (they have no allocator to hand over, and a cudaMalloc mid-step would synchronise
 * the device).  The split-K scratch lives in a fixed 8 MiB device array inside the
 * library (held on every GPU that loads it until the process exits); nothing is
 * allocated.  Arguments and results are those of compressed_decode_attn without the
 * workspace.  A call needing more scratch than 8 MiB (see
 * compressed_decode_attn_workspace_bytes) returns KVC_ERR_WORKSPACE and launches
 * nothing.  The first call on a device looks up the array's device address (with that
 * device current) and should come before any stream capture.  Each call clears the
 * counters it uses; calls that overlap on the GPU share the array and race. */
kvc_status compressed_decode_attn_noalloc(const kvc_decode_params *p, const void *q,
                                          const void *k_new, const void *v_new, void *k_cache,
                                          void *v_cache, int32_t *pos, int32_t *n_valid,
                                          void *out, kvc_stream_t stream);

/* ------------------------------------------------------------------------------ */
/* H2O heavy-hitter + recent-window cache ([H2O] 何を残すのか, 処理の流れ).          */
/* ------------------------------------------------------------------------------ */
typedef struct {
  int32_t n_layers, batch, n_q_heads, n_kv_heads, head_dim; /* as above */
  int32_t n_heavy;   /* heavy hitters kept (>= 0) */
  int32_t n_recent;  /* most recent positions never evicted (>= 1) */
} kvc_h2o_params;   /* slots per unit S_h = n_heavy + n_recent + 1 */

typedef struct {      /* all dev pointers, owned by the caller */
  void *k;            /* bf16 [U, S_h, D] */
  void *v;            /* bf16 [U, S_h, D] */
  float *score;       /* fp32 [U, S_h] cumulative attention score */
  int32_t *pos;       /* int32 [U, S_h] token position, -1 = never used */
  int32_t *n_used;    /* int32 [U] live entries after the last step (<= S_h - 1) */
  int32_t *free_slot; /* int32 [U] slot the next token is written to */
  void *scratch;      /* dev scratch of the split step, h2o_step_scratch_bytes() bytes,
                         zero-filled before its first use (every step that returns
                         normally leaves it reusable); may be NULL (see h2o_decode_step) */
  size_t scratch_bytes;
} kvc_h2o_state;

/* Bytes of state scratch h2o_decode_step needs to split each unit's cache over several
 * CTAs (few units, or more slots than one CTA's shared memory holds). */
size_t h2o_step_scratch_bytes(const kvc_h2o_params *p);

/* CTAs that h2o_decode_step gives each unit on the current device when the state has its
 * scratch: 1 for the one-CTA step, more for the split step; 0 if p is out of range.
 * Host-only (no launch); for callers that size grids or check which step runs. */
int32_t h2o_step_ctas_per_unit(const kvc_h2o_params *p);

/* Bytes of workspace h2o_prefill needs for a prompt of prompt_len tokens. */
size_t h2o_prefill_workspace_bytes(const kvc_h2o_params *p, int32_t prompt_len);

/* Initial cache from the prompt: the cumulative score of position j starts as the
 * causal column sum of the prompt's own attention (every prompt query, summed over
 * the G query heads); kept are the n_heavy largest scores among positions
 * < L - n_recent (equal scores: lower position) and the last n_recent positions, or
 * all L positions if L <= n_heavy + n_recent.  Writes every field of *st.
 * q: dev bf16 [Ly,B,Hq,L,D] (all prompt queries); k, v: dev bf16 [Ly,B,Hkv,L,D]. */
kvc_status h2o_prefill(const kvc_h2o_params *p, int32_t prompt_len, const void *q,
                       const void *k, const void *v, const kvc_h2o_state *st,
                       void *workspace, size_t workspace_bytes, kvc_stream_t stream);

/* h2o_prefill from column sums computed elsewhere: votes fp32 [Ly,B,Hkv,L] (dev, read
 * only) hold each position's initial cumulative score, e.g. snapkv_votes_from_lse with
 * n_query = prompt_len.  The cut, the gathered state and the errors are those of
 * h2o_prefill (h2o_prefill_workspace_bytes(p, prompt_len) bytes of workspace suffice). */
kvc_status h2o_prefill_from_votes(const kvc_h2o_params *p, int32_t prompt_len,
                                  const float *votes, const void *k, const void *v,
                                  const kvc_h2o_state *st, void *workspace,
                                  size_t workspace_bytes, kvc_stream_t stream);

/* One decode step of token position t for every unit: write (k_new, v_new) into
 * free_slot, attend over every live entry (the new one included) giving out, add each
 * entry's probability (summed over the G query heads) to its score; if the unit now
 * holds S_h entries, evict the smallest score among entries at positions
 * <= t - n_recent (equal scores: the higher position) and make its slot the free slot.
 * q, out: dev bf16 [Ly,B,Hq,D]; k_new, v_new: dev bf16 [Ly,B,Hkv,D];
 * evicted_pos_out: dev int32 [U] (evicted position or -1) or NULL.
 * Split step: with st->scratch of at least h2o_step_scratch_bytes(p) bytes, a call with
 * few units (less than eight CTAs per SM at one CTA per unit) splits each unit's cache
 * over several CTAs, and so does a cache whose logits do not fit one CTA's shared
 * memory (4 * (9 * G * D + G * S_h) bytes above 200 KB, i.e. S_h > 50048 at G = 1,
 * D = 128); the results are those of the one-CTA step up to fp32 rounding.  Without the
 * scratch such a cache returns KVC_ERR_WORKSPACE.  Limits: G in 1..8, S_h <= 2^20.
 * Errors: as snapkv_compress. */
kvc_status h2o_decode_step(const kvc_h2o_params *p, const void *q, const void *k_new,
                           const void *v_new, const kvc_h2o_state *st, int32_t t, void *out,
                           int32_t *evicted_pos_out, kvc_stream_t stream);

/* ------------------------------------------------------------------------------ */
/* StreamingLLM sink + recent ring ([StreamingLLM] キャッシュ構造, 推論の流れ).       */
/* ------------------------------------------------------------------------------ */
typedef struct {
  int32_t n_layers, batch, n_kv_heads, head_dim; /* as above */
  int32_t n_sink;    /* S >= 0 sink tokens, never evicted */
  int32_t n_recent;  /* R >= 1 ring slots for the most recent tokens */
} kvc_sink_params;  /* cache rows per unit = S + R */

/* Writes token t's key/value (dev bf16 [Ly,B,Hkv,D]) into row t (t < S) or
 * S + (t - S) mod R of every unit's cache (dev bf16 [Ly,B,Hkv,S+R,D]), evicting the
 * oldest recent token, and records t in pos (dev int32 [Ly,B,Hkv,S+R], or NULL).  The
 * step's attention is then compressed_decode_attn with cap = S + R,
 * n_valid = NULL and n_uniform = min(t + 1, S + R).  Errors: as snapkv_compress. */
kvc_status sink_window_append(const kvc_sink_params *p, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, int32_t *pos, int64_t t,
                              kvc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVCOMPRESS_H */
