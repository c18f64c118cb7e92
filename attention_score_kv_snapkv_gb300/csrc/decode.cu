// Decode attention over a compact (SnapKV) or sink + ring (StreamingLLM) cache: for
// each query head of each (layer, batch, KV head) unit, o = softmax(q . K_c^T / sqrt(D))
// . V_c over the unit's first n rows (SnapKV article, 推論方法: decoding reads only the
// compressed cache; StreamingLLM article, 推論の流れ: attention over sink and recent
// tokens only).  An optional append adds the step's new K/V row first (fused: the CTA
// whose tile holds the new row patches it in shared memory from k_new/v_new, and the
// unit's finishing CTA writes it to the cache, its position and the new n_valid).
//
// Design (sm_103a, HBM-bound: every cached K/V byte is read once):
// * persistent stream-K: all units' 128-row tile slots form one sequence that is split
//   evenly over one resident CTA per SM, so every CTA streams the same number of tiles;
//   a CTA's range covers segments of one or more units.  It works on its last unit
//   first (usually shared with the next CTA), then the others in order, so units split
//   between two CTAs are finished early by both and the tail of the kernel is a whole
//   unit without a merge.  Before waiting for the previous kernel (programmatic
//   dependent launch) the CTA prefetches its first tiles into L2.
// * warp 0 streams each segment's tiles as K0, V0, K1, V1, ... through a 4-stage
//   shared-memory ring with TMA (128-byte swizzle), so K tiles always use the even
//   stages and V tiles the odd ones.  The producer writes the tile index into a per-stage
//   tag before each load and the MMA issuer waits for its tag before it trusts the
//   stage's full-barrier parity.
// * the logits run on the tensor cores: warp 1 issues S^T = K_tile . q^T with
//   tcgen05.mma (M = 128 key rows, N = 16 columns holding the G query heads, K = D;
//   bf16 in, fp32 accumulator in TMEM, two buffers of 16 columns); the K stage and the
//   unit's q buffer are released by the MMA's own commits.  The compute warps write q
//   into rows 0..G-1 of a 16-row operand (double-buffered, 128-byte swizzle) whose other
//   rows stay zero.
// * warps 2-9 (two per TMEM lane quarter) read each key's G logits from TMEM (one lane
//   per key) and keep an online softmax (FlashAttention's rescaling): one warp-wide max
//   per head and tile (redux.sync), per-lane normalisers summed only at the end of the
//   segment, and o rescaled only when a max grew.  V half: lanes over the head dim,
//   each warp over its 16 rows of the tile, packed fp32x2 FMA with the probabilities
//   passed as (p, p) pairs through a small per-warp buffer.  Rows at or past n are
//   never touched.
// * at the end of a segment each compute warp stages its (max, normaliser, o) in shared
//   memory (double-buffered) and moves on; warps 10-13 merge the eight warps' states.
//   A unit covered by one segment is written directly; otherwise each segment's (max,
//   normaliser, o) goes to the workspace and the last CTA to finish one of the unit's
//   segments (atomic counter, no waiting) merges them and writes the bf16 output,
//   resetting the counter.  The counters live in a fixed 512 KB header of the workspace
//   (one int per unit, at most 131072 units) that is zero between calls, whatever the
//   call shapes.
// * every wait is bounded (on expiry the CTA sets the device timeout flag and abandons
//   its work), and the V reader checks the stage tag as a self-check of the ring.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int ROWS = 128;    // rows per tile (the MMA's M)
constexpr int NST = 4;         // ring depth (K or V tiles; K in even stages, V in odd)
constexpr int NCW = 8;         // compute warps: NCW / 4 per TMEM lane quarter
constexpr int WROWS = ROWS / NCW;  // rows of a tile per compute warp in the V half
constexpr int NEW = 4;         // epilogue warps: merge each segment's warp states
constexpr int NTH = 32 * (NCW + NEW + 2);
constexpr int EPI0 = 32 * (NCW + 2);  // first epilogue thread
constexpr int MINB = 1;        // resident CTAs per SM
static_assert(NCW % 4 == 0 && WROWS <= 32 && NST <= 8 && NST % 2 == 0, "geometry");
constexpr int QN = 16;       // MMA N: query heads padded with zero rows
constexpr int TMEM_COLS = 32;  // two 16-column S^T buffers

template <int D, int G>
struct DGeo {
  static constexpr int KB = D / 64;
  static constexpr int KBLK = ROWS * 128;        // bytes of one k-block of a tile
  static constexpr int TB = KB * KBLK;           // bytes of one K or V tile
  static constexpr int QBLK = QN * 128;          // bytes of one k-block of the q operand
  static constexpr int QOP = KB * QBLK;          // bytes of one q operand
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_Q = NST * TB;                     // [2] q operands (1024-aligned)
  static constexpr int OFF_P = OFF_Q + 2 * QOP;              // (p, p) pairs [NCW][WROWS][G]
  static constexpr int OFF_STAGE = OFF_P + NCW * WROWS * G * 8;  // fp32 [2][NCW][G][D] warp o
  static constexpr int OFF_SST = OFF_STAGE + 2 * NCW * G * D * 4;  // float2 [2][NCW][G] (m, l)
  static constexpr int OFF_SCL = OFF_SST + 2 * NCW * G * 8;  // fp32 [NCW][G] warp weights
  static constexpr int OFF_ML = OFF_SCL + NCW * G * 4;       // float2 [G] segment (M, L)
  static constexpr int OFF_BAR = OFF_ML + G * 8;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;
  static constexpr int DV = D / 32;              // head-dim elements per lane in the V half
  static_assert(G <= QN, "the query heads must fit the MMA's N");
  static_assert(QOP % 1024 == 0 && TB % 1024 == 0, "swizzled operands stay 1024-aligned");
};

// barrier offsets (bytes from OFF_BAR)
constexpr int B_FULL = 0;      // [NST] ring stage filled (TMA)
constexpr int B_EMPTY = 64;    // [NST] ring stage free (MMA commit for K, NCW warps for V)
constexpr int B_QFULL = 128;   // [2] q operand written (NCW compute warps)
constexpr int B_QEMPTY = 144;  // [2] q operand no longer read (MMA commit after the unit)
constexpr int B_SFULL = 160;   // [2] S^T buffer written (MMA commit)
constexpr int B_SEMPTY = 176;  // [2] S^T buffer read (NCW warps)
constexpr int B_RFULL = 192;   // [2] segment warp states staged (NCW compute warps)
constexpr int B_REMPTY = 208;  // [2] staged states consumed (epilogue)
constexpr int B_ABORT = 224;   // int
constexpr int B_LAST = 228;    // int
constexpr int B_TMEM = 232;    // uint32
constexpr int B_EOK = 236;     // int: the epilogue's wait succeeded
constexpr int B_TAG = 256;     // int [NST]: the tile index last issued into each stage
static_assert(B_TAG + 4 * NST <= 512, "barrier area");

// L2 prefetch of one box of a 2-D tensor map (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
               :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y) : "memory");
}

// Bounded spin until a stage's tile tag reaches `want` (it is written by the producer
// after the stage was released and before its load is issued, so once it matches, the
// stage's full barrier is at most one phase from the awaited one).
__device__ __forceinline__ bool wait_tag(volatile int *tag, int want, const Abort &ab) {
  if (*tag == want) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    if (*tag == want) return true;
    if (ab.raised()) return false;
    if ((it & 15u) == 0 && globaltimer_ns() - t0 > ab.limit) break;
    __nanosleep(32);
  }
  ab.raise();
  return false;
}

struct DecP {
  const __nv_bfloat16 *q;
  float c;                 // log2(e)/sqrt(D)
  int32_t *n_valid;        // [U] or null
  const __nv_bfloat16 *k_new, *v_new;  // [U, D] or null (append)
  __nv_bfloat16 *kc, *vc;  // the caches [U, cap, D] (append writes one row)
  int32_t *pos;            // [U, cap] or null
  int new_pos;
  int n_uniform, cap;
  int units, tiles_per_unit;  // tile slots of ROWS rows per unit (for n <= cap)
  __nv_bfloat16 *out;
  int ga;                  // query heads per unit in q and out (<= G; heads ga..G-1 pad the MMA)
  float2 *part_ml;         // [U][T][G] per-segment (max, normaliser)
  float *part_o;           // [U][T][G][D] per-segment unnormalised o
  int *cnt;                // [U]
  uint32_t *status;
  unsigned long long timeout;
};

// the two bf16 of a packed word as a fp32x2 pair
__device__ __forceinline__ unsigned long long bf2(uint32_t w) {
  return pk(bf_lo(w), bf_hi(w));
}

// Writes 16-byte chunk e of the appended K/V row into the cache; chunk 0's thread also
// records the position and the new row count.
template <int D>
__device__ __forceinline__ void append_row(const DecP &p, int u, int arow, int n_old, int e) {
  const size_t dst = ((size_t)u * p.cap + arow) * D + (size_t)e * 8;
  *reinterpret_cast<uint4 *>(p.kc + dst) = *reinterpret_cast<const uint4 *>(p.k_new + (size_t)u * D + e * 8);
  *reinterpret_cast<uint4 *>(p.vc + dst) = *reinterpret_cast<const uint4 *>(p.v_new + (size_t)u * D + e * 8);
  if (e == 0) {
    if (p.pos) p.pos[(size_t)u * p.cap + arow] = p.new_pos;
    p.n_valid[u] = n_old + 1;
  }
}

// Patches the appended row `arr` of a K or V tile in shared memory (threads 0..D/8-1).
template <int D>
__device__ __forceinline__ void patch_row(uint8_t *tile, const __nv_bfloat16 *src_row, int arr,
                                          int t) {
  constexpr int KBLK = ROWS * 128;
  if (t < D / 8) {
    const int kb = t >> 3, ci = t & 7;
    uint8_t *dst = tile + kb * KBLK + arr * 128 + ((ci ^ (arr & 7)) << 4);
    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src_row + t * 8);
  }
}

// Balanced split of `total` tile slots over P CTAs: CTA b owns [first(b), first(b+1)).
__device__ __forceinline__ int slot_first(int b, int Q, int R) { return b * Q + min(b, R); }
__device__ __forceinline__ int slot_owner(int slot, int Q, int R) {
  return slot < R * (Q + 1) ? slot / (Q + 1) : R + (slot - R * (Q + 1)) / Q;
}

// Geometry of the segment of unit u that CTA b owns.
struct Seg {
  int r0, r1;      // rows [r0, r1) of the unit (r1 <= n), possibly empty
  int arow;        // appended row of the unit, -1 if none
  int n_old;       // rows before the append
  int nseg, iseg;  // segments of the unit and this one's index among them
};

__device__ __forceinline__ Seg seg_geo(const DecP &p, int u, int b, int s0, int s1, int T, int Q,
                                       int R, bool report) {
  Seg g;
  int n = p.n_valid ? p.n_valid[u] : p.n_uniform;
  if (n > p.cap || n < 0) {
    if (report) set_status(p.status, KVC_DEV_BAD_STATE);
    n = n < 0 ? 0 : p.cap;
  }
  g.n_old = n;
  g.arow = -1;
  if (p.k_new) {
    if (n < p.cap) {
      g.arow = n;
      n = n + 1;
    } else if (report && slot_owner(u * T, Q, R) == b) {
      set_status(p.status, KVC_DEV_CACHE_FULL);
    }
  }
  if (n > T * ROWS) {  // more rows than the planned bound: they are not attended
    if (report) set_status(p.status, KVC_DEV_BAD_STATE);
  }
  const int t_lo = max(s0, u * T) - u * T, t_hi = min(s1, (u + 1) * T) - u * T;
  g.r0 = t_lo * ROWS;
  g.r1 = min(t_hi * ROWS, n);
  if (g.r1 < g.r0) g.r1 = g.r0;
  const int b0 = slot_owner(u * T, Q, R), b1 = slot_owner(u * T + T - 1, Q, R);
  g.nseg = b1 - b0 + 1;
  g.iseg = b - b0;
  return g;
}



template <int D, int G>
__global__ void __launch_bounds__(NTH, MINB) decode_kernel(const __grid_constant__ CUtensorMap tk,
                                                     const __grid_constant__ CUtensorMap tv,
                                                     const DecP p) {
  using Gm = DGeo<D, G>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar = sb + Gm::OFF_BAR;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + B_ABORT);
  volatile int *last_flag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + B_LAST);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Gm::OFF_BAR + B_TMEM);
  volatile int *tag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + B_TAG);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{abort_flag, p.status, p.timeout};
  const int T = p.tiles_per_unit, P = gridDim.x, b = blockIdx.x;
  const int total = p.units * T, Q = total / P, R = total % P;
  const int s0 = slot_first(b, Q, R), s1 = slot_first(b + 1, Q, R);
  const int u_first = s0 / T, u_last = s1 > s0 ? (s1 - 1) / T : u_first - 1;
  // Order of the CTA's units: its last unit (usually shared with the next CTA) first,
  // then the others in order.  Every unit shared with a neighbour is then worked on
  // early by both CTAs, so the split merges happen early and a CTA's final segment is
  // usually a whole unit, written without the merge.
  const int nu = u_last - u_first + 1;
  auto unit_at = [&](int kk) { return kk == 0 ? u_last : u_first + kk - 1; };

  // both q operands start zero: TMA later writes only their rows 0..G-1
  for (int e = threadIdx.x; e < 2 * Gm::QOP / 16; e += NTH)
    reinterpret_cast<uint4 *>(smem + Gm::OFF_Q)[e] = make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // seen by the tensor cores
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NST; ++i) {
      tag[i] = -1;
      mbar_init(bar + B_FULL + 8 * i, 1);
      mbar_init(bar + B_EMPTY + 8 * i, NCW);  // V: 8 warps; K: 8 commits of its MMA
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar + B_QFULL + 8 * i, NCW);  // the compute warps wrote the unit's q
      mbar_init(bar + B_QEMPTY + 8 * i, 1);   // the MMAs of the unit have completed
      mbar_init(bar + B_SFULL + 8 * i, 1);
      mbar_init(bar + B_SEMPTY + 8 * i, NCW);
      mbar_init(bar + B_RFULL + 8 * i, NCW);
      mbar_init(bar + B_REMPTY + 8 * i, 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Programmatic dependent launch: the next kernel of the stream may start launching
  // now (its CTAs take SM slots as this grid's CTAs exit, and wait here until this grid
  // has completed); this grid waits for the previous kernel before reading anything
  // it wrote (q, the caches, n_valid, the workspace counters).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0 && nu > 0) {
    // While the previous kernel finishes: pull the first tiles of this CTA's first unit
    // into L2 (slot range only; the row count is not read before the wait).  L2 stays
    // coherent with that kernel's writes, so this is only a hint.
    const int u = unit_at(0);
    const int t_lo = max(s0, u * T) - u * T, t_hi = min(s1, (u + 1) * T) - u * T;
    for (int t2 = t_lo; t2 < t_hi && t2 < t_lo + NST / 2; ++t2)
      for (int kb = 0; kb < Gm::KB; ++kb) {
        tma_prefetch_l2(&tk, kb * 64, u * p.cap + t2 * ROWS);
        tma_prefetch_l2(&tv, kb * 64, u * p.cap + t2 * ROWS);
      }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ------ TMA producer: per segment its q, then its tiles as K0, V0, K1, V1, ... ------
    if (lane == 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int it = 0, k = 0;
      bool ok = true;
      for (; k < nu && ok; ++k) {
        const int u = unit_at(k);
        const Seg g = seg_geo(p, u, b, s0, s1, T, Q, R, false);
        const int ntiles = (g.r1 - g.r0 + ROWS - 1) / ROWS;
        for (int i = 0; i < 2 * ntiles; ++i, ++it) {
          const int st = it % NST, use = it / NST;
          if (!ab.wait(bar + B_EMPTY + 8 * st, (use & 1) ^ 1)) { ok = false; break; }
          __threadfence_block();  // the release seen above comes before the new tag
          tag[st] = it;
          mbar_arrive_expect_tx(bar + B_FULL + 8 * st, Gm::TB);
          const int row = u * p.cap + g.r0 + (i >> 1) * ROWS;
          const CUtensorMap *map = (i & 1) ? &tv : &tk;
          for (int kb = 0; kb < Gm::KB; ++kb)
            tma_load_2d(sb + Gm::OFF_RING + st * Gm::TB + kb * Gm::KBLK, map, kb * 64, row,
                        bar + B_FULL + 8 * st);
        }
      }
      for (int st = 0; st < NST; ++st) {  // drain
        const int cnt = it / NST + (st < it % NST ? 1 : 0);
        if (cnt > 0) mbar_wait_bounded(bar + B_FULL + 8 * st, (cnt - 1) & 1, p.timeout);
      }
      (void)k;
    }
  } else if (warp == 1) {
    // ---------- MMA issuer: S^T = K_tile . q^T for every K tile, into TMEM ----------
    if (lane == 0) {
      int it = 0, k = 0, sc = 0, last_sb = -1, last_par = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16(ROWS, QN);
      for (; k < nu && ok; ++k) {
        const int u = unit_at(k);
        const Seg g = seg_geo(p, u, b, s0, s1, T, Q, R, false);
        const int qb = k & 1;
        if (!ab.wait(bar + B_QFULL + 8 * qb, (k >> 1) & 1)) { ok = false; break; }
        const uint64_t qd = sdesc_k128(sb + Gm::OFF_Q + qb * Gm::QOP);
        const int ntiles = (g.r1 - g.r0 + ROWS - 1) / ROWS;
        const int arow_local = g.arow - g.r0;
        for (int i = 0; i < ntiles; ++i, ++sc) {
          const int j = it + 2 * i, st = j % NST;
          const int sbf = sc & 1;
          // wait until the producer has reissued the stage before trusting the full
          // barrier's parity (needed whenever a stage's previous use was released by
          // other warps, as with an odd ring depth; cheap otherwise)
          if (!wait_tag(tag + st, j, ab)) { ok = false; break; }
          __threadfence_block();
          if (!ab.wait(bar + B_FULL + 8 * st, (j / NST) & 1)) { ok = false; break; }
          if (!ab.wait(bar + B_SEMPTY + 8 * sbf, ((sc >> 1) & 1) ^ 1)) { ok = false; break; }
          const int arr = arow_local - i * ROWS;
          if (g.arow >= 0 && arr >= 0 && arr < ROWS) {  // the appended row, from k_new
            uint8_t *tile = smem + Gm::OFF_RING + st * Gm::TB;
            for (int c = 0; c < D / 8; ++c) patch_row<D>(tile, p.k_new + (size_t)u * D, arr, c);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          }
          tc_fence_after();
          const uint64_t kd = sdesc_k128(sb + Gm::OFF_RING + st * Gm::TB);
          const uint32_t d = tmem + (uint32_t)(sbf * QN);
#pragma unroll
          for (int kb = 0; kb < Gm::KB; ++kb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ko = (uint64_t)((kb * Gm::KBLK + kk * 32) >> 4);
              const uint64_t qo = (uint64_t)((kb * Gm::QBLK + kk * 32) >> 4);
              umma_bf16(d, kd + ko, qd + qo, idesc, (kb | kk) != 0);
            }
          }
          umma_commit(bar + B_SFULL + 8 * sbf);
          // the K stage is free once these MMAs complete: one commit plus NCW - 1 plain
          // arrivals, so the stage's NCW-count barrier completes on the commit
          umma_commit(bar + B_EMPTY + 8 * st);
#pragma unroll
          for (int r = 1; r < NCW; ++r) mbar_arrive(bar + B_EMPTY + 8 * st);
          last_sb = sbf;
          last_par = (sc >> 1) & 1;
        }
        if (!ok) break;
        it += 2 * ntiles;
        umma_commit(bar + B_QEMPTY + 8 * qb);  // q buffer free once this unit's MMAs complete
      }
      // drain: every commit issued has arrived before the CTA may exit (commits complete
      // in order, so the last one covers the rest)
      if (ok && k > 0) mbar_wait_bounded(bar + B_QEMPTY + 8 * ((k - 1) & 1), ((k - 1) >> 1) & 1, p.timeout);
      else if (last_sb >= 0) mbar_wait_bounded(bar + B_SFULL + 8 * last_sb, last_par, p.timeout);
    }
  } else if (warp < 2 + NCW) {
    // ------------------------------ compute warps ------------------------------
    const int cw = warp - 2;          // 0..NCW-1
    const int quarter = warp & 3;     // TMEM lane quarter = keys quarter*32 .. +31 of a tile
    const int half = cw >> 2;         // this warp's WROWS of the quarter's 32 keys
    const int t = threadIdx.x - 64;   // 0..32*NCW-1
    const bool own = lane / WROWS == half;
    constexpr int DV = Gm::DV;
    // (p, p) pairs of the warp's rows: [WROWS][G]
    unsigned long long *pw = reinterpret_cast<unsigned long long *>(smem + Gm::OFF_P) + cw * WROWS * G;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    // this lane's byte offset inside a row of a V tile (128-byte swizzle undone per row)
    const int vchunk = D == 128 ? lane >> 1 : lane >> 2;
    const int vkb = vchunk >> 3, vci = vchunk & 7;
    const int vsub = D == 128 ? (lane & 1) * 8 : (lane & 3) * 4;
    int it = 0, sc = 0;
    bool ok = true;
    // q of unit uu into operand buffer qb: rows 0..ga-1, one 16-byte chunk per thread
    // (rows ga..15 stay zero)
    auto write_q = [&](int uu, int qb) {
      uint8_t *qo = smem + Gm::OFF_Q + qb * Gm::QOP;
      for (int c = t; c < p.ga * D / 8; c += 32 * NCW) {
        const int g = c / (D / 8), ch = c % (D / 8), kb = ch >> 3, ci = ch & 7;
        *reinterpret_cast<uint4 *>(qo + kb * Gm::QBLK + g * 128 + ((ci ^ (g & 7)) << 4)) =
            *reinterpret_cast<const uint4 *>(p.q + ((size_t)uu * p.ga + g) * D + ch * 8);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // for the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + B_QFULL + 8 * qb);
    };
    if (nu > 0) write_q(unit_at(0), 0);
    if (nu > 1) write_q(unit_at(1), 1);
    for (int k = 0; k < nu; ++k) {
      const int u = unit_at(k);
      const Seg sg = seg_geo(p, u, b, s0, s1, T, Q, R, t == 0);
      // the next unit's q goes where the previous unit's was, once the MMAs of the
      // previous unit have completed (it may have had no tiles here, so its S^T reads
      // prove nothing)
      if (k > 0 && k + 1 < nu) {
        ok = __all_sync(0xffffffffu, ok && ab.wait(bar + B_QEMPTY + 8 * ((k - 1) & 1), ((k - 1) >> 1) & 1));
        if (ok) write_q(unit_at(k + 1), (k + 1) & 1);
      }
      // running max (the same on every lane: it covers the quarter's 32 keys), and per
      // lane the normaliser of its own key rows and o over its head-dim slice
      float m_run[G], l_run[G];
      unsigned long long o2[G][DV / 2];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.f;
#pragma unroll
        for (int d = 0; d < DV / 2; ++d) o2[g][d] = 0ull;
      }
      const int nrows = sg.r1 - sg.r0;
      const int ntiles = (nrows + ROWS - 1) / ROWS;
      const int arow_local = sg.arow - sg.r0;
      for (int i = 0; i < ntiles; ++i, ++sc) {
        // ---------------- logits of this lane's key, from TMEM ----------------
        float lg[G];
        {
          const int sbf = sc & 1;
          const bool got = __all_sync(0xffffffffu, ok && ab.wait(bar + B_SFULL + 8 * sbf, (sc >> 1) & 1));
          ok = got;
#pragma unroll
          for (int g = 0; g < G; ++g) lg[g] = -INFINITY;
          if (got) {
            tc_fence_after();
            float s8[8];
            tmem_ld8(tmem + lane_base + (uint32_t)(sbf * QN), s8);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + B_SEMPTY + 8 * sbf);
            if (i * ROWS + quarter * 32 + lane < nrows)
#pragma unroll
              for (int g = 0; g < G; ++g) lg[g] = s8[g] * p.c;
          }
        }
        // ------- online softmax: one warp max per head, no per-tile sums -------
        bool grew = false;
        float f[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float mx;
          asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(mx) : "f"(lg[g]));
          const float mnew = fmaxf(m_run[g], mx);
          grew |= mnew > m_run[g];
          f[g] = mnew > m_run[g] ? (m_run[g] == -INFINITY ? 0.f : ex2(m_run[g] - mnew)) : 1.f;
          const float e = mnew == -INFINITY ? 0.f : ex2(lg[g] - mnew);  // ex2(-inf) = 0
          if (own) pw[(lane % WROWS) * G + g] = pk(e, e);
          l_run[g] = l_run[g] * f[g] + (own ? e : 0.f);
          m_run[g] = mnew;
        }
        if (grew) {  // warp-uniform: the maxima are the same on every lane
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const unsigned long long ff = pk(f[g], f[g]);
#pragma unroll
            for (int d = 0; d < DV / 2; ++d) {
              unsigned long long z = 0ull;
              ffma2(z, o2[g][d], ff);
              o2[g][d] = z;
            }
          }
        }
        __syncwarp();  // probabilities visible to the whole warp
        // ---------------- V half: o[g] += p[row][g] * v[row] ----------------
        {
          const int j = it + 2 * i + 1, st = j % NST;
          bool got = __all_sync(0xffffffffu, ok && ab.wait(bar + B_FULL + 8 * st, (j / NST) & 1));
          // self-check of the ring protocol: the stage must hold this tile
          if (got && !__all_sync(0xffffffffu, tag[st] == j)) {
            if (lane == 0) {
              set_status(p.status, KVC_DEV_BAD_STATE);
              *abort_flag = 1;
            }
            got = false;
          }
          ok = got;
          uint8_t *tile = smem + Gm::OFF_RING + st * Gm::TB;
          const int arr = arow_local - i * ROWS;
          const bool patched = sg.arow >= 0 && arr >= 0 && arr < ROWS;  // same for the CTA
          if (patched) {  // every compute thread reaches this barrier
            if (got) patch_row<D>(tile, p.v_new + (size_t)u * D, arr, t);
            named_bar(1, 32 * NCW);
          }
          const int r0 = quarter * 32 + half * WROWS;              // first own row of the tile
          const int wrows = min(WROWS, nrows - i * ROWS - r0);      // own rows (<= 0: none)
          if (got) {
            const uint8_t *vrow = tile + vkb * Gm::KBLK + r0 * 128 + vsub;
            auto row = [&](int i2) {
              // r0 is a multiple of 8, so the row's swizzle phase is i2 & 7
              const uint8_t *src = vrow + i2 * 128 + ((vci ^ (i2 & 7)) << 4);
              unsigned long long v01, v23 = 0ull;
              if (D == 128) {
                const uint2 w = *reinterpret_cast<const uint2 *>(src);
                v01 = bf2(w.x);
                v23 = bf2(w.y);
              } else {
                v01 = bf2(*reinterpret_cast<const uint32_t *>(src));
              }
              const unsigned long long *pr = pw + i2 * G;
#pragma unroll
              for (int g = 0; g < G; g += 2) {
                unsigned long long pp0, pp1 = 0ull;
                if (G >= 2) {
                  const ulonglong2 q2 = *reinterpret_cast<const ulonglong2 *>(pr + g);
                  pp0 = q2.x;
                  pp1 = q2.y;
                } else {
                  pp0 = pr[g];
                }
                ffma2(o2[g][0], pp0, v01);
                if (DV == 4) ffma2(o2[g][DV / 2 - 1], pp0, v23);
                if (G >= 2) {
                  ffma2(o2[g + 1 < G ? g + 1 : g][0], pp1, v01);
                  if (DV == 4) ffma2(o2[g + 1 < G ? g + 1 : g][DV / 2 - 1], pp1, v23);
                }
              }
            };
            if (wrows == WROWS) {
#pragma unroll
              for (int i2 = 0; i2 < WROWS; ++i2) row(i2);
            } else {
#pragma unroll 4
              for (int i2 = 0; i2 < WROWS; ++i2) {
                if (i2 >= wrows) break;
                row(i2);
              }
            }
            if (patched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + B_EMPTY + 8 * st);
          }
          __syncwarp();  // pw is rewritten by the next tile
        }
      }
      it += 2 * ntiles;
      // ---- hand the warp's (max, normaliser, o) of this segment to the epilogue ----
      float lw[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float sum = l_run[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        lw[g] = sum;
      }
      const int rb = k & 1;
      if (k >= 2)  // the epilogue has finished with segment k - 2's buffer
        ok = __all_sync(0xffffffffu, ok && ab.wait(bar + B_REMPTY + 8 * rb, ((k - 2) >> 1) & 1));
      if (ok) {
        float *stg = reinterpret_cast<float *>(smem + Gm::OFF_STAGE) + ((size_t)rb * NCW + cw) * G * D;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (DV == 4) {
            const float2 a = upk(o2[g][0]), c2 = upk(o2[g][DV / 2 - 1]);
            *reinterpret_cast<float4 *>(stg + g * D + lane * 4) = make_float4(a.x, a.y, c2.x, c2.y);
          } else {
            *reinterpret_cast<float2 *>(stg + g * D + lane * 2) = upk(o2[g][0]);
          }
        }
        if (lane == 0) {
          float2 *sst = reinterpret_cast<float2 *>(smem + Gm::OFF_SST) + ((size_t)rb * NCW + cw) * G;
#pragma unroll
          for (int g = 0; g < G; ++g) sst[g] = make_float2(m_run[g], lw[g]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar + B_RFULL + 8 * rb);
      }
    }
  } else {
    // --------------- epilogue warps: merge each segment's staged warp states ---------------
    constexpr int NE = 32 * NEW;
    const int te = threadIdx.x - EPI0;  // 0..NE-1
    volatile int *eok_flag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + B_EOK);
    float *scl = reinterpret_cast<float *>(smem + Gm::OFF_SCL);     // [NCW][G]
    float2 *mlv = reinterpret_cast<float2 *>(smem + Gm::OFF_ML);    // [G] (M, L)
    for (int k = 0; k < nu; ++k) {
      const int u = unit_at(k), rb = k & 1;
      const Seg sg = seg_geo(p, u, b, s0, s1, T, Q, R, false);
      if (te == 0) *eok_flag = ab.wait(bar + B_RFULL + 8 * rb, (k >> 1) & 1) ? 1 : 0;
      named_bar(2, NE);
      const bool eok = *eok_flag != 0;  // the same for the whole group
      const float2 *sst = reinterpret_cast<const float2 *>(smem + Gm::OFF_SST) + (size_t)rb * NCW * G;
      const float *stg = reinterpret_cast<const float *>(smem + Gm::OFF_STAGE) + (size_t)rb * NCW * G * D;
      if (eok && te < G) {  // the segment's max and normaliser per head, and warp weights
        const int g = te;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, sst[w * G + g].x);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float2 ml = sst[w * G + g];
          const float s = ml.x == -INFINITY ? 0.f : ex2(ml.x - M);
          scl[w * G + g] = s;
          L += ml.y * s;
        }
        mlv[g] = make_float2(M, L);
      }
      named_bar(2, NE);
      const bool direct = sg.nseg == 1;
      if (eok) {
        for (int e = te; e < G * D; e += NE) {
          const int g = e / D, d = e - g * D;
          float O = 0.f;
#pragma unroll
          for (int w = 0; w < NCW; ++w) O += stg[(size_t)w * G * D + e] * scl[w * G + g];
          const float2 ml = mlv[g];
          if (direct) {
            if (g < p.ga)
              p.out[((size_t)u * p.ga + g) * D + d] = __float2bfloat16(ml.y > 0.f ? O / ml.y : 0.f);
            if (e < D / 8 && sg.arow >= 0) append_row<D>(p, u, sg.arow, sg.n_old, e);
          } else {
            p.part_o[(((size_t)u * T + sg.iseg) * G + g) * D + d] = O;
            if (d == 0) p.part_ml[((size_t)u * T + sg.iseg) * G + g] = ml;
          }
        }
      }
      named_bar(2, NE);  // the staged states, weights and (M, L) have been read
      if (te == 0) mbar_arrive(bar + B_REMPTY + 8 * rb);
      if (eok && !direct) {
        __threadfence();
        named_bar(2, NE);
        if (te == 0) *last_flag = (atomicAdd(&p.cnt[u], 1) == sg.nseg - 1);
        named_bar(2, NE);
        if (*last_flag) {
          __threadfence();
          for (int e = te; e < G * D; e += NE) {
            const int g = e / D, d = e - g * D;
            // independent loads (batched by unrolling), then the merge
            float M = -INFINITY;
#pragma unroll 4
            for (int s2 = 0; s2 < sg.nseg; ++s2)
              M = fmaxf(M, __ldcg(p.part_ml + ((size_t)u * T + s2) * G + g).x);
            float L = 0.f, O = 0.f;
            if (M != -INFINITY) {
#pragma unroll 4
              for (int s2 = 0; s2 < sg.nseg; ++s2) {
                const float2 ml = __ldcg(p.part_ml + ((size_t)u * T + s2) * G + g);
                const float o = __ldcg(p.part_o + (((size_t)u * T + s2) * G + g) * D + d);
                const float fs = ml.y > 0.f ? ex2(ml.x - M) : 0.f;  // empty segments add 0
                L += ml.y * fs;
                O += o * fs;
              }
            }
            if (g < p.ga) p.out[((size_t)u * p.ga + g) * D + d] = __float2bfloat16(L > 0.f ? O / L : 0.f);
          }
          if (sg.arow >= 0)
            for (int e = te; e < D / 8; e += NE) append_row<D>(p, u, sg.arow, sg.n_old, e);
          if (te == 0) p.cnt[u] = 0;
        }
        named_bar(2, NE);  // last_flag is reused by the next segment
      }
    }
  }

  // ---------------------------------- teardown ----------------------------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

template <int D, int G>
cudaError_t launch_t(const Ctx &c, const DecodeArgs &a, DecP p) {
  static bool attr[64];
  static int per_sm[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DGeo<D, G>::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[dev], decode_kernel<D, G>, NTH,
                                                      DGeo<D, G>::SMEM);
    if (e != cudaSuccess) return e;
    if (per_sm[dev] < 1) return cudaErrorInvalidConfiguration;
    attr[dev] = true;
  }
  CUtensorMap tk, tv;
  if (!encode_rows_map(&tk, a.k_cache, (uint64_t)a.units * a.cap, D, ROWS)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&tv, a.v_cache, (uint64_t)a.units * a.cap, D, ROWS)) return cudaErrorInvalidValue;
  // persistent grid: every resident CTA slot, but never more CTAs than tile slots
  const long long slots = (long long)a.units * p.tiles_per_unit;
  long long grid = (long long)c.num_sms * (dev < 64 ? per_sm[dev] : 1);
  if (grid > slots) grid = slots;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(NTH);
  cfg.dynamicSmemBytes = DGeo<D, G>::SMEM;
  cfg.stream = c.stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol above
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<D, G>, tk, tv, p);
}

}  // namespace

constexpr size_t CNT_HEADER = (size_t)KVC_DECODE_MAX_UNITS * sizeof(int);  // per-unit counters,
                                                                            // zero between calls

size_t decode_counter_bytes(int units) { return (size_t)units * sizeof(int); }

// Query heads per unit as the kernel instantiates them: G rounded up to 1, 2, 4 or 8.
int padded_group(int G) { return G <= 1 ? 1 : (G <= 2 ? 2 : (G <= 4 ? 4 : 8)); }

// Workspace: the counter header, then per unit and segment (at most one segment per
// tile slot) the partial (max, normaliser) per head and the partial o per head.
size_t decode_ws_bytes(int units, int G, int D, int cap, int num_sms) {
  G = padded_group(G);
  const size_t smax = (size_t)(cap > 0 ? (cap + ROWS - 1) / ROWS : 1);
  size_t b = CNT_HEADER;
  b += (size_t)units * smax * G * sizeof(float2);
  b += (size_t)units * smax * G * D * sizeof(float);
  (void)num_sms;
  return (b + 255) & ~(size_t)255;
}

cudaError_t launch_decode(const Ctx &c, const DecodeArgs &a) {
  // rows per unit to plan for: n_uniform, or with n_valid the caller's bound on the row
  // count after the append (0: the capacity)
  const int n_max = a.n_valid ? (a.n_uniform > 0 ? a.n_uniform : a.cap) : a.n_uniform;
  const int T = n_max > 0 ? (n_max + ROWS - 1) / ROWS : 1;  // tile slots per unit
  const size_t smax = (size_t)(a.cap > 0 ? (a.cap + ROWS - 1) / ROWS : 1);
  DecP p;
  p.q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
  p.c = (float)(1.4426950408889634 / sqrt((double)a.D));
  p.n_valid = a.n_valid;
  p.k_new = reinterpret_cast<const __nv_bfloat16 *>(a.k_new);
  p.v_new = reinterpret_cast<const __nv_bfloat16 *>(a.v_new);
  p.kc = reinterpret_cast<__nv_bfloat16 *>(a.k_cache);
  p.vc = reinterpret_cast<__nv_bfloat16 *>(a.v_cache);
  p.pos = a.pos;
  p.new_pos = a.new_pos;
  p.n_uniform = a.n_uniform;
  p.cap = a.cap;
  p.units = a.units;
  p.tiles_per_unit = T;
  p.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
  p.ga = a.G;
  const int Gp = padded_group(a.G);
  uint8_t *w = reinterpret_cast<uint8_t *>(a.ws);
  p.cnt = reinterpret_cast<int *>(w);
  p.part_ml = reinterpret_cast<float2 *>(w + CNT_HEADER);
  p.part_o = reinterpret_cast<float *>(w + CNT_HEADER + (size_t)a.units * smax * Gp * sizeof(float2));
  p.status = c.status;
  p.timeout = c.timeout_ns;
#define KVC_DEC(DD, GG) \
  if (a.D == DD && Gp == GG) return launch_t<DD, GG>(c, a, p);
  KVC_DEC(128, 1) KVC_DEC(128, 2) KVC_DEC(128, 4) KVC_DEC(128, 8)
  KVC_DEC(64, 1) KVC_DEC(64, 2) KVC_DEC(64, 4) KVC_DEC(64, 8)
#undef KVC_DEC
  return cudaErrorInvalidValue;
}

}  // namespace kvc
