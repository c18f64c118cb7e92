// Decode attention over a compact (SnapKV) or sink + ring (StreamingLLM) cache: for
// each query head of each (layer, batch, KV head) unit, o = softmax(q . K_c^T / sqrt(D))
// . V_c over the unit's first n rows (SnapKV article, 推論方法: decoding reads only the
// compressed cache; StreamingLLM article, 推論の流れ: attention over sink and recent
// tokens only).  An optional append adds the step's new K/V row first (fused: the CTA
// whose tile holds the new row patches it in shared memory from k_new/v_new, and the
// unit's finishing CTA writes it to the cache, its position and the new n_valid).
//
// Design (sm_103a, HBM-bound: every cached K/V byte is read once):
// * persistent stream-K: all units' 64-row tile slots form one sequence that is split
//   evenly over a grid of resident CTAs (three per SM), so every CTA streams the same
//   number of tiles; a CTA's range covers segments of one or more units.  Warp 0
//   streams each segment's tiles as K0, V0, K1, V1, ... through one continuous 4-stage
//   shared-memory ring with TMA (128-byte swizzle, one mbarrier pair per stage), so the
//   next segment's loads overlap the current segment's epilogue; warps 1-4 compute.
//   The throughput of a CTA is the bytes in flight over the memory latency, so the
//   shared memory goes to the ring: no logit buffer, no block-wide softmax.
// * each compute warp owns 16 rows of every tile, in both halves of the step, and keeps
//   its own online softmax (running max, normaliser and o per head; FlashAttention's
//   rescaling), so a tile needs no synchronisation between the warps.
// * K half: D/8 threads per row, each owning one 16-byte chunk (8 head dims) of the row
//   (conflict-free reads of the swizzled tile); the thread's slice of q, pre-scaled by
//   log2(e)/sqrt(D), lives in registers (a bulk copy brings each unit's q to shared
//   memory ahead of time); packed fp32x2 FMA; a transpose-reduce over the row's lanes
//   leaves one head's logit per lane.  The warp's 16 probabilities per head go through
//   a small per-warp buffer to every lane.
// * V half: lanes over the head dim, packed FMA with those probabilities.  Rows at or
//   past n are never touched.
// * at the end of a segment the four warps' (max, normaliser, o) merge in shared
//   memory; a unit covered by one segment is written directly, otherwise each
//   segment's (max, normaliser, o) goes to the workspace and the last CTA to finish one
//   of the unit's segments (atomic counter, no waiting) merges them and writes the bf16
//   output, resetting the counter.  The counters live in a fixed 256 KB header of the
//   workspace (one int per unit, at most 65535 units) that is zero between calls,
//   whatever the call shapes.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int ROWS = 64;     // rows per tile
constexpr int NST = 4;       // ring depth (K or V tiles)
constexpr int NCW = 4;       // compute warps
constexpr int WROWS = ROWS / NCW;  // rows of a tile per compute warp
constexpr int NTH = 32 * (NCW + 1);

template <int D, int G>
struct DGeo {
  static constexpr int KB = D / 64;
  static constexpr int KBLK = ROWS * 128;        // bytes of one k-block of a tile
  static constexpr int TB = KB * KBLK;           // bytes of one K or V tile
  static constexpr int QB = G * D * 2;           // bytes of one unit's q (bf16)
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_QB = NST * TB;                    // bf16 [2][G][D]
  static constexpr int OFF_P = OFF_QB + 2 * QB;              // fp32 [NCW][WROWS][G] probabilities
  static constexpr int OFF_RED = OFF_P + NCW * WROWS * G * 4;  // fp32 [G][D] merged o
  static constexpr int OFF_WX = OFF_RED + G * D * 4;         // fp32 [NCW][G] tile max / sum
  static constexpr int OFF_ST = OFF_WX + NCW * G * 4;        // float2 [NCW][G] (max, normaliser)
  static constexpr int OFF_BAR = OFF_ST + NCW * G * 8;
  static constexpr int SMEM = OFF_BAR + 128 + 1024;
  static constexpr int DV = D / 32;              // head-dim elements per lane in the V half
  static constexpr int TPR = D / 8;              // K half: threads per row, one chunk each
  static constexpr int RPW = 32 / TPR;           // K half: rows per warp and pass
  static constexpr int NPASS = WROWS / RPW;      // K half: passes over the warp's rows
  static_assert(G <= TPR, "every head's logit needs a lane of the row");
};

struct DecP {
  const __nv_bfloat16 *q;
  float c;                 // log2(e)/sqrt(D)
  int32_t *n_valid;        // [U] or null
  const __nv_bfloat16 *k_new, *v_new;  // [U, D] or null (append)
  __nv_bfloat16 *kc, *vc;  // the caches [U, cap, D] (append writes one row)
  int32_t *pos;            // [U, cap] or null
  int new_pos;
  int n_uniform, cap;
  int units, tiles_per_unit;  // tile slots of 64 rows per unit (for n <= cap)
  __nv_bfloat16 *out;
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
__global__ void __launch_bounds__(NTH, 3) decode_kernel(const __grid_constant__ CUtensorMap tk,
                                                     const __grid_constant__ CUtensorMap tv,
                                                     const DecP p) {
  using Gm = DGeo<D, G>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  float *red = reinterpret_cast<float *>(smem + Gm::OFF_RED);   // [G][D] merged o
  float *wx = reinterpret_cast<float *>(smem + Gm::OFF_WX);     // [NCW][G] tile max / sum
  float2 *wst = reinterpret_cast<float2 *>(smem + Gm::OFF_ST);  // [NCW][G] (max, normaliser)
  // barriers: full[NST] at +0, empty[NST] at +32, qfull[2] at +64, qempty[2] at +80
  const uint32_t bar = sb + Gm::OFF_BAR;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + 96);
  volatile int *last_flag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + 100);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{abort_flag, p.status, p.timeout};
  const int T = p.tiles_per_unit, P = gridDim.x, b = blockIdx.x;
  const int total = p.units * T, Q = total / P, R = total % P;
  const int s0 = slot_first(b, Q, R), s1 = slot_first(b + 1, Q, R);
  const int u_first = s0 / T, u_last = s1 > s0 ? (s1 - 1) / T : u_first - 1;

  for (int e = threadIdx.x; e < G * D; e += NTH) red[e] = 0.f;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar + 8 * i, 1);
      mbar_init(bar + 32 + 8 * i, NCW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar + 64 + 8 * i, 1);
      mbar_init(bar + 80 + 8 * i, NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // Programmatic dependent launch: the next kernel of the stream may start launching
  // now (its CTAs take SM slots as this grid's CTAs exit, and wait here until this grid
  // has completed); this grid waits for the previous kernel before reading anything
  // it wrote (q, the caches, n_valid, the workspace counters).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ------ TMA producer: per segment its q, then its tiles as K0, V0, K1, V1, ... ------
    if (lane == 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int it = 0, k = 0;
      bool ok = true;
      for (int u = u_first; u <= u_last && ok; ++u, ++k) {
        const Seg g = seg_geo(p, u, b, s0, s1, T, Q, R, false);
        const int qb = k & 1;
        if (!ab.wait(bar + 80 + 8 * qb, ((k >> 1) & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(bar + 64 + 8 * qb, Gm::QB);
        bulk_load(sb + Gm::OFF_QB + qb * Gm::QB, p.q + (size_t)u * G * D, Gm::QB, bar + 64 + 8 * qb);
        const int ntiles = (g.r1 - g.r0 + ROWS - 1) / ROWS;
        for (int i = 0; i < 2 * ntiles; ++i, ++it) {
          const int st = it % NST, use = it / NST;
          if (!ab.wait(bar + 32 + 8 * st, (use & 1) ^ 1)) { ok = false; break; }
          mbar_arrive_expect_tx(bar + 8 * st, Gm::TB);
          const int row = u * p.cap + g.r0 + (i >> 1) * ROWS;
          const CUtensorMap *map = (i & 1) ? &tv : &tk;
          for (int kb = 0; kb < Gm::KB; ++kb)
            tma_load_2d(sb + Gm::OFF_RING + st * Gm::TB + kb * Gm::KBLK, map, kb * 64, row,
                        bar + 8 * st);
        }
      }
      for (int st = 0; st < NST; ++st) {  // drain
        const int cnt = it / NST + (st < it % NST ? 1 : 0);
        if (cnt > 0) mbar_wait_bounded(bar + 8 * st, (cnt - 1) & 1, p.timeout);
      }
      for (int qb = 0; qb < 2; ++qb) {
        const int cnt = k / 2 + (qb < k % 2 ? 1 : 0);
        if (cnt > 0) mbar_wait_bounded(bar + 64 + 8 * qb, (cnt - 1) & 1, p.timeout);
      }
    }
    return;
  }

  // ------------------------------ compute warps ------------------------------
  const int cw = warp - 1;         // 0..3: owns rows [cw*WROWS, (cw+1)*WROWS) of every tile
  const int t = threadIdx.x - 32;  // 0..127
  constexpr int TPR = Gm::TPR, RPW = Gm::RPW, NPASS = Gm::NPASS, DV = Gm::DV;
  constexpr int WMASK = TPR / G - 1;  // lanes of a row holding the same head's logit
  const int rg = lane / TPR;          // K half: row within the warp's pass
  const int sl = lane % TPR;          // K half: the thread's 16-byte chunk of the row
  // the head whose logit this lane holds after the transpose-reduce (see below)
  int myhead = 0;
#pragma unroll
  for (int lvl = TPR / 2, nv = G; lvl >= 1; lvl >>= 1)
    if (nv >= 2) {
      if (lane & lvl) myhead += nv / 2;
      nv /= 2;
    }
  const bool row_writer = (lane & WMASK) == 0;        // one lane per (row, head)
  const bool head_writer = row_writer && lane < TPR;  // one lane per head
  float *pw = reinterpret_cast<float *>(smem + Gm::OFF_P) + cw * WROWS * G;  // [WROWS][G]
  float *wxw = wx + cw * G;
  int it = 0, k = 0;
  bool ok = true;
  for (int u = u_first; u <= u_last; ++u, ++k) {
    const Seg sg = seg_geo(p, u, b, s0, s1, T, Q, R, t == 0);
    // q slice of this thread: chunk sl of every head, fp32 pairs, pre-scaled
    unsigned long long qr[G][4];
    {
      const int qb = k & 1;
      const bool got = __all_sync(0xffffffffu, ok && ab.wait(bar + 64 + 8 * qb, (k >> 1) & 1));
      ok = got;
      const uint8_t *qsm = smem + Gm::OFF_QB + qb * Gm::QB;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint4 w = got ? *reinterpret_cast<const uint4 *>(qsm + (g * D + sl * 8) * 2)
                            : make_uint4(0, 0, 0, 0);
        qr[g][0] = pk(bf_lo(w.x) * p.c, bf_hi(w.x) * p.c);
        qr[g][1] = pk(bf_lo(w.y) * p.c, bf_hi(w.y) * p.c);
        qr[g][2] = pk(bf_lo(w.z) * p.c, bf_hi(w.z) * p.c);
        qr[g][3] = pk(bf_lo(w.w) * p.c, bf_hi(w.w) * p.c);
      }
      __syncwarp();
      if (got && lane == 0) mbar_arrive(bar + 80 + 8 * qb);
    }
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
    for (int i = 0; i < ntiles; ++i, it += 2) {
      const int arr = arow_local - i * ROWS;
      const bool patched = sg.arow >= 0 && arr >= 0 && arr < ROWS;  // same for the CTA
      const int wrows = min(WROWS, nrows - i * ROWS - cw * WROWS);   // this warp's rows (<= 0: none)
      // ---------------- K half: logits of the warp's rows ----------------
      float lg[NPASS];
      {
        const int st = it % NST;
        const bool got = __all_sync(0xffffffffu, ok && ab.wait(bar + 8 * st, (it / NST) & 1));
        ok = got;
        uint8_t *tile = smem + Gm::OFF_RING + st * Gm::TB;
        if (patched) {  // every compute thread reaches this barrier
          if (got) patch_row<D>(tile, p.k_new + (size_t)u * D, arr, t);
          named_bar(1, 128);
        }
#pragma unroll
        for (int pass = 0; pass < NPASS; ++pass) lg[pass] = -INFINITY;
        if (got) {
#pragma unroll
          for (int pass = 0; pass < NPASS; ++pass) {
            const int r = cw * WROWS + pass * RPW + rg;  // row of the tile
            // chunk sl: k-block sl / 8, slot sl % 8 (the 8 lanes of a phase hit 8 slots)
            const uint4 w = *reinterpret_cast<const uint4 *>(
                tile + (sl >> 3) * Gm::KBLK + r * 128 + (((sl & 7) ^ (r & 7)) << 4));
            const unsigned long long k01 = bf2(w.x), k23 = bf2(w.y), k45 = bf2(w.z),
                                     k67 = bf2(w.w);
            float v[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
              unsigned long long acc = 0ull;
              ffma2(acc, qr[g][0], k01);
              ffma2(acc, qr[g][1], k23);
              ffma2(acc, qr[g][2], k45);
              ffma2(acc, qr[g][3], k67);
              const float2 a = upk(acc);
              v[g] = a.x + a.y;
            }
            // transpose-reduce over the row's TPR lanes: each split level halves the heads a
            // lane keeps (the lane's bits at those levels name the head it keeps, myhead)
#pragma unroll
            for (int lvl = TPR / 2, nv = G; lvl >= 1; lvl >>= 1) {
              if (nv >= 2) {
                const bool upper = (lane & lvl) != 0;
#pragma unroll
                for (int x = 0; x < G / 2; ++x) {
                  if (x < nv / 2) {
                    const float send = upper ? v[x] : v[x + nv / 2];
                    const float keep = upper ? v[x + nv / 2] : v[x];
                    v[x] = keep + __shfl_xor_sync(0xffffffffu, send, lvl);
                  }
                }
                nv /= 2;
              } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], lvl);
              }
            }
            if (pass * RPW + rg < wrows) lg[pass] = v[0];
          }
          if (patched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(bar + 32 + 8 * st);  // the K stage may be refilled
        }
      }
      // ------- online softmax of the warp's rows (no other warp is involved) -------
      float mnew[G], f[G];
      {
        float tmax = lg[0];
#pragma unroll
        for (int pass = 1; pass < NPASS; ++pass) tmax = fmaxf(tmax, lg[pass]);
        // lanes holding the same head differ in the row bits (lane / TPR)
#pragma unroll
        for (int o = TPR; o < 32; o <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
        if (head_writer) wxw[myhead] = tmax;
        __syncwarp();
#pragma unroll
        for (int g = 0; g < G; ++g) {
          mnew[g] = fmaxf(m_run[g], wxw[g]);
          f[g] = m_run[g] == -INFINITY ? 0.f : ex2(m_run[g] - mnew[g]);  // rescale of the past
        }
        __syncwarp();  // wxw is reused for the sums
        float mh = mnew[0];
#pragma unroll
        for (int g = 1; g < G; ++g)
          if (myhead == g) mh = mnew[g];
        float ps = 0.f;
#pragma unroll
        for (int pass = 0; pass < NPASS; ++pass) {
          const float e = lg[pass] == -INFINITY ? 0.f : ex2(lg[pass] - mh);
          ps += e;
          if (row_writer) pw[(pass * RPW + rg) * G + myhead] = e;
        }
#pragma unroll
        for (int o = TPR; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        if (head_writer) wxw[myhead] = ps;
        __syncwarp();  // sums and probabilities visible to the whole warp
#pragma unroll
        for (int g = 0; g < G; ++g) {
          l_run[g] = l_run[g] * f[g] + wxw[g];
          m_run[g] = mnew[g];
          const unsigned long long ff = pk(f[g], f[g]);
#pragma unroll
          for (int d = 0; d < DV / 2; ++d) {
            unsigned long long z = 0ull;
            ffma2(z, o2[g][d], ff);
            o2[g][d] = z;
          }
        }
      }
      // ---------------- V half: o[g] += p[row][g] * v[row] ----------------
      {
        const int st = (it + 1) % NST;
        const bool got = __all_sync(0xffffffffu, ok && ab.wait(bar + 8 * st, ((it + 1) / NST) & 1));
        ok = got;
        uint8_t *tile = smem + Gm::OFF_RING + st * Gm::TB;
        if (patched) {
          if (got) patch_row<D>(tile, p.v_new + (size_t)u * D, arr, t);
          named_bar(1, 128);
        }
        if (got) {
#pragma unroll 4
          for (int i2 = 0; i2 < WROWS; ++i2) {
            if (i2 >= wrows) break;
            const int rr = cw * WROWS + i2;
            unsigned long long v01, v23 = 0ull;
            if (D == 128) {
              const int chunk = lane >> 1, kb = chunk >> 3, ci = chunk & 7;
              const uint2 w = *reinterpret_cast<const uint2 *>(
                  tile + kb * Gm::KBLK + rr * 128 + ((ci ^ (rr & 7)) << 4) + (lane & 1) * 8);
              v01 = bf2(w.x);
              v23 = bf2(w.y);
            } else {
              const int ci = lane >> 2;
              const uint32_t w = *reinterpret_cast<const uint32_t *>(
                  tile + rr * 128 + ((ci ^ (rr & 7)) << 4) + (lane & 3) * 4);
              v01 = bf2(w);
            }
            const float *pr = pw + i2 * G;
            float pv[G];
            if (G >= 4) {
#pragma unroll
              for (int g = 0; g < G; g += 4) {
                const float4 q4 = *reinterpret_cast<const float4 *>(pr + g);
                pv[g] = q4.x;
                pv[(g + 1) % G] = q4.y;
                pv[(g + 2) % G] = q4.z;
                pv[(g + 3) % G] = q4.w;
              }
            } else {
#pragma unroll
              for (int g = 0; g < G; ++g) pv[g] = pr[g];
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const unsigned long long pp = pk(pv[g], pv[g]);
              ffma2(o2[g][0], pp, v01);
              if (DV == 4) ffma2(o2[g][DV / 2 - 1], pp, v23);
            }
          }
          if (patched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(bar + 32 + 8 * st);
        }
        __syncwarp();  // pw and wxw are rewritten by the next tile
      }
    }
    // ---- merge the four warps' (max, normaliser, o) of this segment ----
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < G; ++g) wst[cw * G + g] = make_float2(m_run[g], l_run[g]);
    named_bar(1, 128);
    float Mg[G], Lg[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float M = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < NCW; ++w2) M = fmaxf(M, wst[w2 * G + g].x);
      float L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w2 = 0; w2 < NCW; ++w2) {
          const float2 ml = wst[w2 * G + g];
          if (ml.x != -INFINITY) L += ml.y * ex2(ml.x - M);
        }
      }
      Mg[g] = M;
      Lg[g] = L;
      const float fw = m_run[g] == -INFINITY ? 0.f : ex2(m_run[g] - M);
#pragma unroll
      for (int d = 0; d < DV / 2; ++d) {
        const float2 v = upk(o2[g][d]);
        atomicAdd(&red[g * D + lane * DV + 2 * d], v.x * fw);
        atomicAdd(&red[g * D + lane * DV + 2 * d + 1], v.y * fw);
      }
    }
    named_bar(1, 128);
    const bool direct = sg.nseg == 1;
    for (int e = t; e < G * D; e += 128) {
      const int g = e / D, d = e - g * D;
      float M = Mg[0], L = Lg[0];
#pragma unroll
      for (int h = 1; h < G; ++h)
        if (g == h) {
          M = Mg[h];
          L = Lg[h];
        }
      const float O = red[e];
      red[e] = 0.f;  // ready for the next segment (only this thread touches element e here)
      if (direct) {
        p.out[(size_t)u * G * D + e] = __float2bfloat16(L > 0.f ? O / L : 0.f);
        if (e < D / 8 && sg.arow >= 0) append_row<D>(p, u, sg.arow, sg.n_old, e);
      } else {
        p.part_o[(((size_t)u * T + sg.iseg) * G + g) * D + d] = O;
        if (d == 0) p.part_ml[((size_t)u * T + sg.iseg) * G + g] = make_float2(M, L);
      }
    }
    if (!direct) {
      __threadfence();
      named_bar(1, 128);
      if (t == 0) *last_flag = (atomicAdd(&p.cnt[u], 1) == sg.nseg - 1);
      named_bar(1, 128);
      if (*last_flag) {
        __threadfence();
        for (int e = t; e < G * D; e += 128) {
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
          p.out[(size_t)u * G * D + e] = __float2bfloat16(L > 0.f ? O / L : 0.f);
        }
        if (sg.arow >= 0)
          for (int e = t; e < D / 8; e += 128) append_row<D>(p, u, sg.arow, sg.n_old, e);
        if (t == 0) p.cnt[u] = 0;
      }
    }
    named_bar(1, 128);  // qs, red and last_flag are reused by the next segment
  }
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

constexpr size_t CNT_HEADER = 65536 * sizeof(int);  // per-unit counters, zero between calls

// Workspace: the counter header, then per unit and segment (at most one segment per
// tile slot) the partial (max, normaliser) per head and the partial o per head.
size_t decode_ws_bytes(int units, int G, int D, int cap, int num_sms) {
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
  uint8_t *w = reinterpret_cast<uint8_t *>(a.ws);
  p.cnt = reinterpret_cast<int *>(w);
  p.part_ml = reinterpret_cast<float2 *>(w + CNT_HEADER);
  p.part_o = reinterpret_cast<float *>(w + CNT_HEADER + (size_t)a.units * smax * a.G * sizeof(float2));
  p.status = c.status;
  p.timeout = c.timeout_ns;
#define KVC_DEC(DD, GG) \
  if (a.D == DD && a.G == GG) return launch_t<DD, GG>(c, a, p);
  KVC_DEC(128, 1) KVC_DEC(128, 2) KVC_DEC(128, 4) KVC_DEC(128, 8)
  KVC_DEC(64, 1) KVC_DEC(64, 2) KVC_DEC(64, 4) KVC_DEC(64, 8)
#undef KVC_DEC
  return cudaErrorInvalidValue;
}

}  // namespace kvc
