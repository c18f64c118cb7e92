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
//   streams each segment's K tiles and then its V tiles through one continuous 3-stage
//   shared-memory ring with TMA (128-byte swizzle, one mbarrier pair per stage), so the
//   next segment's loads overlap the current segment's epilogue; warps 1-4 compute.
// * K phase: D/8 threads per row, each owning one 16-byte chunk (8 head dims) of every
//   row (conflict-free reads of the swizzled tile); the thread's slice of q, pre-scaled
//   by log2(e)/sqrt(D), lives in registers (a bulk copy brings each unit's q to shared
//   memory ahead of time); packed fp32x2 FMA; a transpose-reduce over the row's lanes
//   leaves one head's logit per lane; the logits of the chunk go to shared memory.
// * one block reduction per chunk gives each head's maximum and normaliser; the logits
//   become exp2(s - max) in place (chunks of a long segment are merged with a running
//   maximum, rescaling the sums kept in registers).
// * V phase: lanes over the head dim, each warp over 16 rows of a tile, packed FMA
//   with the stored probabilities.  Rows at or past n are never touched.
// * the four warps' sums merge in shared memory; a unit covered by one segment is
//   written directly, otherwise each segment's (max, normaliser, o) goes to the
//   workspace and the last CTA to finish one of the unit's segments (atomic counter,
//   no waiting) merges them and writes the bf16 output, resetting the counter.  The counters live in a fixed 256 KB header of the workspace (one int per
//   unit, at most 65535 units) that is zero between calls, whatever the call shapes.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int ROWS = 64;     // rows per tile
constexpr int NST = 3;       // ring depth (K or V tiles)
constexpr int NCW = 4;       // compute warps
constexpr int NTH = 32 * (NCW + 1);

template <int D, int G>
struct DGeo {
  static constexpr int KB = D / 64;
  static constexpr int KBLK = ROWS * 128;        // bytes of one k-block of a tile
  static constexpr int TB = KB * KBLK;           // bytes of one K or V tile
  static constexpr int CMAX = 4096 / G;          // rows of one chunk (logits = 16 KB)
  static constexpr int QB = G * D * 2;           // bytes of one unit's q (bf16)
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_LOG = NST * TB;                   // fp32 [CMAX][G]; the merge
                                                             // buffer [NCW][G][D] reuses it
  static constexpr int OFF_QB = OFF_LOG + CMAX * G * 4;      // bf16 [2][G][D]
  static constexpr int OFF_ST = OFF_QB + 2 * QB;             // fp32 [NCW][G]
  static constexpr int OFF_BAR = OFF_ST + NCW * G * 4 + 64;
  static constexpr int SMEM = OFF_BAR + 128 + 1024;
  static constexpr int DV = D / 32;              // head-dim elements per lane in the V phase
  static constexpr int TPR = D / 8;              // K phase: threads per row, one chunk each
  static_assert(NCW * G * D * 4 <= CMAX * G * 4, "merge buffer must fit the logit buffer");
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
  float *slog = reinterpret_cast<float *>(smem + Gm::OFF_LOG);  // [row][G]
  float *red = slog;  // merge buffer, used only after a segment's V phase
  float *wst = reinterpret_cast<float *>(smem + Gm::OFF_ST);    // [NCW][G] per-warp partials
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
    // ------ TMA producer: per segment its q, then per sub-chunk K tiles, V tiles ------
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
        for (int c0 = g.r0; c0 < g.r1 && ok; c0 += Gm::CMAX) {
          const int ntiles = (min(g.r1, c0 + Gm::CMAX) - c0 + ROWS - 1) / ROWS;
          for (int i = 0; i < 2 * ntiles; ++i, ++it) {
            const int st = it % NST, use = it / NST;
            if (!ab.wait(bar + 32 + 8 * st, (use & 1) ^ 1)) { ok = false; break; }
            mbar_arrive_expect_tx(bar + 8 * st, Gm::TB);
            const int tt = i < ntiles ? i : i - ntiles;
            const int row = u * p.cap + c0 + tt * ROWS;
            const CUtensorMap *map = i < ntiles ? &tk : &tv;
            for (int kb = 0; kb < Gm::KB; ++kb)
              tma_load_2d(sb + Gm::OFF_RING + st * Gm::TB + kb * Gm::KBLK, map, kb * 64, row,
                          bar + 8 * st);
          }
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
  const int cw = warp - 1;         // 0..3
  const int t = threadIdx.x - 32;  // 0..127
  constexpr int TPR = Gm::TPR;
  const int rg = lane / TPR;       // K phase: row within the warp's group of 32/TPR rows
  const int sl = lane % TPR;       // K phase: the thread's 16-byte chunk of the row
  constexpr int DV = Gm::DV;
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
    for (int c0 = sg.r0; c0 < sg.r1; c0 += Gm::CMAX) {
      const int nrows = min(sg.r1, c0 + Gm::CMAX) - c0;
      const int ntiles = (nrows + ROWS - 1) / ROWS;
      const int arow_local = sg.arow - c0;
      // ---- K phase: logits of the sub-chunk's rows (8 threads per row) ----
      for (int i = 0; i < ntiles; ++i) {
        const int j = it + i, st = j % NST;
        const bool got = __all_sync(0xffffffffu, ok && ab.wait(bar + 8 * st, (j / NST) & 1));
        ok = got;
        uint8_t *tile = smem + Gm::OFF_RING + st * Gm::TB;
        const int arr = arow_local - i * ROWS;
        const bool patched = sg.arow >= 0 && arr >= 0 && arr < ROWS;  // same for the CTA
        if (patched) {  // every compute thread reaches this barrier
          if (got) patch_row<D>(tile, p.k_new + (size_t)u * D, arr, t);
          named_bar(1, 128);
        }
        if (got) {
          constexpr int RPW = 32 / TPR;  // rows per warp and pass
#pragma unroll 2
          for (int pass = 0; pass < ROWS / (NCW * RPW); ++pass) {
            const int r = (pass * NCW + cw) * RPW + rg;  // row of the tile
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
            // lane keeps; afterwards the lane's high bits name the head it holds
            int head = 0;
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
                if (upper) head += nv / 2;
                nv /= 2;
              } else {
                v[0] += __shfl_xor_sync(0xffffffffu, v[0], lvl);
              }
            }
            const int row = i * ROWS + r;
            constexpr int WMASK = TPR / G > 1 ? TPR / G - 1 : 0;
            if ((lane & WMASK) == 0 && row < nrows) slog[row * G + head] = v[0];
          }
          if (patched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(bar + 32 + 8 * st);
        }
      }
      named_bar(1, 128);
      // ---- sub-chunk max; new running max; p = exp2(s - max) in place; sums ----
      float mnew[G], f[G];
      {
        float mx[G];
#pragma unroll
        for (int g = 0; g < G; ++g) mx[g] = -INFINITY;
        for (int r = t; r < nrows; r += 128)
#pragma unroll
          for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], slog[r * G + g]);
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], o));
          if (lane == 0) wst[cw * G + g] = mx[g];
        }
        named_bar(1, 128);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float m2 = m_run[g];
#pragma unroll
          for (int w2 = 0; w2 < NCW; ++w2) m2 = fmaxf(m2, wst[w2 * G + g]);
          mnew[g] = m2;
          f[g] = m_run[g] == -INFINITY ? 0.f : ex2(m_run[g] - m2);  // rescale of earlier sums
        }
        float sm[G];
#pragma unroll
        for (int g = 0; g < G; ++g) sm[g] = 0.f;
        for (int r = t; r < nrows; r += 128)
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float e = ex2(slog[r * G + g] - mnew[g]);
            slog[r * G + g] = e;
            sm[g] += e;
          }
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sm[g] += __shfl_xor_sync(0xffffffffu, sm[g], o);
        }
        named_bar(1, 128);  // every warp read the maxima before wst is reused for sums
        if (lane == 0)
#pragma unroll
          for (int g = 0; g < G; ++g) wst[cw * G + g] = sm[g];
        named_bar(1, 128);  // sums and probabilities visible to all compute warps
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float l2 = 0.f;
#pragma unroll
          for (int w2 = 0; w2 < NCW; ++w2) l2 += wst[w2 * G + g];
          l_run[g] = l_run[g] * f[g] + l2;
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
      // ---- V phase: o[g] += p[row][g] * v[row], lanes over the head dim ----
      for (int i = 0; i < ntiles; ++i) {
        const int j = it + ntiles + i, st = j % NST;
        const bool got = __all_sync(0xffffffffu, ok && ab.wait(bar + 8 * st, (j / NST) & 1));
        ok = got;
        uint8_t *tile = smem + Gm::OFF_RING + st * Gm::TB;
        const int arr = arow_local - i * ROWS;
        const bool patched = sg.arow >= 0 && arr >= 0 && arr < ROWS;
        if (patched) {
          if (got) patch_row<D>(tile, p.v_new + (size_t)u * D, arr, t);
          named_bar(1, 128);
        }
        if (got) {
          const int rmax = min(16, nrows - i * ROWS - cw * 16);  // this warp's rows in the tile
#pragma unroll 4
          for (int i2 = 0; i2 < 16; ++i2) {
            if (i2 >= rmax) break;
            const int rr = cw * 16 + i2;
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
            const float *pr = slog + (i * ROWS + rr) * G;
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
      }
      it += 2 * ntiles;
      named_bar(1, 128);  // slog and wst of this sub-chunk are done with
    }
    // ---- merge the four warps' sums of this segment ----
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int d = 0; d < DV / 2; ++d) {
        const float2 v = upk(o2[g][d]);
        red[(cw * G + g) * D + lane * DV + 2 * d] = v.x;
        red[(cw * G + g) * D + lane * DV + 2 * d + 1] = v.y;
      }
    named_bar(1, 128);
    const bool direct = sg.nseg == 1;
    for (int e = t; e < G * D; e += 128) {
      const int g = e / D, d = e - g * D;
      float O = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < NCW; ++w2) O += red[(w2 * G + g) * D + d];
      if (direct) {
        p.out[(size_t)u * G * D + e] = __float2bfloat16(l_run[g] > 0.f ? O / l_run[g] : 0.f);
        if (e < D / 8 && sg.arow >= 0) append_row<D>(p, u, sg.arow, sg.n_old, e);
      } else {
        p.part_o[(((size_t)u * T + sg.iseg) * G + g) * D + d] = O;
        if (d == 0) p.part_ml[((size_t)u * T + sg.iseg) * G + g] = make_float2(m_run[g], l_run[g]);
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
