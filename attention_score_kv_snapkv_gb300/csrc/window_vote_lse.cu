// SnapKV votes (SnapKV article, 処理の流れ steps 1 and 2) -- and H2O's initial cumulative
// scores, with every prompt row voting -- when each voting row's softmax normaliser is
// already known: the prompt's attention computes it (the log-sum-exp lse of the row's
// causal scores), so the vote of key j is
//     v_j = sum over the voting rows i that see j of exp(q_i . k_j / sqrt(D) - lse_i),
// one exp per score and one pass over the keys, with no statistics to gather first.
//
// Design (sm_103a): the unit's R voting rows are cut into row groups of up to 256 rows
// (the largest N of one tcgen05.mma); the work is the flat list of (unit, row group,
// 128-key tile) items (the causal key tiles of each group only), cut into one contiguous
// range per CTA of a persistent grid (one CTA per SM): items are independent, so the
// split is even and no CTA waits for another.  Per item one tcgen05.mma chain forms
// S^T = K . Q^T (M = 128 keys on the TMEM lanes, N = the group's rows rounded up to 16,
// fp32) into one of NB tensor-memory buffers, so each key tile read serves up to 256
// rows.  Vote warps (one per lane quarter, in VS sets taking the items in turn) sum
// exp2(s.c - lse_i.log2 e) over the rows in registers with packed fp32x2 arithmetic -- no
// cross-lane reduction -- and store the vote (adding when several row groups vote on the
// same keys); a set reads the next row group's lse one item ahead.  Warp 0 = TMA
// producer (the group's Q tile, reloaded when the group changes; K tiles in a ring as
// deep as shared memory allows), warp 1 = TMEM owner and MMA issuer.  Every wait is
// bounded.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int TILE = 128;        // keys per tile
constexpr int QMAX = 256;        // rows per row group at most (N of one MMA)
constexpr int MAXSTAGE = 8;      // K tile ring depth at most
constexpr int VS = 2;            // vote-warp sets (items in turn)
constexpr int NVW = 4 * VS;      // vote warps
constexpr int NWARPS = 2 + NVW;
constexpr int NTHREADS = 32 * NWARPS;
constexpr int TMEM_COLS = 512;
constexpr int MAXNB = 32;
constexpr int SMEM_CAP = 227 * 1024;

// control region byte offsets
constexpr int C_QFULL = 0;       // [2]
constexpr int C_QEMPTY = 16;     // [2]
constexpr int C_KFULL = 32;      // [MAXSTAGE]
constexpr int C_KEMPTY = 96;     // [MAXSTAGE]
constexpr int C_SFULL = 160;     // [MAXNB]
constexpr int C_TFREE = 416;     // [MAXNB]
constexpr int C_TMEM = 672;
constexpr int C_ABORT = 676;
constexpr int C_LSE = 1024;                      // float [NVW][QMAX]: -lse . log2(e) per row
constexpr int C_ROWPOS = C_LSE + NVW * QMAX * 4; // int [NVW][QMAX]: the rows' positions
constexpr int C_END = C_ROWPOS + NVW * QMAX * 4;

struct LseP {
  int L, R, Wq, G, units;
  int qr;                // rows per row group (N of the MMA, a multiple of 16, <= 256)
  int row_groups;        // row groups per unit
  int nb, nstage;        // tensor-memory buffers, K ring depth
  int bcols;             // columns per tensor-memory buffer (qr rounded up to 32)
  int nqb;               // Q tile buffers (2 when a tile is at most 32 KB)
  int qbuf, off_k, off_ctrl;  // shared-memory layout (bytes from the 1024-aligned base)
  long long items;       // total (unit, row group, key tile) items
  long long ipu;         // items per unit
  int keep_k;            // 1: keep key tiles in L2 (several row groups read them)
  float c;               // log2(e) / sqrt(D)
  const float *lse;      // [units, G, L] natural-log log-sum-exp of every prompt row
  float *votes;          // [units, L]
  int atomic_votes;
  uint32_t *status;
  unsigned long long timeout;
};

// An item: unit, row group, key tile, with the group's geometry.
struct It {
  int u, rg, kt;
  int rho0, nrows, rpad, nkt, pmin, kend;
};

__device__ __forceinline__ void set_rg(const LseP &p, It &x) {
  x.rho0 = x.rg * p.qr;
  x.nrows = min(p.qr, p.R - x.rho0);
  x.rpad = (x.nrows + 15) & ~15;
  const int r0 = x.rho0 % p.Wq;
  const bool wraps = (r0 + x.nrows) > p.Wq;  // the group holds rows of several heads
  const int rmax = wraps ? p.Wq - 1 : r0 + x.nrows - 1;
  const int rmin = wraps ? 0 : r0;
  x.kend = p.L - p.Wq + rmax + 1;
  x.pmin = p.L - p.Wq + rmin;
  x.nkt = (x.kend + TILE - 1) / TILE;
}

// The item at flat index i (one walk over the row groups of a unit).
__device__ __forceinline__ It item_at(const LseP &p, long long i) {
  It x;
  x.u = (int)(i / p.ipu);
  long long r = i - (long long)x.u * p.ipu;
  x.rg = 0;
  set_rg(p, x);
  while (r >= x.nkt) {
    r -= x.nkt;
    ++x.rg;
    set_rg(p, x);
  }
  x.kt = (int)r;
  return x;
}

__device__ __forceinline__ void advance(const LseP &p, It &x) {
  if (++x.kt < x.nkt) return;
  x.kt = 0;
  if (++x.rg == p.row_groups) {
    x.rg = 0;
    ++x.u;
  }
  set_rg(p, x);
}

// A compact item position for the vote warps (the geometry is recomputed per item).
struct Pos {
  int u, rg, kt;
};

__device__ __forceinline__ It geo_of(const LseP &p, const Pos &x) {
  It g;
  g.u = x.u;
  g.rg = x.rg;
  g.kt = x.kt;
  set_rg(p, g);
  return g;
}

// Moves x forward by k items.
__device__ __forceinline__ void advance_by(const LseP &p, Pos &x, int k) {
  x.kt += k;
  for (;;) {
    const int nkt = geo_of(p, x).nkt;
    if (x.kt < nkt) return;
    x.kt -= nkt;
    if (++x.rg == p.row_groups) {
      x.rg = 0;
      ++x.u;
    }
  }
}

// Row `row` of the item's row group: its prompt position (-1 for padding) and its raw
// lse (NaN for padding).  Only issues the load: the value is consumed later (neg_log2).
__device__ __forceinline__ void row_load(const LseP &p, const It &x, int row, int &pos,
                                         float &raw) {
  pos = -1;
  raw = NAN;
  if (row < x.nrows) {
    const int rr = x.rho0 + row;                 // row index within the unit's R rows
    const int g = rr / p.Wq, w = rr - g * p.Wq;  // query head of the group, window row
    pos = p.L - p.Wq + w;
    raw = __ldg(p.lse + ((size_t)x.u * p.G + g) * p.L + pos);
  }
}

// -lse . log2(e); -inf (the row adds nothing) for padding or a non-finite lse.
__device__ __forceinline__ float neg_log2(float raw, int pos) {
  return (pos < 0 || !(fabsf(raw) < INFINITY)) ? -INFINITY : -raw * 1.4426950408889634f;
}

// Adds exp2(s c + nl_r) over the W rows of one chunk into four packed accumulators; with
// MASK, rows whose position lies before the lane's key add nothing.
template <int W, bool MASK>
__device__ __forceinline__ void vote_chunk(const float *sv, const float *nl, const int *rp, int key,
                                           unsigned long long cc, unsigned long long *acc) {
#pragma unroll
  for (int r = 0; r < W; r += 8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = r + 2 * j;
      const unsigned long long n2 = *reinterpret_cast<const unsigned long long *>(nl + c);
      const float2 t = upk(fma2(pk(sv[c], sv[c + 1]), cc, n2));
      float e0 = ex2(t.x), e1 = ex2(t.y);
      if (MASK) {
        const int2 p2 = *reinterpret_cast<const int2 *>(rp + c);
        if (key > p2.x) e0 = 0.f;
        if (key > p2.y) e1 = 0.f;
      }
      acc[j] = add2(acc[j], pk(e0, e1));
    }
  }
}

// QG: the launch's row groups hold at most QG rows (128 or 256); each vote warp's lanes
// take rows lane + 32 k of a group.
template <int D, int QG>
__global__ void __launch_bounds__(NTHREADS, 1)
    window_vote_lse_kernel(const __grid_constant__ CUtensorMap tq,
                           const __grid_constant__ CUtensorMap tk, const LseP p) {
  constexpr int KB = D / 64;                 // 64-column (128-byte) blocks per row
  constexpr int KBLK = TILE * 128;           // bytes of one block of a K tile
  constexpr int TILE_BYTES = KB * KBLK;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb, sK = sb + p.off_k, ctl = sb + p.off_ctrl;
  uint8_t *ctrl = smem + p.off_ctrl;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctrl + C_TMEM);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl + C_ABORT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{abort_flag, p.status, p.timeout};
  const int QR = p.qr, NB = p.nb, NS = p.nstage;
  const int QKBLK = QR * 128;  // bytes of one block of the Q tile
  const int qbytes = KB * QKBLK;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int qb = 0; qb < p.nqb; ++qb) {
      mbar_init(ctl + C_QFULL + 8 * qb, 1);
      mbar_init(ctl + C_QEMPTY + 8 * qb, 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(ctl + C_KFULL + 8 * s, 1);
      mbar_init(ctl + C_KEMPTY + 8 * s, 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(ctl + C_SFULL + 8 * b, 1);
      mbar_init(ctl + C_TFREE + 8 * b, 4);  // the four warps of the set that takes it
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // this CTA's contiguous range of items
  const long long i0 = p.items * blockIdx.x / gridDim.x;
  const long long i1 = p.items * (blockIdx.x + 1) / gridDim.x;
  const int n = (int)(i1 - i0);

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0 && n > 0) {
      It x = item_at(p, i0);
      int nq = 0, nk = 0;  // Q loads, K loads issued
      int qb = 0, qph = 0, s = 0, kph = 0;  // Q slot and K stage with their use parities
      const uint64_t pol_k = p.keep_k ? l2_policy_evict_last() : l2_policy_evict_first();
      for (int i = 0; i < n; ++i) {
        if (i == 0 || x.kt == 0) {  // a new row group: its Q tile, once the slot is free
          if (i > 0 && ++qb == p.nqb) {
            qb = 0;
            qph ^= 1;
          }
          if (!ab.wait(ctl + C_QEMPTY + 8 * qb, qph ^ 1)) break;
          mbar_arrive_expect_tx(ctl + C_QFULL + 8 * qb, qbytes);
          for (int kb = 0; kb < KB; ++kb)
            tma_load_2d(sQ + qb * p.qbuf + kb * QKBLK, &tq, kb * 64, x.u * p.R + x.rho0,
                        ctl + C_QFULL + 8 * qb);
          ++nq;
        }
        if (!ab.wait(ctl + C_KEMPTY + 8 * s, kph ^ 1)) break;
        mbar_arrive_expect_tx(ctl + C_KFULL + 8 * s, TILE_BYTES);
        for (int kb = 0; kb < KB; ++kb)
          tma_load_2d_hint(sK + s * TILE_BYTES + kb * KBLK, &tk, kb * 64,
                           x.u * p.L + x.kt * TILE, ctl + C_KFULL + 8 * s, pol_k);
        ++nk;
        if (++s == NS) {
          s = 0;
          kph ^= 1;
        }
        advance(p, x);
      }
      // before the CTA exits, every copy issued has landed (a stage or the Q buffer holds
      // at most one copy in flight: the earlier ones were consumed), also after an abort
      for (int s = 0; s < NS; ++s) {
        const int cnt = nk / NS + (s < nk % NS ? 1 : 0);
        if (cnt > 0) mbar_wait_bounded(ctl + C_KFULL + 8 * s, (cnt - 1) & 1, p.timeout);
      }
      for (int qb = 0; qb < p.nqb; ++qb) {
        const int cnt = nq / p.nqb + (qb < nq % p.nqb ? 1 : 0);
        if (cnt > 0) mbar_wait_bounded(ctl + C_QFULL + 8 * qb, (cnt - 1) & 1, p.timeout);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0 && n > 0) {
      It x = item_at(p, i0);
      int nq = 0, last_bar = -1, last_par = 0;
      int qb = 0, qph = 0, s = 0, kph = 0, b = 0, bph = 0;  // slots and use parities
      bool ok = true;
      uint32_t idesc = 0;
      uint64_t qd = 0;
      for (int i = 0; i < n && ok; ++i) {
        if (i == 0 || x.kt == 0) {
          if (i > 0) {
            umma_commit(ctl + C_QEMPTY + 8 * qb);  // the previous group's MMAs read it last
            if (++qb == p.nqb) {
              qb = 0;
              qph ^= 1;
            }
          }
          if (!ab.wait(ctl + C_QFULL + 8 * qb, qph)) { ok = false; break; }
          ++nq;
          tc_fence_after();
          idesc = idesc_bf16(128, x.rpad);
          qd = sdesc_k128(sQ + qb * p.qbuf);
        }
        if (!ab.wait(ctl + C_KFULL + 8 * s, kph)) { ok = false; break; }
        if (!ab.wait(ctl + C_TFREE + 8 * b, bph ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * p.bcols);
        const uint64_t kd = sdesc_k128(sK + s * TILE_BYTES);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ko = (uint64_t)((kb * KBLK + kk * 32) >> 4);
            const uint64_t qo = (uint64_t)((kb * QKBLK + kk * 32) >> 4);
            umma_bf16(d, kd + ko, qd + qo, idesc, (kb | kk) != 0);
          }
        }
        umma_commit(ctl + C_KEMPTY + 8 * s);
        umma_commit(ctl + C_SFULL + 8 * b);
        last_bar = b;
        last_par = bph;
        if (++s == NS) {
          s = 0;
          kph ^= 1;
        }
        if (++b == NB) {
          b = 0;
          bph ^= 1;
        }
        advance(p, x);
      }
      if (ok && nq > 0) umma_commit(ctl + C_QEMPTY + 8 * qb);
      if (last_bar >= 0) mbar_wait_bounded(ctl + C_SFULL + 8 * last_bar, last_par, p.timeout);
    }
  } else {
    // ------------- votes: one warp per TMEM lane quarter and set, every row -------------
    const int vw = warp - 2;
    const int q = warp & 3;
    const int vset = vw >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float *nls = reinterpret_cast<float *>(ctrl + C_LSE) + vw * QMAX;  // -lse . log2(e)
    int *rps = reinterpret_cast<int *>(ctrl + C_ROWPOS) + vw * QMAX;
    const unsigned long long cc = pk(p.c, p.c);
    // the set's items: vset, vset + VS, ...
    if (vset < n) {
      // The rows' lse of the next row group are loaded into registers one item ahead and
      // stored to the tables after the item.
      Pos x;
      {
        const It f = item_at(p, i0 + vset);
        x.u = f.u;
        x.rg = f.rg;
        x.kt = f.kt;
      }
      constexpr int RPL = QG / 32;  // rows per lane
      float raw[RPL];
      int rpos[RPL];
      {
        const It g = geo_of(p, x);
#pragma unroll
        for (int k = 0; k < RPL; ++k) row_load(p, g, lane + 32 * k, rpos[k], raw[k]);
      }
#pragma unroll
      for (int k = 0; k < RPL; ++k) {
        rps[lane + 32 * k] = rpos[k];
        nls[lane + 32 * k] = neg_log2(raw[k], rpos[k]);
      }
      __syncwarp();
      bool ok = true;
      int b = vset, bph = 0;  // the item's buffer and its use parity
      for (int i = vset; i < n; i += VS) {
        Pos nx = x;
        advance_by(p, nx, VS);
        const bool refill = i + VS < n && (nx.u != x.u || nx.rg != x.rg);
        if (refill) {
          const It g = geo_of(p, nx);
#pragma unroll
          for (int k = 0; k < RPL; ++k)
            row_load(p, g, lane + 32 * k, rpos[k], raw[k]);
        }
        const It g = geo_of(p, x);
        const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_SFULL + 8 * b, bph));
        ok = got;
        const int key = g.kt * TILE + q * 32 + lane;
        float vote = 0.f;
        if (got) {
          tc_fence_after();
          // warp-uniform: some key of the warp lies past some row's position, or padding
          const bool masked = (g.kt * TILE + q * 32 + 31 > g.pmin) || (g.nrows < g.rpad);
          const uint32_t ta = tmem + lane_base + (uint32_t)(b * p.bcols);
          unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
          int c0 = 0;
          const int c1 = g.rpad;
          if (!masked) {
#pragma unroll 1
            for (; c0 + 64 <= c1; c0 += 64) {
              float sv[64];
              tmem_ld32(ta + c0, sv);
              tmem_ld32(ta + c0 + 32, sv + 32);
              tmem_wait_ld();
              vote_chunk<64, false>(sv, nls + c0, rps + c0, key, cc, acc);
            }
          }
#pragma unroll 1
          for (; c0 < c1; c0 += 32) {
            float sv[32];
            if (c1 - c0 >= 32) {
              tmem_ld32(ta + c0, sv);
              tmem_wait_ld();
              if (masked) vote_chunk<32, true>(sv, nls + c0, rps + c0, key, cc, acc);
              else vote_chunk<32, false>(sv, nls + c0, rps + c0, key, cc, acc);
            } else {
              tmem_ld16(ta + c0, sv);
              tmem_wait_ld();
              if (masked) vote_chunk<16, true>(sv, nls + c0, rps + c0, key, cc, acc);
              else vote_chunk<16, false>(sv, nls + c0, rps + c0, key, cc, acc);
            }
          }
          const float2 t = upk(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])));
          vote = t.x + t.y;
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(ctl + C_TFREE + 8 * b);
        }
        if (got && key < g.kend) {
          float *dst = p.votes + (size_t)g.u * p.L + key;
          if (p.atomic_votes)
            atomicAdd(dst, vote);
          else
            *dst = vote;
        }
        if (refill) {
#pragma unroll
          for (int k = 0; k < RPL; ++k) {
            rps[lane + 32 * k] = rpos[k];
            nls[lane + 32 * k] = neg_log2(raw[k], rpos[k]);
          }
          __syncwarp();
        }
        x = nx;
        if ((b += VS) >= NB) {  // NB is a multiple of VS
          b -= NB;
          bph ^= 1;
        }
      }
    }
  }

  // ---------------------------------- teardown ----------------------------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

bool g_attr_done[4][64];

}  // namespace

cudaError_t launch_window_vote_lse(const Ctx &c, const WindowVoteLseArgs &a) {
  int dev = 0;
  cudaGetDevice(&dev);
  LseP p;
  p.L = a.L;
  p.R = a.G * a.Wq;
  p.Wq = a.Wq;
  p.G = a.G;
  p.units = a.units;
  p.qr = p.R >= QMAX ? QMAX : ((p.R + 15) & ~15);
  const bool big = p.qr > 128;
  const int di = (a.D == 128 ? 2 : 0) + (big ? 1 : 0);
  const void *fn = a.D == 128 ? (big ? (const void *)window_vote_lse_kernel<128, 256>
                                     : (const void *)window_vote_lse_kernel<128, 128>)
                              : (big ? (const void *)window_vote_lse_kernel<64, 256>
                                     : (const void *)window_vote_lse_kernel<64, 128>);
  if (dev < 64 && !g_attr_done[di][dev]) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_CAP);
    if (e != cudaSuccess) return e;
    g_attr_done[di][dev] = true;
  }
  p.row_groups = (p.R + p.qr - 1) / p.qr;
  // a multiple of VS, so that buffer b always serves vote set b % VS (each barrier phase
  // is then awaited by one set only, in order)
  p.bcols = (p.qr + 31) & ~31;
  p.nb = (TMEM_COLS / p.bcols) / VS * VS;
  if (p.nb > MAXNB) p.nb = MAXNB;
  // shared memory: the Q tile (two buffers when small), then as many K stages as fit
  // beside the control region
  const int tile_bytes = a.D / 64 * TILE * 128;
  p.qbuf = (a.D / 64 * p.qr * 128 + 1023) & ~1023;
  p.nqb = p.qbuf <= 32 * 1024 ? 2 : 1;
  const int ns = (SMEM_CAP - 1024 - p.nqb * p.qbuf - C_END) / tile_bytes;
  p.nstage = ns > MAXSTAGE ? MAXSTAGE : ns;
  p.off_k = p.nqb * p.qbuf;
  p.off_ctrl = p.off_k + p.nstage * tile_bytes;
  int smem = p.off_ctrl + C_END + 1024;      // + base alignment slack
  if (smem < 116 * 1024) smem = 116 * 1024;  // one CTA per SM: each takes all 512 columns
  long long ipu = 0;
  for (int rg = 0; rg < p.row_groups; ++rg) {
    const int rho0 = rg * p.qr;
    const int nrows = (p.R - rho0) < p.qr ? p.R - rho0 : p.qr;
    const int r0 = rho0 % p.Wq;
    const bool wraps = r0 + nrows > p.Wq;
    const int rmax = wraps ? p.Wq - 1 : r0 + nrows - 1;
    ipu += (p.L - p.Wq + rmax + 1 + TILE - 1) / TILE;
  }
  p.ipu = ipu;
  p.items = ipu * a.units;
  // the keys of a unit are read again by its other row groups: keep them in L2 then
  p.keep_k = p.row_groups > 1;
  p.c = (float)(1.4426950408889634 / sqrt((double)a.D));
  p.lse = a.lse;
  p.votes = a.votes;
  p.atomic_votes = p.row_groups > 1;
  p.status = c.status;
  p.timeout = c.timeout_ns;
  CUtensorMap tq, tk;
  if (!encode_rows_map(&tq, a.q, (uint64_t)a.units * p.R, a.D, p.qr)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&tk, a.k, (uint64_t)a.units * a.L, a.D, TILE)) return cudaErrorInvalidValue;
  int blocks_per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, fn, NTHREADS, smem);
  if (e != cudaSuccess) return e;
  if (blocks_per_sm != 1) return cudaErrorInvalidConfiguration;
  if (p.atomic_votes) {
    e = cudaMemsetAsync(a.votes, 0, (size_t)a.units * a.L * sizeof(float), c.stream);
    if (e != cudaSuccess) return e;
  }
  const long long grid = p.items < c.num_sms ? p.items : c.num_sms;
  if (grid < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  if (a.D == 128) {
    if (big) return cudaLaunchKernelEx(&cfg, window_vote_lse_kernel<128, 256>, tq, tk, p);
    return cudaLaunchKernelEx(&cfg, window_vote_lse_kernel<128, 128>, tq, tk, p);
  }
  if (big) return cudaLaunchKernelEx(&cfg, window_vote_lse_kernel<64, 256>, tq, tk, p);
  return cudaLaunchKernelEx(&cfg, window_vote_lse_kernel<64, 128>, tq, tk, p);
}

}  // namespace kvc
