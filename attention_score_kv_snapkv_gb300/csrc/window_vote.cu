// SnapKV steps 1-2 (SnapKV article, 処理の流れ steps 1 and 2): every trailing window
// query of the G query heads of a KV head takes softmax(q . k / sqrt(D)) over the keys
// it may see (all keys up to and including its own position), and the probabilities
// are summed per key into the vote.  With every prompt query as a "window" query this
// is also H2O's initial cumulative score (causal column sums of the prompt attention).
//
// Design (sm_103a):
// * A job is (unit u, tile of up to 128 query rows).  Its key range is cut into
//   128-key tiles; the tiles are split over a group of g CTAs of a persistent,
//   cooperatively launched grid (one CTA per SM).
// * Pass 1, per key tile: S = Q . K^T on the tensor cores (tcgen05.mma, M = 128 query
//   rows, N = 128 keys, fp32 accumulator in TMEM).  The pass-1 warps (one thread per
//   row and column half) keep each row's running max m and normaliser z (log2 domain).
// * Row statistics are combined across the g CTAs of the job through global memory:
//   each CTA publishes its partial (max, normaliser) per row and bumps the job's
//   arrival counter; every CTA's pass-2 warps wait (bounded) for the count to reach g
//   and merge the g partials themselves (20 loads in flight per row).
// * Pass 2, per key tile: S^T = K . Q^T (M = 128 keys, N = rows rounded up to 16);
//   the pass-2 warps (one thread per key and row half) sum exp2(s*c - (m + log2 z))
//   over their rows in registers -- no cross-lane reduction -- and write the vote.
// * Pass 2 of job k is interleaved with pass 1 of job k+1 (after a lead of two
//   tiles), so the re-read of job k's keys comes from L2 and the statistics exchange
//   is hidden behind useful work.
// * Warp roles: warp 0 = TMA producer (Q tiles double-buffered, K tiles in a 4-stage
//   ring, 128-byte swizzle), warp 1 = TMEM owner and pass-1 MMA issuer, warp 18 =
//   pass-2 MMA issuer (separate issuers: tcgen05.mma issue is paced by the tensor pipe,
//   and a pass-2 tile waiting for statistics must not stall pass 1), warps 2-9 = pass 1
//   (two warps per TMEM lane quarter, each on half of the tile's key columns), warps
//   10-17 = pass 2 (two per lane quarter, each on half of the query rows; the halves
//   of a key's vote meet in shared memory).  Every wait is bounded (KVC_DEV_TIMEOUT).
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int TILE = 128;       // keys per tile; query rows per job
constexpr int NSTAGE = 4;       // K tile ring depth
constexpr int NQ = 2;           // Q tile buffers (a job's tile stays until its pass 2 is done)
constexpr int LAG = 1;          // round r streams pass 1 of job r and pass 2 of job r - LAG
static_assert(NQ >= LAG + 1, "the Q tiles of jobs r - LAG .. r must be resident together");
constexpr int NWARPS = 19;      // TMA, pass-1 MMA, 8 pass-1 warps, 8 pass-2 warps, pass-2 MMA
constexpr int NTHREADS = 32 * NWARPS;
constexpr int TMEM_COLS = 512;  // 4 accumulators of 128 fp32 columns
constexpr int LEAD = 2;         // pass-1 tiles of a round issued before its first pass-2 tile
constexpr int XB = 20;          // partial statistics loaded per batch (group sizes up to 20: one)
constexpr int TR_ROWS = 32;     // row tiles up to this size run pass 1 transposed (keys on lanes)
constexpr float TR_SLACK = 8.f; // transposed pass 1 moves a row's reference only past this (log2)

template <int D>
struct Geo {
  static constexpr int KB = D / 64;           // 128-byte k-blocks per row
  static constexpr int KBLK = TILE * 128;     // bytes of one k-block of a 128-row tile
  static constexpr int TILE_BYTES = KB * KBLK;
  static constexpr int OFF_Q = 0;             // NQ Q tiles
  static constexpr int OFF_K = NQ * TILE_BYTES;
  static constexpr int OFF_CTRL = OFF_K + NSTAGE * TILE_BYTES;
  static constexpr int CTRL_BYTES = 8192;
  static constexpr int NEED = OFF_CTRL + CTRL_BYTES + 1024;  // + base alignment slack
  // At least 116 KB so that two CTAs never share an SM: each CTA allocates all 512
  // TMEM columns, and the persistent grid relies on one resident CTA per SM.
  static constexpr int SMEM = NEED > 116 * 1024 ? NEED : 116 * 1024;
};

// control-region byte offsets
constexpr int C_QFULL = 0;      // NQ (<= 4) barriers
constexpr int C_QEMPTY = 32;    // NQ
constexpr int C_KFULL = 64;     // NSTAGE (<= 4)
constexpr int C_KEMPTY = 96;    // NSTAGE
constexpr int C_SFULL = 128;    // 4 (TMEM accumulators)
constexpr int C_SEMPTY = 160;   // 4
constexpr int C_XFULL = 192;    // 2 (local statistics hand-off, g == 1)
constexpr int C_XEMPTY = 208;   // 2
constexpr int C_TMEM = 224;
constexpr int C_ABORT = 228;
static_assert(NQ <= 4 && NSTAGE <= 4, "barrier slots");
constexpr int C_XSTAT = 256;    // float2 [2][128]  (2048 B)
constexpr int C_OFF = 2304;     // float [128] (16-byte aligned: read as float4)
constexpr int C_ROWPOS = 2816;  // int [128]
constexpr int C_GO = 3328;      // int: pass-2 warps may proceed (g > 1)
constexpr int C_HSTAT = 3456;   // float2 [2][128]: second column half's row statistics
constexpr int C_VPART = 5504;   // float [2][128]: second row half's partial votes
constexpr int C_TAG = 6528;     // int [NSTAGE]: index of the tile most recently loaded into each stage

struct WVP {
  int L, R, Wq, row_tiles, jobs, g, ngroups;
  float c;               // log2(e) / sqrt(D)
  float *votes;          // [units, L]
  int atomic_votes;      // several row tiles add into the same votes
  float2 *part;          // [jobs][g][128] per-CTA row statistics (g > 1)
  int *arrive;           // [jobs] arrival counters (zeroed before launch)
  uint32_t *status;
  unsigned long long timeout;
};

struct Job {
  int u, rho0, nrows, rpad, t0, t1, pmin, kend;
};

__device__ __forceinline__ Job job_geo(const WVP &p, int j, int xg) {
  Job J;
  J.u = j / p.row_tiles;
  const int rt = j - J.u * p.row_tiles;
  J.rho0 = rt * TILE;
  J.nrows = min(TILE, p.R - J.rho0);
  J.rpad = (J.nrows + 15) & ~15;
  const int r0 = J.rho0 % p.Wq;
  const bool wraps = (r0 + J.nrows) > p.Wq;
  const int rmax = wraps ? p.Wq - 1 : r0 + J.nrows - 1;
  const int rmin = wraps ? 0 : r0;
  J.kend = p.L - p.Wq + rmax + 1;
  J.pmin = p.L - p.Wq + rmin;
  const int nkt = (J.kend + TILE - 1) / TILE;
  J.t0 = (int)(((long long)xg * nkt) / p.g);
  J.t1 = (int)(((long long)(xg + 1) * nkt) / p.g);
  return J;
}

// Bounded wait until the producer has tagged a ring stage with tile `want`.
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

// (M, Z) <- the statistics of the union of two key sets, Z relative to max M (log2 domain)
__device__ __forceinline__ void merge_stat(float &M, float &Z, float2 o) {
  const float Mn = fmaxf(M, o.x);
  if (Mn != -INFINITY) Z = Z * ex2(M - Mn) + o.y * ex2(o.x - Mn);
  M = Mn;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of 64 values: eight independent chains of three-input max, then a short tree
// (a single chain would expose the max latency 32 times).
__device__ __forceinline__ float max64(const float *s) {
  float m[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = fmax3(s[j], s[j + 8], s[j + 16]);
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = fmax3(m[j], s[j + 24], s[j + 32]);
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = fmax3(m[j], s[j + 40], s[j + 48]);
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], s[j + 56]);
  return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// Adds exp2(s[i] * c + off[i]) for i < N (N a multiple of 8) into four packed fp32x2
// accumulators (independent chains).  off is 16-byte aligned.
template <int N>
__device__ __forceinline__ void exp2_sum(const float *s, const float *off, unsigned long long cc,
                                         unsigned long long (&a)[4]) {
#pragma unroll
  for (int c = 0; c < N; c += 8) {
    const float4 o0 = *reinterpret_cast<const float4 *>(off + c);
    const float4 o1 = *reinterpret_cast<const float4 *>(off + c + 4);
    const float2 x0 = upk(fma2(pk(s[c], s[c + 1]), cc, pk(o0.x, o0.y)));
    const float2 x1 = upk(fma2(pk(s[c + 2], s[c + 3]), cc, pk(o0.z, o0.w)));
    const float2 x2 = upk(fma2(pk(s[c + 4], s[c + 5]), cc, pk(o1.x, o1.y)));
    const float2 x3 = upk(fma2(pk(s[c + 6], s[c + 7]), cc, pk(o1.z, o1.w)));
    a[0] = add2(a[0], pk(ex2(x0.x), ex2(x0.y)));
    a[1] = add2(a[1], pk(ex2(x1.x), ex2(x1.y)));
    a[2] = add2(a[2], pk(ex2(x2.x), ex2(x2.y)));
    a[3] = add2(a[3], pk(ex2(x3.x), ex2(x3.y)));
  }
}

// The sum of the four packed accumulators.
__device__ __forceinline__ float sum4(const unsigned long long (&a)[4]) {
  const float2 t = upk(add2(add2(a[0], a[1]), add2(a[2], a[3])));
  return t.x + t.y;
}

// Pass 2 over w rows (w = 32, 16 or 8) of one key off the causal diagonal:
// exp2(s * c + noff) with noff = -(row max + log2 normaliser), -inf for padding rows.
__device__ __forceinline__ void vote_full(const float *s, const float *noff, unsigned long long cc,
                                          int w, unsigned long long (&a)[4]) {
  if (w == 32) exp2_sum<32>(s, noff, cc, a);
  else if (w == 16) exp2_sum<16>(s, noff, cc, a);
  else exp2_sum<8>(s, noff, cc, a);
}
// The same for a key on the causal diagonal: rows whose position precedes the key add 0.
template <int W>
__device__ __forceinline__ float vote_masked(const float *s, const float *noff, const int *rowpos,
                                             float c, int key, int w) {
  float v = 0.f;
#pragma unroll
  for (int i = 0; i < W; ++i) {
    if (i < w) {
      const float e = ex2(fmaf(s[i], c, noff[i]));
      v += (key <= rowpos[i]) ? e : 0.f;
    }
  }
  return v;
}

// Order of the tile events of one round: first LEAD pass-1 tiles of the new job (A),
// then alternate pass-2 tiles of the previous job (B) and pass-1 tiles.
__device__ __forceinline__ bool next_is_a(int ia, int ib, int na, int nb) {
  if (ia >= na) return false;
  if (ib >= nb) return true;
  return ia < LEAD || (ia - LEAD) < ib;
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    window_vote_kernel(const __grid_constant__ CUtensorMap tq,
                       const __grid_constant__ CUtensorMap tk, const WVP p) {
  using G = Geo<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + G::OFF_Q, sK = sb + G::OFF_K, ctl = sb + G::OFF_CTRL;
  uint8_t *ctrl = smem + G::OFF_CTRL;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctrl + C_TMEM);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl + C_ABORT);
  float2 *xstat = reinterpret_cast<float2 *>(ctrl + C_XSTAT);
  float *noff = reinterpret_cast<float *>(ctrl + C_OFF);  // -(row max + log2 normaliser)
  int *rowpos = reinterpret_cast<int *>(ctrl + C_ROWPOS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{abort_flag, p.status, p.timeout};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NQ; ++i) {
      mbar_init(ctl + C_QFULL + 8 * i, 1);
      mbar_init(ctl + C_QEMPTY + 8 * i, 2);  // both passes release the Q tile
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(ctl + C_XFULL + 8 * i, 4);
      mbar_init(ctl + C_XEMPTY + 8 * i, 4);
    }
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(ctl + C_KFULL + 8 * s, 1);
      mbar_init(ctl + C_KEMPTY + 8 * s, 1);
      reinterpret_cast<volatile int *>(ctrl + C_TAG)[s] = -1;
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(ctl + C_SFULL + 8 * b, 1);
      mbar_init(ctl + C_SEMPTY + 8 * b, 8);  // the 8 warps of the pass
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
  // (No early griddepcontrol.launch_dependents here: an early trigger, which lets the
  // selection grid launch and wait behind this persistent grid, measured 3-7% slower.)

  const int gamma = blockIdx.x / p.g, xg = blockIdx.x - gamma * p.g;
  // Round k gives the groups jobs k*ngroups .. k*ngroups + ngroups - 1, in group order on
  // even rounds and reversed on odd ones: when the row tiles of a unit differ in size (the
  // causal prefill of H2O), a group's jobs then mix small and large tiles instead of
  // repeating the same few row-tile sizes.  CTAs past the last whole group (when g does
  // not divide the grid) have no jobs.
  // With several row tiles per unit and at least 8 units per group, a group takes whole
  // units instead (units gamma, gamma + ngroups, ..., each unit's row tiles in order): a
  // unit's keys are then re-read by one group while they are still in L2, and every
  // group gets the same mix of row-tile sizes.
  const int units = p.jobs / p.row_tiles;
  const bool unit_major = p.row_tiles > 1 && units >= 8 * p.ngroups;
  const int full_rounds = p.jobs / p.ngroups, rem = p.jobs - full_rounds * p.ngroups;
  const int njobs = gamma >= p.ngroups ? 0
                    : unit_major ? ((units - gamma + p.ngroups - 1) / p.ngroups) * p.row_tiles
                    : full_rounds + ((full_rounds & 1) ? (p.ngroups - 1 - gamma < rem) : (gamma < rem));
  auto job_of = [&](int kk) {
    if (unit_major) return (gamma + (kk / p.row_tiles) * p.ngroups) * p.row_tiles + kk % p.row_tiles;
    return kk * p.ngroups + ((kk & 1) ? p.ngroups - 1 - gamma : gamma);
  };

  volatile int *tag = reinterpret_cast<volatile int *>(ctrl + C_TAG);
  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      int kit = 0, qcnt[NQ] = {};
      const uint64_t pol_keep = l2_policy_evict_last(), pol_drop = l2_policy_evict_first();
      bool ok = true;
      for (int k = 0; k < njobs + LAG && ok; ++k) {
        Job Ja{}, Jb{};
        int na = 0, nb = 0;
        if (k < njobs) {
          Ja = job_geo(p, job_of(k), xg);
          na = Ja.t1 - Ja.t0;
        }
        if (k >= LAG) {
          Jb = job_geo(p, job_of(k - LAG), xg);
          nb = Jb.t1 - Jb.t0;
        }
        if (na > 0) {  // Q tile of job k into buffer k % NQ
          const int qb = k % NQ;
          if (!ab.wait(ctl + C_QEMPTY + 8 * qb, (qcnt[qb] & 1) ^ 1)) { ok = false; break; }
          mbar_arrive_expect_tx(ctl + C_QFULL + 8 * qb, G::TILE_BYTES);
          for (int kb = 0; kb < G::KB; ++kb)
            tma_load_2d(sQ + qb * G::TILE_BYTES + kb * G::KBLK, &tq, kb * 64,
                        Ja.u * p.R + Ja.rho0, ctl + C_QFULL + 8 * qb);
          ++qcnt[qb];
        }
        for (int ia = 0, ib = 0; ia < na || ib < nb;) {
          int row;
          const bool is_a = next_is_a(ia, ib, na, nb);
          if (is_a) {
            row = Ja.u * p.L + (Ja.t0 + ia) * TILE;
            ++ia;
          } else {
            row = Jb.u * p.L + (Jb.t1 - 1 - ib) * TILE;
            ++ib;
          }
          const int s = kit % NSTAGE, use = kit / NSTAGE;
          if (!ab.wait(ctl + C_KEMPTY + 8 * s, (use & 1) ^ 1)) { ok = false; break; }
          tag[s] = kit;  // this stage's phase now belongs to tile kit
          mbar_arrive_expect_tx(ctl + C_KFULL + 8 * s, G::TILE_BYTES);
          // a pass-1 load is read again by pass 2 (keep it in L2); a pass-2 load is the
          // tile's last use (let it go first)
          for (int kb = 0; kb < G::KB; ++kb)
            tma_load_2d_hint(sK + s * G::TILE_BYTES + kb * G::KBLK, &tk, kb * 64, row,
                             ctl + C_KFULL + 8 * s, is_a ? pol_keep : pol_drop);
          ++kit;
        }
      }
      // drain: every issued copy must have landed before the CTA may exit
      for (int s = 0; s < NSTAGE; ++s) {
        const int cnt = kit / NSTAGE + (s < kit % NSTAGE ? 1 : 0);
        if (cnt > 0) mbar_wait_bounded(ctl + C_KFULL + 8 * s, (cnt - 1) & 1, p.timeout);
      }
      for (int qb = 0; qb < NQ; ++qb)
        if (qcnt[qb] > 0) mbar_wait_bounded(ctl + C_QFULL + 8 * qb, (qcnt[qb] - 1) & 1, p.timeout);
    }
  } else if (warp == 1 || warp == NWARPS - 1) {
    // ---------- MMA issuers: warp 1 for pass-1 tiles, the last warp for pass-2 tiles ----------
    // Both walk the producer's tile order (which gives each tile's ring stage) and issue
    // only their own pass's tiles, so a pass-2 tile held up by the statistics exchange
    // never holds up pass 1.
    if (lane == 0) {
      const bool mine_a = warp == 1;
      int kit = 0, it = 0, last_bar = -1, last_par = 0, qcnt[NQ] = {};
      bool ok = true;
      for (int k = 0; k < njobs + LAG && ok; ++k) {
        Job Ja{}, Jb{};
        int na = 0, nb = 0;
        if (k < njobs) {
          Ja = job_geo(p, job_of(k), xg);
          na = Ja.t1 - Ja.t0;
        }
        if (k >= LAG) {
          Jb = job_geo(p, job_of(k - LAG), xg);
          nb = Jb.t1 - Jb.t0;
        }
        // this issuer's job of the round (pass 1: job k, pass 2: job k - LAG), its Q buffer
        const int nmine = mine_a ? na : nb;
        const int qb = (mine_a ? k : k - LAG + NQ) % NQ;
        if (nmine > 0) {
          if (!ab.wait(ctl + C_QFULL + 8 * qb, qcnt[qb] & 1)) { ok = false; break; }
          ++qcnt[qb];
          tc_fence_after();
        }
        // pass 1 of a job with at most TR_ROWS query rows also uses the transposed product
        // S^T = K . Q^T (keys on TMEM lanes), like pass 2
        const bool tra = mine_a && Ja.rpad <= TR_ROWS;
        const uint32_t idesc = idesc_bf16(128, mine_a ? (tra ? Ja.rpad : TILE) : (Jb.rpad > 0 ? Jb.rpad : 16));
        const uint64_t qd = sdesc_k128(sQ + qb * G::TILE_BYTES);
        for (int ia = 0, ib = 0; ia < na || ib < nb;) {
          const bool isa = next_is_a(ia, ib, na, nb);
          if (isa) ++ia; else ++ib;
          const int s = kit % NSTAGE, kuse = kit / NSTAGE;
          ++kit;
          if (isa != mine_a) continue;
          const int b = (mine_a ? 0 : 2) + (it & 1), use = it >> 1;
          ++it;
          // An issuer may run a whole round ahead of the producer; the stage's parity only
          // identifies the tile once the producer has started loading it.
          if (!wait_tag(tag + s, kit - 1, ab)) { ok = false; break; }
          if (!ab.wait(ctl + C_KFULL + 8 * s, kuse & 1)) { ok = false; break; }
          if (!ab.wait(ctl + C_SEMPTY + 8 * b, (use & 1) ^ 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(b * 128);
          // descriptors of the tile's first 16-wide k-step; later k-steps advance the
          // start address field (bytes / 16) by a constant
          const uint64_t kd = sdesc_k128(sK + s * G::TILE_BYTES);
          const uint64_t ad = (mine_a && !tra) ? qd : kd, bd = (mine_a && !tra) ? kd : qd;
#pragma unroll
          for (int kb = 0; kb < G::KB; ++kb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t o = (uint64_t)((kb * G::KBLK + kk * 32) >> 4);
              umma_bf16(d, ad + o, bd + o, idesc, (kb | kk) != 0);
            }
          }
          umma_commit(ctl + C_KEMPTY + 8 * s);
          umma_commit(ctl + C_SFULL + 8 * b);
          last_bar = b;
          last_par = use & 1;
        }
        if (!ok) break;
        if (nmine > 0) umma_commit(ctl + C_QEMPTY + 8 * qb);  // this pass is done with the Q tile
      }
      // drain: wait for the completion of the last MMA batch issued
      if (last_bar >= 0) mbar_wait_bounded(ctl + C_SFULL + 8 * last_bar, last_par, p.timeout);
    }
  } else if (warp < 10) {
    // --------- pass 1: row statistics (8 warps: TMEM lane quarter x column half) ---------
    // Control flow (loops, named barriers) is identical for every thread of the pass; a
    // failed wait only turns the remaining work off (ok = false).
    const int quarter = warp & 3;
    const int ch = (warp - 2) >> 2;  // which 64 of the tile's 128 key columns
    const int lrow = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    float2 *hstat = reinterpret_cast<float2 *>(ctrl + C_HSTAT);
    int it1 = 0;
    bool ok = true;
    for (int k = 0; k < njobs; ++k) {
      const int j = job_of(k);
      const Job J = job_geo(p, j, xg);
      const int n = J.t1 - J.t0;
      const bool rvalid = lrow < J.nrows;
      const int prow = rvalid ? p.L - p.Wq + (J.rho0 + lrow) % p.Wq : -1;
      float m = -INFINITY, z = 0.f;
      if (J.rpad <= TR_ROWS) {
        // ---- transposed: keys on TMEM lanes, this warp's 16 rows in registers ----
        // Per row a warp-wide max (redux) moves the row's reference only when the max
        // passes it by TR_SLACK, and each lane keeps its own partial normaliser; the
        // lanes and the four key quarters are summed once per job.
        const bool wact = ch * 16 < J.rpad;  // warp-uniform
        const bool padrows = J.nrows < J.rpad;
        float tm[16], tl[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          tm[r] = -INFINITY;
          tl[r] = 0.f;
        }
        for (int i = 0; i < n; ++i, ++it1) {
          const int b = it1 & 1;
          const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_SFULL + 8 * b, (it1 >> 1) & 1));
          ok = got;
          if (!got) continue;
          tc_fence_after();
          if (wact) {
            float s[16];
            tmem_ld16(tmem + lane_base + (uint32_t)(b * 128 + ch * 16), s);
            tmem_wait_ld();
            const int key = (J.t0 + i) * TILE + quarter * 32 + lane;
            if (padrows || key > J.pmin) {  // causal mask inside the window, padding rows
#pragma unroll
              for (int r = 0; r < 16; ++r) {
                const int row = ch * 16 + r;
                const int pr = row < J.nrows ? p.L - p.Wq + (J.rho0 + row) % p.Wq : -1;
                if (key > pr) s[r] = -INFINITY;
              }
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) {
              float mx;
              asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(mx) : "f"(s[r]));
              mx *= p.c;                    // c > 0: the max of the scaled logits
              if (mx > tm[r] + TR_SLACK) {  // warp-uniform
                tl[r] *= ex2(tm[r] - mx);   // ex2(-inf) = 0 for a first reference
                tm[r] = mx;
              }
            }
            const unsigned long long cc = pk(p.c, p.c);
#pragma unroll
            for (int r = 0; r < 16; r += 2) {
              const float o0 = tm[r] == -INFINITY ? -INFINITY : -tm[r];
              const float o1 = tm[r + 1] == -INFINITY ? -INFINITY : -tm[r + 1];
              const float2 x = upk(fma2(pk(s[r], s[r + 1]), cc, pk(o0, o1)));
              const float2 t = upk(add2(pk(tl[r], tl[r + 1]), pk(ex2(x.x), ex2(x.y))));
              tl[r] = t.x;
              tl[r + 1] = t.y;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(ctl + C_SEMPTY + 8 * b);
        }
        float2 *ts = hstat + (k & 1) * TILE;  // [key quarter][32 rows]
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float v = tl[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (wact && lane == r) ts[quarter * 32 + ch * 16 + r] = make_float2(tm[r], v);
        }
        named_bar(2, 256);
        if (ch == 0 && lrow < J.rpad)  // quarter 0's lanes: one row each
#pragma unroll
          for (int q = 0; q < 4; ++q) merge_stat(m, z, ts[q * 32 + lrow]);
      } else {
        const bool warp_active = quarter * 32 < J.nrows;
        for (int i = 0; i < n; ++i, ++it1) {
          const int b = it1 & 1;
          const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_SFULL + 8 * b, (it1 >> 1) & 1));
          ok = got;
          if (!got) continue;
          tc_fence_after();
          if (warp_active) {
            const int kbase = (J.t0 + i) * TILE + ch * 64;
            float s[64];
            tmem_ld32(tmem + lane_base + (uint32_t)(b * 128 + ch * 64), s);
            tmem_ld32(tmem + lane_base + (uint32_t)(b * 128 + ch * 64 + 32), s + 32);
            tmem_wait_ld();
            if (kbase + 63 > prow) {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (kbase + c > prow) s[c] = -INFINITY;
            }
            const float mnew = fmaxf(m, max64(s) * p.c);
            if (mnew != -INFINITY) {
              // exp2(s * c - m) summed in packed fp32x2 pairs, four independent chains
              const unsigned long long cc = pk(p.c, p.c), nm = pk(-mnew, -mnew);
              unsigned long long a[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
              for (int c = 0; c < 64; c += 8) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float2 x = upk(fma2(pk(s[c + 2 * q], s[c + 2 * q + 1]), cc, nm));
                  a[q] = add2(a[q], pk(ex2(x.x), ex2(x.y)));
                }
              }
              z = z * ex2(m - mnew) + sum4(a);
              m = mnew;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(ctl + C_SEMPTY + 8 * b);
        }
        // ---- merge the two column halves ----
        if (ch == 1) hstat[(k & 1) * TILE + lrow] = make_float2(m, z);
        named_bar(2, 256);
        if (ch == 0) {
          const float2 o = hstat[(k & 1) * TILE + lrow];
          const float mn = fmaxf(m, o.x);
          if (mn != -INFINITY) z = z * ex2(m - mn) + o.y * ex2(o.x - mn);
          m = mn;
        }
      }
      // ---- publish this job's row statistics ----
      if (ch == 0) {
        if (p.g == 1) {
          const int xb = k & 1;
          const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_XEMPTY + 8 * xb, ((k >> 1) & 1) ^ 1));
          ok = got;
          if (got) {
            xstat[xb * TILE + lrow] = make_float2(m, z);
            __syncwarp();
            if (lane == 0) mbar_arrive(ctl + C_XFULL + 8 * xb);
          }
        } else {
          // publish this CTA's partial statistics (the barrier orders every thread's
          // store before the one releasing arrival); the consumers combine all g of them
          p.part[((size_t)j * p.g + xg) * TILE + lrow] = make_float2(m, z);
          named_bar(4, 128);
          if (lrow == 0) red_release_gpu(&p.arrive[j], 1);
        }
      }
    }
  } else {
    // ------------- pass 2: votes (8 warps: TMEM lane quarter (keys) x row half) -------------
    const int quarter = warp & 3;
    const int rh = (warp - 10) >> 2;  // which half of the job's query rows
    const int lkey = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int t2 = threadIdx.x - 320;  // 0..255; the first 128 own one row each
    float *vpart = reinterpret_cast<float *>(ctrl + C_VPART);
    volatile int *go = reinterpret_cast<volatile int *>(ctrl + C_GO);
    int it2 = 0;
    bool ok = true;
    for (int k = 0; k < njobs; ++k) {
      const int j = job_of(k);
      const Job J = job_geo(p, j, xg);
      const int n = J.t1 - J.t0;
      // statistics of this job -> per-row offsets in shared memory
      float M = 0.f, Z = 0.f;
      if (p.g == 1) {
        if (rh == 0) {
          const int xb = k & 1;
          const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_XFULL + 8 * xb, (k >> 1) & 1));
          ok = got;
          if (got) {
            const float2 o = xstat[xb * TILE + t2];
            M = o.x;
            Z = o.y;
            __syncwarp();
            if (lane == 0) mbar_arrive(ctl + C_XEMPTY + 8 * xb);
          }
        }
      } else {
        if (t2 == 0) {
          bool fine = ok && !ab.raised();
          if (fine && !spin_count_bounded(&p.arrive[j], p.g, p.status, p.timeout)) {
            ab.raise();
            fine = false;
          }
          *go = fine ? 1 : 0;
        }
        named_bar(3, 256);
        ok = ok && (*go != 0);
        // combine the g partials of each live row: tpr consecutive threads per row, each
        // over a strided share of the CTAs with up to XB loads in flight, then merged by
        // shuffles (a fixed order, so the result is the same on every call)
        const int tpr = J.nrows <= 32 ? 8 : (J.nrows <= 64 ? 4 : 2);  // tpr * rows <= 256
        const int row = t2 / tpr, sub = t2 - row * tpr;
        M = -INFINITY;
        if (row < J.nrows && ok) {
          const float2 *src = p.part + (size_t)j * p.g * TILE + row;
          for (int r = sub; r < p.g; r += XB * tpr) {
            float2 v[XB];
#pragma unroll
            for (int i = 0; i < XB; ++i)
              v[i] = r + i * tpr < p.g ? __ldcg(src + (size_t)(r + i * tpr) * TILE)
                                       : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int i = 0; i < XB; ++i) merge_stat(M, Z, v[i]);
          }
        }
        for (int o = 1; o < tpr; o <<= 1) {
          const float Mo = __shfl_xor_sync(0xffffffffu, M, o), Zo = __shfl_xor_sync(0xffffffffu, Z, o);
          merge_stat(M, Z, make_float2(Mo, Zo));
        }
        if (sub == 0 && row < J.nrows) {
          noff[row] = Z > 0.f ? -(M + lg2(Z)) : -INFINITY;
          rowpos[row] = p.L - p.Wq + (J.rho0 + row) % p.Wq;
        }
        if (t2 >= J.nrows && t2 < TILE) {  // padding rows
          noff[t2] = -INFINITY;
          rowpos[t2] = -1;
        }
      }
      if (p.g == 1 && t2 < TILE) {
        const bool rvalid = t2 < J.nrows;
        noff[t2] = (rvalid && Z > 0.f) ? -(M + lg2(Z)) : -INFINITY;
        rowpos[t2] = rvalid ? p.L - p.Wq + (J.rho0 + t2) % p.Wq : -1;
      }
      named_bar(3, 256);
      const int half = J.rpad >> 1;  // rows per half: a multiple of 8
      const int r_lo = rh * half;
      const unsigned long long cc = pk(p.c, p.c);
      for (int i = 0; i < n; ++i, ++it2) {
        const int b = 2 + (it2 & 1);
        const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_SFULL + 8 * b, (it2 >> 1) & 1));
        ok = got;
        const int key = (J.t1 - 1 - i) * TILE + lkey;
        float v0 = 0.f;
        if (got) {
          tc_fence_after();
          const bool kfull = key <= J.pmin;
          unsigned long long a[4] = {0ull, 0ull, 0ull, 0ull};
          const uint32_t ta = tmem + lane_base + (uint32_t)(b * 128 + r_lo);
          for (int c0 = 0; c0 < half;) {
            const int w = half - c0 >= 32 ? 32 : (half - c0 >= 16 ? 16 : 8);
            const int r0 = r_lo + c0;
            float s[32];
            if (w == 32) tmem_ld32(ta + c0, s);
            else if (w == 16) tmem_ld16(ta + c0, s);
            else tmem_ld8(ta + c0, s);
            tmem_wait_ld();
            if (kfull) vote_full(s, noff + r0, cc, w, a);
            else v0 += vote_masked<32>(s, noff + r0, rowpos + r0, p.c, key, w);
            c0 += w;
          }
          v0 += sum4(a);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(ctl + C_SEMPTY + 8 * b);
        }
        // the two row halves of this key meet in shared memory (one pair barrier per tile)
        const int par = it2 & 1;
        if (rh == 1) vpart[par * TILE + lkey] = v0;
        named_bar(8 + quarter, 64);
        if (rh == 0 && got && key < J.kend) {
          const float v = v0 + vpart[par * TILE + lkey];
          float *dst = p.votes + (size_t)J.u * p.L + key;
          if (p.atomic_votes)
            atomicAdd(dst, v);
          else
            *dst = v;
        }
      }
      named_bar(3, 256);  // everyone done with off/rowpos of this job
    }
  }

  // ---------------------------------- teardown ----------------------------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

bool g_attr_done[2][64];

// Group size g (CTAs per job).  A round (every group on one job) costs about the busiest
// CTA's key tiles plus a fixed statistics exchange worth about four tiles; the pass-2
// re-read comes from L2 only while every CTA's pending tiles fit there, which costs a
// little per tile beyond eight (measured on the 32-layer Mistral-shaped prompt: g = 8
// 590 us vs g = 19 617 us; on the 8-layer L = 131072 prompt: g = 38 2.31 ms vs g = 152
// 2.97 ms).  When g does not divide the grid the CTAs past the last group stay idle.
int choose_group(int min_nkt, int max_nkt, long long jobs, int P) {
  int best = 1;
  double best_cost = 1e300;
  for (int g = 1; g <= P && g <= min_nkt; ++g) {
    const long long ngroups = P / g;
    const int tpc = (max_nkt + g - 1) / g;
    const long long rounds = (jobs + ngroups - 1) / ngroups;
    double cost = (double)rounds * (tpc + (g > 1 ? 4.0 : 0.0));
    if (tpc > 8) cost *= 1.0 + 0.01 * (tpc - 8);
    if (cost < best_cost) {
      best_cost = cost;
      best = g;
    }
  }
  return best;
}

}  // namespace

WindowVotePlan plan_window_vote(int units, int L, int R, int Wq, int num_sms) {
  WindowVotePlan pl;
  if (plan_window_vote_tmem(units, L, R, Wq, num_sms, &pl)) return pl;
  pl.single = 0;
  pl.row_tiles = (R + TILE - 1) / TILE;
  pl.jobs = units * pl.row_tiles;
  pl.min_nkt = 1 << 30;
  pl.max_nkt = 0;
  for (int rt = 0; rt < pl.row_tiles; ++rt) {  // key tiles of each row tile
    const int nrows = (R - rt * TILE) < TILE ? R - rt * TILE : TILE;
    const int r0 = (rt * TILE) % Wq;
    const bool wraps = r0 + nrows > Wq;
    const int rmax = wraps ? Wq - 1 : r0 + nrows - 1;
    const int nkt = (L - Wq + rmax + 1 + TILE - 1) / TILE;
    if (nkt < pl.min_nkt) pl.min_nkt = nkt;
    if (nkt > pl.max_nkt) pl.max_nkt = nkt;
  }
  pl.g = choose_group(pl.min_nkt, pl.max_nkt, pl.jobs, num_sms);
  pl.ngroups = num_sms / pl.g;
  size_t b = 0;
  if (pl.g > 1) {
    b += (size_t)pl.jobs * pl.g * TILE * sizeof(float2);  // part
    b += (size_t)pl.jobs * sizeof(int);                   // arrive
  }
  pl.ws_bytes = (b + 255) & ~(size_t)255;
  return pl;
}

cudaError_t launch_window_vote(const Ctx &c, const WindowVoteArgs &a) {
  const WindowVotePlan pl = plan_window_vote(a.units, a.L, a.R, a.Wq, c.num_sms);
  if (pl.single) return launch_window_vote_tmem(c, a, pl);
  int dev = 0;
  cudaGetDevice(&dev);
  const int di = a.D == 128 ? 1 : 0;
  const void *fn = a.D == 128 ? (const void *)window_vote_kernel<128>
                              : (const void *)window_vote_kernel<64>;
  const int smem = a.D == 128 ? Geo<128>::SMEM : Geo<64>::SMEM;
  if (dev < 64 && !g_attr_done[di][dev]) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    g_attr_done[di][dev] = true;
  }
  CUtensorMap tq, tk;
  if (!encode_rows_map(&tq, a.q, (uint64_t)a.units * a.R, a.D, TILE)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&tk, a.k, (uint64_t)a.units * a.L, a.D, TILE)) return cudaErrorInvalidValue;

  int blocks_per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, fn, NTHREADS, smem);
  if (e != cudaSuccess) return e;
  if (blocks_per_sm != 1) return cudaErrorInvalidConfiguration;
  WVP p;
  p.L = a.L;
  p.R = a.R;
  p.Wq = a.Wq;
  p.row_tiles = pl.row_tiles;
  p.jobs = pl.jobs;
  p.g = pl.g;
  p.ngroups = pl.ngroups;
  p.c = (float)(1.4426950408889634 / sqrt((double)a.D));
  p.votes = a.votes;
  p.atomic_votes = p.row_tiles > 1;
  uint8_t *w = reinterpret_cast<uint8_t *>(a.ws);
  const size_t jobs = (size_t)p.jobs;
  p.part = reinterpret_cast<float2 *>(w);
  p.arrive = reinterpret_cast<int *>(p.part + jobs * p.g * TILE);
  p.status = c.status;
  p.timeout = c.timeout_ns;
  const int P = c.num_sms;  // one persistent CTA per SM

  if (p.g > 1) {
    e = cudaMemsetAsync(p.arrive, 0, jobs * sizeof(int), c.stream);
    if (e != cudaSuccess) return e;
  }
  if (p.atomic_votes) {
    e = cudaMemsetAsync(a.votes, 0, (size_t)a.units * a.L * sizeof(float), c.stream);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.D == 128) return cudaLaunchKernelEx(&cfg, window_vote_kernel<128>, tq, tk, p);
  return cudaLaunchKernelEx(&cfg, window_vote_kernel<64>, tq, tk, p);
}

}  // namespace kvc
