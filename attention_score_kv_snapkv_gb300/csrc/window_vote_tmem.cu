// SnapKV steps 1-2 with one pass over the keys (SnapKV article, 処理の流れ steps 1 and 2):
// every trailing window query of the G query heads of a KV head takes
// softmax(q . k / sqrt(D)) over the keys it may see (all keys up to and including its own
// position), and the probabilities are summed per key into the vote.  With every prompt
// query as a "window" query this is also H2O's initial cumulative score.
//
// Design (sm_103a): each key tile crosses HBM -> shared memory once and meets the
// tensor cores once.
// * A job is (unit u, tile of up to 128 query rows).  Its key range is cut into 128-key
//   tiles, split over a group of g CTAs of a persistent cooperative grid (one CTA per SM).
// * Per key tile, one tcgen05.mma forms S^T = K . Q^T (M = 128 keys on the TMEM lanes,
//   N = the job's rows rounded up to 16, fp32) into one of NB tensor-memory buffers of
//   the CTA (NB = 512 columns / rows per buffer).  The buffer stays allocated until the
//   votes of the tile are formed, so a CTA's share of a job must fit in NB tiles; the
//   launcher picks g accordingly (the two-pass kernel of window_vote.cu serves shapes
//   where no g does).
// * Statistics warps (one per TMEM lane quarter and 32-row chunk): per row a reference
//   ref that moves only when a logit passes it by SLACK (in log2 units; the exact
//   warp-wide maximum is taken only then), p~ = 2^(s.c - ref) written back in place of
//   the logits, per-lane partial sums of p~ accumulated over the CTA's tiles of the job
//   and reduced across the lanes once per job (transpose reduction).  The reference of
//   every tile, quarter and row is recorded.
// * The g CTAs of a job exchange their row statistics (max, normaliser) through global
//   memory (publish, fence, arrival counter; bounded wait) -- or through shared memory
//   when g = 1 -- and the vote warps turn them into lse = max + log2(normaliser).
// * Vote warps (one per lane quarter): vote(key) = sum over rows of p~ . 2^(ref - lse):
//   one FMA per score, no cross-lane reduction; then the buffer is released.
// * Warp roles: warp 0 = TMA producer (Q tiles double-buffered, K tiles in a 4-stage
//   ring, 128-byte swizzle), warp 1 = TMEM owner and MMA issuer, warps 2-17 = statistics,
//   warps 18-21 = votes.  Every wait is bounded (KVC_DEV_TIMEOUT).
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int TILE = 128;        // keys per tile (TMEM lanes); query rows per job at most
constexpr int NSTAGE = 4;        // K tile ring depth
constexpr int NQ = 2;            // Q tile buffers
constexpr int W_P1 = 2;          // first statistics warp

// Warp roles for jobs of at most 32 * NCH rows: statistics warps, one per TMEM lane
// quarter and 32-row chunk; vote warps, one per lane quarter in each of VS sets that
// take alternate tiles (two sets when a tile's votes are short, so that the tensor-
// memory buffers turn over sooner).
template <int NCH>
struct Roles {
  static constexpr int NP1 = 4 * NCH;
  static constexpr int VS = NCH <= 2 ? 2 : 1;
  static constexpr int NP2 = 4 * VS;
  static constexpr int W_P2 = W_P1 + NP1;
  static constexpr int NWARPS = W_P2 + NP2;
  static constexpr int NTHREADS = 32 * NWARPS;
};
constexpr int TMEM_COLS = 512;
constexpr int MAXNB = 32;        // tensor-memory buffers at 16 rows each
constexpr float SLACK = 8.f;     // a row's reference moves only past this (log2 units)
constexpr float NOREF = 3.0e38f; // -ref of a row with no reference yet (finite, so that
                                 // s.c - ref is +huge for a finite logit and -inf for -inf)
// Partial statistics a merging thread loads per batch.  Every CTA of a group reads all
// g partials of a job at the same moment (g x g x rows loads: 147 x 147 x 32 on the
// long-context prompt), so the batch trades the exchange's latency against a burst of L2
// requests that also delays the key stream.  Measured on that prompt (8 layers, g = 147,
// 32 rows, 4 threads per row): batches of 10 take 1.82 ms, against 1.93 ms with batches
// of 20, 1.85 / 1.84 ms with 8 / 13, 2.07 ms with 5 and about 2.3 ms with all 37 in one
// batch.
constexpr int XB = 10;

// control region byte offsets
constexpr int C_QFULL = 0;       // [NQ]
constexpr int C_QEMPTY = 16;     // [NQ]
constexpr int C_KFULL = 32;      // [NSTAGE]
constexpr int C_KEMPTY = 64;     // [NSTAGE]
constexpr int C_XFULL = 96;      // [2] local statistics hand-off (g == 1)
constexpr int C_XEMPTY = 112;    // [2]
constexpr int C_SFULL = 128;     // [MAXNB] MMA done
constexpr int C_PDONE = 384;     // [MAXNB] p~ written
constexpr int C_TFREE = 640;     // [MAXNB] votes formed, buffer free
constexpr int C_TMEM = 896;
constexpr int C_ABORT = 900;
constexpr int C_GO = 904;
constexpr int C_TAG = 912;       // int [NSTAGE]
constexpr int C_XSTAT = 1024;    // float2 [2][128]
constexpr int C_STAT = 3072;     // float2 [2][4][128] per-quarter row statistics of a job
constexpr int C_REFCUR = 11264;  // float [4][128]: -ref of each (quarter, row), current job
constexpr int C_REFREC = 13312;  // float [512][4]... [b][quarter][QR]: -ref of every tile
constexpr int C_LSE = 21504;     // float [2][128]
constexpr int C_F = 22528;       // float [8][128] per vote warp: weights 2^(ref - lse)
constexpr int C_ROWPOS = 26624;  // int [16][32] prompt position of each statistics warp's rows
constexpr int C_END = 28672;

template <int D>
struct Geo {
  static constexpr int KB = D / 64;           // 128-byte k-blocks per row
  static constexpr int KBLK = TILE * 128;     // bytes of one k-block of a key tile
  static constexpr int TILE_BYTES = KB * KBLK;
  static constexpr int QBUF = TILE_BYTES;     // a Q buffer holds up to 128 rows
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = NQ * QBUF;
  static constexpr int OFF_CTRL = OFF_K + NSTAGE * TILE_BYTES;
  static constexpr int NEED = OFF_CTRL + C_END + 1024;  // + base alignment slack
  // At least 116 KB so that two CTAs never share an SM (each allocates all 512 TMEM
  // columns, and the persistent grid relies on one resident CTA per SM).
  static constexpr int SMEM = NEED > 116 * 1024 ? NEED : 116 * 1024;
};

struct WVP1 {
  int L, R, Wq, row_tiles, jobs, g, ngroups;
  int qr;                // rows per Q tile and per tensor-memory buffer (multiple of 16)
  int nb;                // tensor-memory buffers (512 / qr)
  float c;               // log2(e) / sqrt(D)
  float *votes;          // [units, L]
  int atomic_votes;      // several row tiles add into the same votes
  float2 *part;          // [jobs][g][qr] per-CTA row statistics (g > 1)
  int *arrive;           // [jobs] arrival counters (zeroed before launch)
  uint32_t *status;
  unsigned long long timeout;
};

struct Job {
  int u, rho0, r0, nrows, rpad, t0, t1, pmin, kend;  // r0 = rho0 % Wq: first row's window row
  bool wraps;            // the tile's rows span the ends of two query heads' windows
};

__device__ __forceinline__ Job job_geo(const WVP1 &p, int j, int xg) {
  Job J;
  J.u = j / p.row_tiles;
  const int rt = j - J.u * p.row_tiles;
  J.rho0 = rt * TILE;
  J.nrows = min(TILE, p.R - J.rho0);
  J.rpad = (J.nrows + 15) & ~15;
  J.r0 = J.rho0 % p.Wq;
  J.wraps = (J.r0 + J.nrows) > p.Wq;
  const int rmax = J.wraps ? p.Wq - 1 : J.r0 + J.nrows - 1;
  const int rmin = J.wraps ? 0 : J.r0;
  J.kend = p.L - p.Wq + rmax + 1;
  J.pmin = p.L - p.Wq + rmin;
  const int nkt = (J.kend + TILE - 1) / TILE;
  J.t0 = (int)(((long long)xg * nkt) / p.g);
  J.t1 = (int)(((long long)(xg + 1) * nkt) / p.g);
  return J;
}

// Prompt position of row `row` of a job (-1 for a padding row, so every key is masked).
__device__ __forceinline__ int row_pos(const WVP1 &p, const Job &J, int row) {
  if (row >= J.nrows) return -1;
  return p.L - p.Wq + (J.wraps ? (J.rho0 + row) % p.Wq : J.r0 + row);
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

__device__ __forceinline__ float redux_max(float x) {
  float m;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(x));
  return m;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Sum over the warp's 32 lanes of each of x[0..W-1] (W = 32 or 16); afterwards lane l
// holds the sum of x[l % W].  Levels at or above W add the partner lane's values; the
// levels below keep half of the values and add the partner's other half.
template <int W>
__device__ __forceinline__ float transpose_sum(float (&x)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= W; o >>= 1) {
#pragma unroll
    for (int i = 0; i < W; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], o);
  }
#pragma unroll
  for (int o = W / 2; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? x[i] : x[i + o];
      const float keep = up ? x[i + o] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return x[0];
}

// Causal mask inside the window (and padding rows): logits of keys after a row's
// position become -inf.  rp: the rows' positions (shared memory, this warp's own).
template <int W>
__device__ __forceinline__ void mask_rows(float (&v)[32], const int *rp, int key) {
#pragma unroll
  for (int r = 0; r < W; r += 4) {
    const int4 p4 = *reinterpret_cast<const int4 *>(rp + r);
    if (key > p4.x) v[r] = -INFINITY;
    if (key > p4.y) v[r + 1] = -INFINITY;
    if (key > p4.z) v[r + 2] = -INFINITY;
    if (key > p4.w) v[r + 3] = -INFINITY;
  }
}

// One statistics step on W (32 or 16) rows of one key tile for this lane's key: mask,
// p~ = 2^(s.c - ref) with lazily moved references, partial sums, p~ back to TMEM.
// nref: -ref of the chunk's rows (shared memory, this warp's own); c = log2(e)/sqrt(D).
template <int W>
__device__ __forceinline__ void stats_chunk(float c, uint32_t taddr, int key, bool masked,
                                            const int *rp, float *nref, float (&acc)[32],
                                            int lane) {
  float v[32];
  if (W == 32) tmem_ld32(taddr, v);
  else tmem_ld16(taddr, v);
  tmem_wait_ld();
  if (masked) mask_rows<W>(v, rp, key);
  // x = s.c - ref, and whether any lane passes its row's reference by more than SLACK
  float lm = -INFINITY;
#pragma unroll
  for (int r = 0; r < W; r += 4) {
    const float4 n4 = *reinterpret_cast<const float4 *>(nref + r);
    v[r] = fmaf(v[r], c, n4.x);
    v[r + 1] = fmaf(v[r + 1], c, n4.y);
    v[r + 2] = fmaf(v[r + 2], c, n4.z);
    v[r + 3] = fmaf(v[r + 3], c, n4.w);
    lm = fmax3(lm, fmaxf(v[r], v[r + 1]), fmaxf(v[r + 2], v[r + 3]));
  }
  if (__any_sync(0xffffffffu, lm > SLACK)) {
    // move the references of the rows whose maximum passed them (warp-uniform per row)
    if (W == 32) tmem_ld32(taddr, v);
    else tmem_ld16(taddr, v);
    tmem_wait_ld();
    if (masked) mask_rows<W>(v, rp, key);
#pragma unroll
    for (int r = 0; r < W; ++r) {
      const float mx = redux_max(v[r]) * c;    // c > 0
      const float nr = nref[r];
      const float old = nr >= NOREF ? -INFINITY : -nr;
      float nn = nr;
      if (mx > old + SLACK) {                  // warp-uniform
        acc[r] *= ex2(old - mx);               // 0 when there was no reference
        nn = -mx;
      }
      v[r] = fmaf(v[r], c, nn);
      __syncwarp();
      if (lane == 0) nref[r] = nn;
    }
    __syncwarp();
  }
#pragma unroll
  for (int r = 0; r < W; r += 2) {
    const float2 e = make_float2(ex2(v[r]), ex2(v[r + 1]));
    v[r] = e.x;
    v[r + 1] = e.y;
    const float2 t = upk(add2(pk(acc[r], acc[r + 1]), pk(e.x, e.y)));
    acc[r] = t.x;
    acc[r + 1] = t.y;
  }
  if (W == 32) tmem_st32(taddr, v);
  else tmem_st16(taddr, v);
}

// One CTA per SM.  The register file is split over the SM's four sub-partitions: with
// 22 warps (NCH = 4) six sit on two of them, so at most 80 registers a thread (the few
// spills sit in the once-per-job transpose reduction).
template <int D, int NCH>
__global__ void __launch_bounds__(Roles<NCH>::NTHREADS, 1)
    window_vote_tmem_kernel(const __grid_constant__ CUtensorMap tq,
                            const __grid_constant__ CUtensorMap tk, const WVP1 p) {
  using G = Geo<D>;
  constexpr int NP1 = Roles<NCH>::NP1, NP2 = Roles<NCH>::NP2, VS = Roles<NCH>::VS;
  constexpr int W_P2 = Roles<NCH>::W_P2, NTHREADS = Roles<NCH>::NTHREADS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t sQ = sb + G::OFF_Q, sK = sb + G::OFF_K, ctl = sb + G::OFF_CTRL;
  uint8_t *ctrl = smem + G::OFF_CTRL;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(ctrl + C_TMEM);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ctrl + C_ABORT);
  float2 *xstat = reinterpret_cast<float2 *>(ctrl + C_XSTAT);
  float2 *stat = reinterpret_cast<float2 *>(ctrl + C_STAT);
  float *refcur = reinterpret_cast<float *>(ctrl + C_REFCUR);
  float *refrec = reinterpret_cast<float *>(ctrl + C_REFREC);
  float *lse = reinterpret_cast<float *>(ctrl + C_LSE);
  volatile int *tag = reinterpret_cast<volatile int *>(ctrl + C_TAG);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{abort_flag, p.status, p.timeout};
  const int QR = p.qr, NB = p.nb;
  const int QKBLK = QR * 128;     // bytes of one k-block of a Q tile
  const int qbytes = G::KB * QKBLK;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NQ; ++i) {
      mbar_init(ctl + C_QFULL + 8 * i, 1);
      mbar_init(ctl + C_QEMPTY + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(ctl + C_XFULL + 8 * i, 4);
      mbar_init(ctl + C_XEMPTY + 8 * i, NP2);
    }
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(ctl + C_KFULL + 8 * s, 1);
      mbar_init(ctl + C_KEMPTY + 8 * s, 1);
      tag[s] = -1;
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(ctl + C_SFULL + 8 * b, 1);
      mbar_init(ctl + C_PDONE + 8 * b, NP1);
      mbar_init(ctl + C_TFREE + 8 * b, 4);  // the vote set that takes the tile
    }
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 4 * TILE; i += NTHREADS) refcur[i] = NOREF;
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

  // Round k gives the groups jobs k*ngroups .. k*ngroups + ngroups - 1, in group order on
  // even rounds and reversed on odd ones (row tiles of different sizes mix); CTAs past
  // the last whole group have no jobs.
  const int gamma = blockIdx.x / p.g, xg = blockIdx.x - gamma * p.g;
  const int full_rounds = p.jobs / p.ngroups, rem = p.jobs - full_rounds * p.ngroups;
  const int njobs = gamma >= p.ngroups ? 0
                    : full_rounds + ((full_rounds & 1) ? (p.ngroups - 1 - gamma < rem) : (gamma < rem));
  auto job_of = [&](int kk) {
    return kk * p.ngroups + ((kk & 1) ? p.ngroups - 1 - gamma : gamma);
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      int kit = 0, qcnt[NQ] = {};
      const uint64_t pol_once = l2_policy_evict_first();
      bool ok = true;
      for (int k = 0; k < njobs && ok; ++k) {
        const Job J = job_geo(p, job_of(k), xg);
        const int n = J.t1 - J.t0;
        if (n <= 0) continue;
        const int qb = k % NQ;
        if (!ab.wait(ctl + C_QEMPTY + 8 * qb, (qcnt[qb] & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(ctl + C_QFULL + 8 * qb, qbytes);
        for (int kb = 0; kb < G::KB; ++kb)
          tma_load_2d(sQ + qb * G::QBUF + kb * QKBLK, &tq, kb * 64, J.u * p.R + J.rho0,
                      ctl + C_QFULL + 8 * qb);
        ++qcnt[qb];
        for (int i = 0; i < n; ++i) {
          const int s = kit % NSTAGE, use = kit / NSTAGE;
          if (!ab.wait(ctl + C_KEMPTY + 8 * s, (use & 1) ^ 1)) { ok = false; break; }
          tag[s] = kit;  // this stage's phase now belongs to tile kit
          mbar_arrive_expect_tx(ctl + C_KFULL + 8 * s, G::TILE_BYTES);
          for (int kb = 0; kb < G::KB; ++kb)
            tma_load_2d_hint(sK + s * G::TILE_BYTES + kb * G::KBLK, &tk, kb * 64,
                             J.u * p.L + (J.t0 + i) * TILE, ctl + C_KFULL + 8 * s, pol_once);
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
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      int kit = 0, last_bar = -1, last_par = 0, qcnt[NQ] = {};
      int b = 0, bph = 0;  // the tile's buffer and its use parity (no division per tile)
      bool ok = true;
      for (int k = 0; k < njobs && ok; ++k) {
        const Job J = job_geo(p, job_of(k), xg);
        const int n = J.t1 - J.t0;
        if (n <= 0) continue;
        const int qb = k % NQ;
        if (!ab.wait(ctl + C_QFULL + 8 * qb, qcnt[qb] & 1)) { ok = false; break; }
        ++qcnt[qb];
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, J.rpad);
        const uint64_t qd = sdesc_k128(sQ + qb * G::QBUF);
        for (int i = 0; i < n; ++i) {
          const int s = kit % NSTAGE, kuse = kit / NSTAGE;
          ++kit;
          // the stage's parity identifies the tile only once the producer has started it
          if (!wait_tag(tag + s, kit - 1, ab)) { ok = false; break; }
          if (!ab.wait(ctl + C_KFULL + 8 * s, kuse & 1)) { ok = false; break; }
          if (!ab.wait(ctl + C_TFREE + 8 * b, bph ^ 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(b * QR);
          const uint64_t kd = sdesc_k128(sK + s * G::TILE_BYTES);
#pragma unroll
          for (int kb = 0; kb < G::KB; ++kb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ko = (uint64_t)((kb * G::KBLK + kk * 32) >> 4);
              const uint64_t qo = (uint64_t)((kb * QKBLK + kk * 32) >> 4);
              umma_bf16(d, kd + ko, qd + qo, idesc, (kb | kk) != 0);
            }
          }
          umma_commit(ctl + C_KEMPTY + 8 * s);
          umma_commit(ctl + C_SFULL + 8 * b);
          last_bar = b;
          last_par = bph;
          if (++b == NB) {
            b = 0;
            bph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(ctl + C_QEMPTY + 8 * qb);  // done with the Q tile
      }
      if (last_bar >= 0) mbar_wait_bounded(ctl + C_SFULL + 8 * last_bar, last_par, p.timeout);
    }
  } else if (warp < W_P2) {
    // --------- statistics: warp = (TMEM lane quarter, chunk of 32 rows) ---------
    // Control flow (loops, named barriers, barrier arrivals) is the same for every
    // statistics warp; a failed wait only turns the remaining work off.
    const int q = warp & 3;
    const int chunk = (warp - W_P1) >> 2;
    const int row0 = chunk * 32;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float *nref = refcur + q * TILE + row0;  // this warp's rows
    int *rp = reinterpret_cast<int *>(ctrl + C_ROWPOS) + (warp - W_P1) * 32;
    const int t1id = threadIdx.x - 32 * W_P1;  // 0..511
    float acc[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) acc[r] = 0.f;
    int it = 0;
    int sb_b = 0, sb_ph = 0;  // the tile's buffer and its use parity
    bool ok = true;
    for (int k = 0; k < njobs; ++k) {
      const int j = job_of(k);
      const Job J = job_geo(p, j, xg);
      const int n = J.t1 - J.t0;
      const int w = J.rpad - row0;           // rows of this chunk in the job (warp-uniform)
      const bool active = w > 0;
      rp[lane] = row_pos(p, J, row0 + lane);  // read only by this warp
      __syncwarp();
      for (int i = 0; i < n; ++i, ++it) {
        const int b = sb_b;
        const int bph = sb_ph;
        if (++sb_b == NB) {
          sb_b = 0;
          sb_ph ^= 1;
        }
        const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_SFULL + 8 * b, bph));
        ok = got;
        if (!got) continue;
        tc_fence_after();
        if (active) {
          const int kt = J.t0 + i;
          const int key = kt * TILE + q * 32 + lane;
          const bool masked = (kt * TILE + q * 32 + 31 > J.pmin) || (J.nrows < J.rpad);
          const uint32_t ta = tmem + lane_base + (uint32_t)(b * QR + row0);
          if (w >= 32) stats_chunk<32>(p.c, ta, key, masked, rp, nref, acc, lane);
          else stats_chunk<16>(p.c, ta, key, masked, rp, nref, acc, lane);
          // record this tile's references for the vote warps
          if (lane < (w >= 32 ? 32 : 16)) refrec[(b * 4 + q) * QR + row0 + lane] = nref[lane];
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ctl + C_PDONE + 8 * b);
      }
      // ---- this CTA's row statistics of the job ----
      float2 *st = stat + (k & 1) * 4 * TILE;
      if (active) {
        const float z = w >= 32 ? transpose_sum<32>(acc, lane) : transpose_sum<16>(acc, lane);
        if (lane < (w >= 32 ? 32 : 16)) {
          const float nr = nref[lane];
          st[q * TILE + row0 + lane] = make_float2(nr >= NOREF ? -INFINITY : -nr, z);
        }
        __syncwarp();
        if (lane < 32) nref[lane] = NOREF;   // fresh references for the next job
#pragma unroll
        for (int r = 0; r < 32; ++r) acc[r] = 0.f;
      }
      named_bar(1, 32 * NP1);
      if (t1id < TILE) {
        const int row = t1id;
        float M = -INFINITY, Z = 0.f;
        if (row < J.rpad) {
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) merge_stat(M, Z, st[qq * TILE + row]);
        }
        if (p.g == 1) {
          const int xb = k & 1;
          const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_XEMPTY + 8 * xb, ((k >> 1) & 1) ^ 1));
          ok = got;
          if (got) {
            xstat[xb * TILE + row] = make_float2(M, Z);
            __syncwarp();
            if (lane == 0) mbar_arrive(ctl + C_XFULL + 8 * xb);
          }
        } else {
          // publish this CTA's partial statistics (the barrier orders every thread's
          // store before the one releasing arrival); every CTA of the group combines all g
          if (row < QR) p.part[((size_t)j * p.g + xg) * QR + row] = make_float2(M, Z);
          named_bar(3, TILE);
          if (row == 0) red_release_gpu(&p.arrive[j], 1);
        }
      }
    }
  } else {
    // ------------- votes: one warp per TMEM lane quarter and set, every row -------------
    const int q = warp & 3;
    const int vset = (warp - W_P2) >> 2;     // this warp's set takes tiles it % VS == vset
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int t2 = threadIdx.x - 32 * W_P2;  // 0 .. 32 * NP2 - 1
    float *fw = reinterpret_cast<float *>(ctrl + C_F) + (warp - W_P2) * TILE;
    volatile int *go = reinterpret_cast<volatile int *>(ctrl + C_GO);
    int it = 0;
    int vb_b = 0, vb_ph = 0;  // the tile's buffer and its use parity
    bool ok = true;
    for (int k = 0; k < njobs; ++k) {
      const int j = job_of(k);
      const Job J = job_geo(p, j, xg);
      const int n = J.t1 - J.t0;
      float *ls = lse + (k & 1) * TILE;
      // ---- the job's row statistics -> lse per row ----
      float M = -INFINITY, Z = 0.f;
      if (p.g == 1) {
        const int xb = k & 1;
        const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_XFULL + 8 * xb, (k >> 1) & 1));
        ok = got;
        if (got) {
          const float2 o = xstat[xb * TILE + (t2 & (TILE - 1))];
          M = o.x;
          Z = o.y;
          __syncwarp();
          if (lane == 0) mbar_arrive(ctl + C_XEMPTY + 8 * xb);
        }
        if (t2 < TILE) ls[t2] = (t2 < J.nrows && Z > 0.f) ? M + lg2(Z) : -INFINITY;
      } else {
        if (t2 == 0) {
          bool fine = ok && !ab.raised();
          if (fine && !spin_count_bounded(&p.arrive[j], p.g, p.status, p.timeout)) {
            ab.raise();
            fine = false;
          }
          *go = fine ? 1 : 0;
        }
        named_bar(2, 32 * NP2);
        ok = ok && (*go != 0);
        // tpr consecutive threads per row, each over a strided share of the g CTAs with
        // up to XB loads in flight, merged by shuffles in a fixed order
        const int tpr = J.rpad <= 16 ? 8 : (J.rpad <= 32 ? 4 : (J.rpad <= 64 ? 2 : 1));
        const int row = (t2 & (TILE - 1)) / tpr, sub = (t2 & (TILE - 1)) - row * tpr;
        if (row < J.nrows && ok && t2 < TILE) {
          const float2 *src = p.part + (size_t)j * p.g * QR + row;
          for (int r = sub; r < p.g; r += XB * tpr) {
            float2 v[XB];
#pragma unroll
            for (int i = 0; i < XB; ++i)
              v[i] = r + i * tpr < p.g ? __ldcg(src + (size_t)(r + i * tpr) * QR)
                                       : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int i = 0; i < XB; ++i) merge_stat(M, Z, v[i]);
          }
        }
        for (int o = 1; o < tpr; o <<= 1) {
          const float Mo = __shfl_xor_sync(0xffffffffu, M, o), Zo = __shfl_xor_sync(0xffffffffu, Z, o);
          merge_stat(M, Z, make_float2(Mo, Zo));
        }
        if (t2 < TILE) {
          if (sub == 0) ls[row] = (row < J.nrows && Z > 0.f) ? M + lg2(Z) : -INFINITY;
          if (tpr > 1 && t2 >= J.rpad) ls[t2] = -INFINITY;
        }
      }
      named_bar(2, 32 * NP2);
      for (int i = 0; i < n; ++i, ++it) {
        const int b = vb_b;
        const int bph = vb_ph;
        if (++vb_b == NB) {
          vb_b = 0;
          vb_ph ^= 1;
        }
        if (VS > 1 && (it & (VS - 1)) != vset) continue;  // the other set's tile
        const bool got = __all_sync(0xffffffffu, ok && ab.wait(ctl + C_PDONE + 8 * b, bph));
        ok = got;
        const int kt = J.t0 + i;
        const int key = kt * TILE + q * 32 + lane;
        float vote = 0.f;
        if (got) {
          tc_fence_after();
          // weights 2^(ref - lse) of this quarter's rows for this tile
          const float *rr = refrec + (b * 4 + q) * QR;
          for (int row = lane; row < J.rpad; row += 32) {
            const float l = ls[row], nr = rr[row];
            fw[row] = (l == -INFINITY || nr >= NOREF) ? 0.f : ex2(-nr - l);
          }
          __syncwarp();
          unsigned long long a2[2] = {0ull, 0ull};
          const uint32_t ta = tmem + lane_base + (uint32_t)(b * QR);
          // p~ . weight over the rows, 32-row chunks (16 for a ragged last chunk); with at
          // most two chunks both loads are in flight before the wait
          auto fma_chunk = [&](const float (&sv)[32], int c0, int wc) {
#pragma unroll
            for (int r = 0; r < 32; r += 4) {
              if (r < wc) {
                const float4 f4 = *reinterpret_cast<const float4 *>(fw + c0 + r);
                ffma2(a2[0], pk(sv[r], sv[r + 1]), pk(f4.x, f4.y));
                ffma2(a2[1], pk(sv[r + 2], sv[r + 3]), pk(f4.z, f4.w));
              }
            }
          };
          if (NCH <= 2) {
            float s0[32], s1[32];
            const int w0 = J.rpad >= 32 ? 32 : 16, w1 = J.rpad - 32;  // warp-uniform
            if (w0 == 32) tmem_ld32(ta, s0);
            else tmem_ld16(ta, s0);
            if (w1 >= 32) tmem_ld32(ta + 32, s1);
            else if (w1 > 0) tmem_ld16(ta + 32, s1);
            tmem_wait_ld();
            fma_chunk(s0, 0, w0);
            if (w1 > 0) fma_chunk(s1, 32, w1 >= 32 ? 32 : 16);
          } else {
            for (int c0 = 0; c0 < J.rpad; c0 += 32) {
              float sv[32];
              const bool full = J.rpad - c0 >= 32;  // warp-uniform
              if (full) tmem_ld32(ta + c0, sv);
              else tmem_ld16(ta + c0, sv);
              tmem_wait_ld();
              fma_chunk(sv, c0, full ? 32 : 16);
            }
          }
          const float2 t = upk(add2(a2[0], a2[1]));
          vote = t.x + t.y;
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(ctl + C_TFREE + 8 * b);
        }
        if (got && key < J.kend) {
          float *dst = p.votes + (size_t)J.u * p.L + key;
          if (p.atomic_votes)
            atomicAdd(dst, vote);
          else
            *dst = vote;
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

bool g_attr_done[8][64];

}  // namespace

// Plan of the single-pass kernel, or false where the two-pass kernel serves the shape
// better.  A CTA's share of a job (tpc key tiles) stays in tensor memory until the
// job's row statistics are complete, so the kernel keeps HBM busy only if two jobs fit
// at once (2 tpc <= NB: the next job streams while this one's statistics are exchanged
// and its votes formed) and, when the g CTAs of a job exchange statistics through
// global memory (a few microseconds, straggling CTAs included), a job gives each CTA at
// least MIN_TPC tiles to stream meanwhile.  Measured on GB300: with 128 query rows per
// job (NB = 4) neither holds and the two-pass kernel is faster.  Among the group sizes
// that qualify, a round (every group on one job) costs about the busiest CTA's key
// tiles, plus its Q tile (qr/128 of a key tile) and, when g > 1, the exchange.  Of equal
// costs the smallest g is taken: its CTAs' shares are the most even.  Measured on the
// long-context prompt (1024 key tiles per job, 8 layers): g = 147 (7 tiles on all but 5
// CTAs) 1.82 ms, against 1.99 ms for g = 152 (6 or 7 tiles), 1.96 ms for g = 128 (8
// each, tensor memory full with two jobs) and 2.16 ms for g = 140.
constexpr int MIN_TPC = 4;
bool plan_window_vote_tmem(int units, int L, int R, int Wq, int num_sms, WindowVotePlan *pl) {
  const int row_tiles = (R + TILE - 1) / TILE;
  int min_nkt = 1 << 30, max_nkt = 0;
  for (int rt = 0; rt < row_tiles; ++rt) {
    const int nrows = (R - rt * TILE) < TILE ? R - rt * TILE : TILE;
    const int r0 = (rt * TILE) % Wq;
    const bool wraps = r0 + nrows > Wq;
    const int rmax = wraps ? Wq - 1 : r0 + nrows - 1;
    const int nkt = (L - Wq + rmax + 1 + TILE - 1) / TILE;
    if (nkt < min_nkt) min_nkt = nkt;
    if (nkt > max_nkt) max_nkt = nkt;
  }
  const int qr = R >= TILE ? TILE : ((R + 15) & ~15);
  const int nb = TMEM_COLS / qr;
  const long long jobs = (long long)units * row_tiles;
  int best = 0;
  double best_cost = 1e300;
  for (int g = 1; g <= num_sms; ++g) {
    const int tpc = (max_nkt + g - 1) / g;
    if (2 * tpc > nb || (g > 1 && tpc < MIN_TPC)) continue;
    const long long ngroups = num_sms / g;
    const long long rounds = (jobs + ngroups - 1) / ngroups;
    const double cost = (double)rounds * (tpc + qr / 128.0 + (g > 1 ? 1.0 : 0.0));
    if (cost < best_cost) {
      best_cost = cost;
      best = g;
    }
  }
  if (best == 0) return false;
  pl->single = 1;
  pl->row_tiles = row_tiles;
  pl->jobs = (int)jobs;
  pl->min_nkt = min_nkt;
  pl->max_nkt = max_nkt;
  pl->g = best;
  pl->ngroups = num_sms / best;
  pl->qr = qr;
  size_t b = 0;
  if (best > 1) {
    b += (size_t)jobs * best * qr * sizeof(float2);  // part
    b += (size_t)jobs * sizeof(int);                 // arrive
  }
  pl->ws_bytes = (b + 255) & ~(size_t)255;
  return true;
}

cudaError_t launch_window_vote_tmem(const Ctx &c, const WindowVoteArgs &a,
                                    const WindowVotePlan &pl) {
  int dev = 0;
  cudaGetDevice(&dev);
  const int nch = (pl.qr + 31) / 32;
  const int di = (a.D == 128 ? 4 : 0) + nch - 1;
  const void *fn = nullptr;
  int nthreads = 0;
#define KVC_WVT(DD, NC)                                                  \
  if (a.D == DD && nch == NC) {                                          \
    fn = (const void *)window_vote_tmem_kernel<DD, NC>;                  \
    nthreads = Roles<NC>::NTHREADS;                                      \
  }
  KVC_WVT(128, 1) KVC_WVT(128, 2) KVC_WVT(128, 3) KVC_WVT(128, 4)
  KVC_WVT(64, 1) KVC_WVT(64, 2) KVC_WVT(64, 3) KVC_WVT(64, 4)
#undef KVC_WVT
  if (!fn) return cudaErrorInvalidValue;
  const int smem = a.D == 128 ? Geo<128>::SMEM : Geo<64>::SMEM;
  if (dev < 64 && !g_attr_done[di][dev]) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    g_attr_done[di][dev] = true;
  }
  CUtensorMap tq, tk;
  if (!encode_rows_map(&tq, a.q, (uint64_t)a.units * a.R, a.D, pl.qr)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&tk, a.k, (uint64_t)a.units * a.L, a.D, TILE)) return cudaErrorInvalidValue;
  int blocks_per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, fn, nthreads, smem);
  if (e != cudaSuccess) return e;
  if (blocks_per_sm != 1) return cudaErrorInvalidConfiguration;
  WVP1 p;
  p.L = a.L;
  p.R = a.R;
  p.Wq = a.Wq;
  p.row_tiles = pl.row_tiles;
  p.jobs = pl.jobs;
  p.g = pl.g;
  p.ngroups = pl.ngroups;
  p.qr = pl.qr;
  p.nb = TMEM_COLS / pl.qr;
  if (p.nb > MAXNB) p.nb = MAXNB;
  p.c = (float)(1.4426950408889634 / sqrt((double)a.D));
  p.votes = a.votes;
  p.atomic_votes = p.row_tiles > 1;
  uint8_t *w = reinterpret_cast<uint8_t *>(a.ws);
  p.part = reinterpret_cast<float2 *>(w);
  p.arrive = reinterpret_cast<int *>(p.part + (size_t)p.jobs * p.g * p.qr);
  p.status = c.status;
  p.timeout = c.timeout_ns;
  if (p.g > 1) {
    e = cudaMemsetAsync(p.arrive, 0, (size_t)p.jobs * sizeof(int), c.stream);
    if (e != cudaSuccess) return e;
  }
  if (p.atomic_votes) {
    e = cudaMemsetAsync(a.votes, 0, (size_t)a.units * a.L * sizeof(float), c.stream);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.num_sms);
  cfg.blockDim = dim3(nthreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
#define KVC_WVT(DD, NC) \
  if (a.D == DD && nch == NC) return cudaLaunchKernelEx(&cfg, window_vote_tmem_kernel<DD, NC>, tq, tk, p);
  KVC_WVT(128, 1) KVC_WVT(128, 2) KVC_WVT(128, 3) KVC_WVT(128, 4)
  KVC_WVT(64, 1) KVC_WVT(64, 2) KVC_WVT(64, 3) KVC_WVT(64, 4)
#undef KVC_WVT
  return cudaErrorInvalidValue;
}

}  // namespace kvc
