// Prompt self-attention with the SnapKV votes as a by-product (SnapKV article, 推論方法:
// the compression runs right after the prompt has been processed, so the window's
// attention can come out of the prefill itself).  For every (layer, batch, query head):
// O = softmax(Q K^T / sqrt(D) + causal mask) V over the whole prompt, and for the last
// Wq rows (the observation window) their probabilities summed per key into the votes of
// the head's KV head: the same v_j as snapkv_compress's window vote (rows see keys up to
// their own position).
//
// Design (sm_103a; flash-attention forward on tcgen05):
// * jobs are (query head, 128-row query tile), heaviest tiles first, spread over a
//   persistent grid (one CTA per SM) in rounds whose CTA order alternates;
// * warp 0 streams, per job, its Q tile and then K0, V0, K1, V1, ... (keys 0..end of
//   the tile) through two 3-stage TMA rings, one for K and one for V (128-byte swizzle);
//   warp 1 issues S = Q.K^T into one of two TMEM score buffers, and warp 6 issues
//   O += P.V into a TMEM accumulator (P, bf16, read as the A operand straight from tensor
//   memory; V read MN-major from its ring stage): a tcgen05.mma holds its issuing thread
//   for about its execution time, so the two products get a thread each, and each ring
//   has one consumer; warps 2-5 own one query row per thread: the row's 128 scores come
//   from TMEM at once, the online softmax runs in registers (a row's reference max moves
//   only when the max passes it by more than 2^8, and then the row of O is rescaled in
//   TMEM), and P goes back to tensor memory with tcgen05.st;
// * a query tile that holds window rows is swept twice: first K only, for each row's
//   exact max and normaliser, then the output sweep, where those rows' final
//   probabilities are also summed per key (a transpose-reduce across the warp) and added
//   into the votes; no other tile needs a second look at K.
// * every wait is bounded; a timeout sets the device status word and abandons the work.
#include <math.h>

#include "prefill.cuh"

namespace kvc {
namespace {

constexpr int ROWS = 128;      // query rows per tile (MMA M)
constexpr int KT = 128;        // keys per tile (MMA N of S, K of P.V)
constexpr int NSK = 3;         // K tile ring (consumed by the S issuer only)
constexpr int NSV = 3;         // V tile ring (consumed by the P.V issuer only)
constexpr int NSW = 4;         // softmax warps: one query row per thread
constexpr int WPV = 2 + NSW;   // the P.V issuer's warp (after the TMA, S-issuer and softmax warps)
constexpr int NTH = 32 * (3 + NSW);
constexpr float SLACK = 8.f;   // log2 headroom before a row's reference max moves
constexpr int TMEM_COLS = 512; // S0, S1, O, P

template <int D>
struct PGeo {
  static constexpr int KB = D / 64;
  static constexpr int KBLK = ROWS * 128;       // one 64-column block of a 128-row tile
  static constexpr int TB = KB * KBLK;          // Q, K or V tile bytes
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + TB;         // K ring
  static constexpr int OFF_VRING = OFF_RING + NSK * TB;  // V ring
  static constexpr int OFF_BAR = OFF_VRING + NSV * TB;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;
  static_assert(TB % 1024 == 0, "swizzled operands stay 1024-aligned");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// barrier offsets (bytes from OFF_BAR)
constexpr int B_FULLK = 0;     // [NSK <= 4] K stage loaded
constexpr int B_EMPTYK = 32;   // [NSK] K stage read by its S (commit)
constexpr int B_FULLV = 64;    // [NSV <= 4] V stage loaded
constexpr int B_EMPTYV = 96;   // [NSV] V stage read by its P.V (commit)
constexpr int B_QFULL = 128;   // Q tile loaded
constexpr int B_QEMPTY = 136;  // the job's MMAs are done with Q (commit)
constexpr int B_SFULL = 144;   // [2] score buffer written (commit)
constexpr int B_SEMPTY = 160;  // [2] score buffer read (NSW warps)
constexpr int B_PFULL = 176;   // P written (NSW warps)
constexpr int B_PDONE = 184;   // P.V complete: P free, O stable (commit)
constexpr int B_OFREE = 192;   // the job's O has been read out (NSW warps)
constexpr int B_ABORT = 200;   // int
constexpr int B_TMEM = 204;    // uint32
static_assert(NSK <= 4 && NSV <= 4, "ring barrier slots");

struct PreP {
  const __nv_bfloat16 *q;  // [Uq, L, D]
  __nv_bfloat16 *o;        // [Uq, L, D]
  float *votes;            // [Ukv, L] (zeroed by the launcher) or null
  float *lse;              // [Uq, L] or null: natural-log log-sum-exp of each row's scores
  int L, G, Wq, uq, nqt;   // uq = query-head units, nqt = query tiles per head
  float c;                 // log2(e) / sqrt(D)
  uint32_t *status;
  unsigned long long timeout;
};

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
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory descriptor of a 128-byte-swizzled MN-major operand (V as the B of
// P.V: 64 contiguous head-dim values per 128-byte row, one row per key): the 64-wide
// column blocks are `lbo` bytes apart, the 8-key groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_mn128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Job geometry: job index -> (query-head unit, query tile), heaviest tiles first.
struct PJob {
  int uq, qt, nkt;   // unit, query tile, key tiles 0..nkt-1
  bool twice;        // the tile holds window rows: a statistics sweep first
};
__device__ __forceinline__ PJob pjob(const PreP &p, int j) {
  PJob J;
  J.qt = p.nqt - 1 - j / p.uq;
  J.uq = j - (j / p.uq) * p.uq;
  J.nkt = J.qt + 1;  // causal: keys up to the tile's last row
  J.twice = p.votes != nullptr && J.qt * ROWS + ROWS > p.L - p.Wq;
  return J;
}


// D (+)= A . B with A (128 x 16 bf16) read from tensor memory: row m on lane m, the 16
// K values packed two per 32-bit column (8 columns, the lower K index in the low half).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// Sum over the warp's 32 lanes of each of x[0..31]; afterwards lane c holds the sum of
// x[c] (recursive halving: each step keeps half of the values and adds the partner's).
__device__ __forceinline__ float transpose_reduce32(float (&x)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
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

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of s[0..127]: eight independent chains of three-input max, then a short tree.
__device__ __forceinline__ float max128(const float *s) {
  float m[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = fmax3(s[j], s[j + 8], s[j + 16]);
#pragma unroll
  for (int t = 3; t < 15; t += 2)
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = fmax3(m[j], s[j + 8 * t], s[j + 8 * t + 8]);
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], s[j + 120]);
  return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// Sum of exp2(s[i] c + nm) over i < 128 (c and nm packed twice), four packed chains.
__device__ __forceinline__ float exp2_sum128(const float *s, unsigned long long cc,
                                             unsigned long long nm) {
  unsigned long long a[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int i = 0; i < 128; i += 8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = upk(fma2(pk(s[i + 2 * j], s[i + 2 * j + 1]), cc, nm));
      a[j] = add2(a[j], pk(ex2(x.x), ex2(x.y)));
    }
  }
  const float2 t = upk(add2(add2(a[0], a[1]), add2(a[2], a[3])));
  return t.x + t.y;
}

// s[i] <- exp2(s[i] c + nm) for i < 128; returns their sum (four packed chains).
__device__ __forceinline__ float exp2_inplace128(float *s, unsigned long long cc,
                                                 unsigned long long nm) {
  unsigned long long a[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int i = 0; i < 128; i += 8) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 x = upk(fma2(pk(s[i + 2 * j], s[i + 2 * j + 1]), cc, nm));
      s[i + 2 * j] = ex2(x.x);
      s[i + 2 * j + 1] = ex2(x.y);
      a[j] = add2(a[j], pk(s[i + 2 * j], s[i + 2 * j + 1]));
    }
  }
  const float2 t = upk(add2(add2(a[0], a[1]), add2(a[2], a[3])));
  return t.x + t.y;
}

template <int D>
__global__ void __launch_bounds__(NTH, 1) prefill_kernel(const __grid_constant__ CUtensorMap tq,
                                                         const __grid_constant__ CUtensorMap tk,
                                                         const __grid_constant__ CUtensorMap tv,
                                                         const PreP p) {
  using Gm = PGeo<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar = sb + Gm::OFF_BAR;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + B_ABORT);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Gm::OFF_BAR + B_TMEM);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{abort_flag, p.status, p.timeout};

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NSK; ++i) {
      mbar_init(bar + B_FULLK + 8 * i, 1);
      mbar_init(bar + B_EMPTYK + 8 * i, 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(bar + B_FULLV + 8 * i, 1);
      mbar_init(bar + B_EMPTYV + 8 * i, 1);
    }
    mbar_init(bar + B_QFULL, 1);
    mbar_init(bar + B_QEMPTY, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar + B_SFULL + 8 * i, 1);
      mbar_init(bar + B_SEMPTY + 8 * i, NSW);
    }
    mbar_init(bar + B_PFULL, NSW);
    mbar_init(bar + B_PDONE, 1);
    mbar_init(bar + B_OFREE, NSW);
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
  const uint32_t tO = tmem + 256;  // O accumulator columns 256 .. 256 + D - 1
  const uint32_t tP = tmem + 384;  // P of the tile, bf16 pairs: columns 384 .. 447

  // jobs of this CTA: rounds of gridDim.x jobs, CTA order reversed on odd rounds
  const int P = gridDim.x, jobs = p.uq * p.nqt;
  const int full = jobs / P, rem = jobs - full * P, b = blockIdx.x;
  const int njobs = full + ((full & 1) ? (P - 1 - b < rem) : (b < rem));
  auto job_of = [&](int k) { return k * P + ((k & 1) ? P - 1 - b : b); };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      int ik = 0, iv = 0;
      bool ok = true;
      // next K tile into the K ring, or V tile into the V ring (key tile at `row`)
      auto load = [&](bool isv, int row) {
        const int n = isv ? NSV : NSK, i = isv ? iv : ik, st = i % n;
        const uint32_t full = bar + (isv ? B_FULLV : B_FULLK) + 8 * st;
        if (!ab.wait(bar + (isv ? B_EMPTYV : B_EMPTYK) + 8 * st, ((i / n) & 1) ^ 1)) return false;
        mbar_arrive_expect_tx(full, Gm::TB);
        const uint32_t dst = sb + (isv ? Gm::OFF_VRING : Gm::OFF_RING) + st * Gm::TB;
        for (int kb = 0; kb < Gm::KB; ++kb)
          tma_load_2d(dst + kb * Gm::KBLK, isv ? &tv : &tk, kb * 64, row, full);
        if (isv) ++iv; else ++ik;
        return true;
      };
      for (int k = 0; k < njobs && ok; ++k) {
        const PJob J = pjob(p, job_of(k));
        const int ukv = J.uq / p.G;
        if (!ab.wait(bar + B_QEMPTY, (k & 1) ^ 1)) break;
        mbar_arrive_expect_tx(bar + B_QFULL, Gm::TB);
        for (int kb = 0; kb < Gm::KB; ++kb)
          tma_load_2d(sb + Gm::OFF_Q + kb * Gm::KBLK, &tq, kb * 64, J.uq * p.L + J.qt * ROWS,
                      bar + B_QFULL);
        if (J.twice)
          for (int kt = 0; kt < J.nkt && ok; ++kt) ok = load(false, ukv * p.L + kt * KT);
        for (int kt = 0; kt < J.nkt && ok; ++kt) {
          ok = load(false, ukv * p.L + kt * KT);
          if (ok) ok = load(true, ukv * p.L + kt * KT);
        }
      }
      for (int st = 0; st < NSK; ++st) {  // drain
        const int cnt = ik / NSK + (st < ik % NSK ? 1 : 0);
        if (cnt > 0) mbar_wait_bounded(bar + B_FULLK + 8 * st, (cnt - 1) & 1, p.timeout);
      }
      for (int st = 0; st < NSV; ++st) {
        const int cnt = iv / NSV + (st < iv % NSV ? 1 : 0);
        if (cnt > 0) mbar_wait_bounded(bar + B_FULLV + 8 * st, (cnt - 1) & 1, p.timeout);
      }
      if (njobs > 0) mbar_wait_bounded(bar + B_QFULL, (njobs - 1) & 1, p.timeout);
    }
  } else if (warp == 1) {
    // ------------------------------ S issuer ------------------------------
    // S = Q . K^T per K tile into the two score buffers.  The P.V products have their own
    // issuer (warp WPV): an MMA's issue holds its thread for about its execution time,
    // so one thread issuing both would serialise them with its own waits.
    if (lane == 0) {
      int ik = 0, sc = 0;
      bool ok = true;
      const uint32_t id_s = idesc_bf16(ROWS, KT);
      const uint64_t qd = sdesc_k128(sb + Gm::OFF_Q);
      // S of the next K tile, into buffer sc & 1
      auto issue_s = [&]() {
        const int st = ik % NSK, sbf = sc & 1;
        if (!ab.wait(bar + B_FULLK + 8 * st, (ik / NSK) & 1)) return false;
        if (!ab.wait(bar + B_SEMPTY + 8 * sbf, ((sc >> 1) & 1) ^ 1)) return false;
        tc_fence_after();
        const uint64_t kd = sdesc_k128(sb + Gm::OFF_RING + st * Gm::TB);
#pragma unroll
        for (int kb = 0; kb < Gm::KB; ++kb)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t o = (uint64_t)((kb * Gm::KBLK + kk * 32) >> 4);
            umma_bf16(tmem + (uint32_t)(sbf * 128), qd + o, kd + o, id_s, (kb | kk) != 0);
          }
        umma_commit(bar + B_EMPTYK + 8 * st);
        umma_commit(bar + B_SFULL + 8 * sbf);
        ++sc;
        ++ik;
        return true;
      };
      for (int k = 0; k < njobs && ok; ++k) {
        const PJob J = pjob(p, job_of(k));
        if (!ab.wait(bar + B_QFULL, k & 1)) break;
        tc_fence_after();
        if (J.twice)
          for (int kt = 0; kt < J.nkt && ok; ++kt) ok = issue_s();
        for (int kt = 0; kt < J.nkt && ok; ++kt) {
          ok = issue_s();
          if (ok && kt == J.nkt - 1) umma_commit(bar + B_QEMPTY);  // Q no longer read
        }
      }
      // drain: the last commit covers every S this thread issued
      if (ik > 0) mbar_wait_bounded(bar + B_EMPTYK + 8 * ((ik - 1) % NSK), ((ik - 1) / NSK) & 1, p.timeout);
    }
  } else if (warp == WPV) {
    // ------------------------------ P.V issuer ------------------------------
    if (lane == 0) {
      int iv = 0, pc = 0;
      bool ok = true;
      const uint32_t id_pv = idesc_bf16(ROWS, D) | (1u << 16);  // B (V) MN-major
      // O (+)= P . V with the next V tile
      auto issue_pv = [&](bool first) {
        const int st = iv % NSV;
        if (!ab.wait(bar + B_PFULL, pc & 1)) return false;
        if (!ab.wait(bar + B_FULLV + 8 * st, (iv / NSV) & 1)) return false;
        tc_fence_after();
        const uint32_t vbase = sb + Gm::OFF_VRING + st * Gm::TB;
#pragma unroll
        for (int ks = 0; ks < KT / 16; ++ks) {  // P from tensor memory, 16 keys (8 columns) a step
          const uint64_t vd = sdesc_mn128(vbase + ks * 16 * 128, Gm::KBLK);
          umma_bf16_ts(tO, tP + (uint32_t)(ks * 8), vd, id_pv, (!first || ks > 0) ? 1u : 0u);
        }
        umma_commit(bar + B_EMPTYV + 8 * st);
        umma_commit(bar + B_PDONE);
        ++pc;
        ++iv;
        return true;
      };
      for (int k = 0; k < njobs && ok; ++k) {
        const PJob J = pjob(p, job_of(k));
        for (int kt = 0; kt < J.nkt && ok; ++kt) {
          if (kt == 0 && k > 0 && !ab.wait(bar + B_OFREE, (k - 1) & 1)) { ok = false; break; }
          ok = issue_pv(kt == 0);
        }
      }
      // drain: the last commit (P.V) covers every MMA this thread issued
      if (pc > 0) mbar_wait_bounded(bar + B_PDONE, (pc - 1) & 1, p.timeout);
    }
  } else {
    // ---------------- softmax warps: one query row per thread ----------------
    // A tile's 128 scores of the row are loaded into registers at once (the score
    // buffer is released right away), the row max comes from a three-input max tree,
    // the exponentials are formed and packed to bf16 before waiting for the previous P.V
    // (only the tcgen05.st of P into tensor memory waits for it), and FFMA / FADD run
    // packed two lanes at a time.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const unsigned long long cc = pk(p.c, p.c);
    int sc = 0, pc = 0;
    bool ok = true;
    for (int k = 0; k < njobs; ++k) {
      const PJob J = pjob(p, job_of(k));
      const int row = J.qt * ROWS + r;  // position in the prompt
      const bool valid = row < p.L;
      const int ukv = J.uq / p.G;
      // Scores of tile kt (buffer sbf) into s[0..127], the buffer then released.  Only
      // the diagonal tile (kt == qt) holds keys after the row; rows past the prompt
      // (the last query tile) keep finite scores of zero-filled queries and never reach
      // the output or the votes.
      auto release = [&](int sbf) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar + B_SEMPTY + 8 * sbf);
      };
      auto load_tile = [&](int sbf, int kt, float (&sv)[KT], bool rel) {
#pragma unroll
        for (int ch = 0; ch < KT / 32; ++ch)
          tmem_ld32(tmem + lane_base + (uint32_t)(sbf * 128 + ch * 32), sv + ch * 32);
        tmem_wait_ld();
        if (rel) release(sbf);
        if (kt == J.qt) {
#pragma unroll
          for (int i = 0; i < KT; ++i)
            if (kt * KT + i > row) sv[i] = -INFINITY;
        }
      };
      float m = -INFINITY, l = 0.f;
      if (J.twice) {  // statistics sweep: exact max and normaliser of every row
        for (int kt = 0; kt < J.nkt; ++kt, ++sc) {
          const int sbf = sc & 1;
          ok = __all_sync(0xffffffffu, ok && ab.wait(bar + B_SFULL + 8 * sbf, (sc >> 1) & 1));
          if (!ok) continue;
          tc_fence_after();
          float sv[KT];
          load_tile(sbf, kt, sv, true);
          const float mn = fmaxf(m, max128(sv) * p.c);
          const float mref = mn == -INFINITY ? 0.f : mn;  // a row with no visible key adds 0
          const float add = exp2_sum128(sv, cc, pk(-mref, -mref));
          if (mn != -INFINITY) {
            l = l * ex2(m - mn) + add;  // ex2(-inf) = 0 for the first finite max
            m = mn;
          }
        }
      }
      // output sweep
      const bool fixed = J.twice;  // the reference max is final: no rescaling
      const float inv_z = (fixed && l > 0.f) ? 1.f / l : 0.f;
      const bool wrow = fixed && valid && row >= p.L - p.Wq;   // a window row: it votes
      const bool wwarp = __any_sync(0xffffffffu, wrow);
      if (!fixed) {
        m = -INFINITY;
        l = 0.f;
      }
      for (int kt = 0; kt < J.nkt; ++kt, ++sc) {
        const int sbf = sc & 1;
        ok = __all_sync(0xffffffffu, ok && ab.wait(bar + B_SFULL + 8 * sbf, (sc >> 1) & 1));
        uint32_t pw[KT / 2];  // P of the row, bf16 pairs
        float alpha = 1.f;
        bool rescale = false;
        if (ok) {
          float sv[KT];
          tc_fence_after();
          load_tile(sbf, kt, sv, !wwarp);  // window warps read the scores again below
          if (!fixed) {
            const float tm = max128(sv) * p.c;
            if (tm > m + SLACK || (m == -INFINITY && tm != -INFINITY)) {
              alpha = m == -INFINITY ? 0.f : ex2(m - tm);
              rescale = m != -INFINITY;
              l *= alpha;
              m = tm;
            }
          }
          // P = exp2(s c - m) in place (m = -inf: the row sees no key yet, P = 0)
          const float nm = m == -INFINITY ? -INFINITY : -m;
          const float add = exp2_inplace128(sv, cc, pk(nm, nm));
          if (!fixed) l += add;
#pragma unroll
          for (int i = 0; i < KT / 2; ++i) pw[i] = pack_bf16(sv[2 * i], sv[2 * i + 1]);
        }
        // P buffer and O are free once the previous P.V has completed
        if (pc > 0) ok = __all_sync(0xffffffffu, ok && ab.wait(bar + B_PDONE, (pc - 1) & 1));
        if (ok) {
          tc_fence_after();
          if (__any_sync(0xffffffffu, rescale)) {  // rows whose reference moved: O *= alpha
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              float o[32];
              tmem_ld32(tO + lane_base + (uint32_t)c0, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha;
              tmem_st32(tO + lane_base + (uint32_t)c0, o);
            }
            tmem_wait_st();
          }
          // the P row into tensor memory (lane r, keys 2i and 2i + 1 in column i)
          tmem_st32(tP + lane_base, reinterpret_cast<const float *>(pw));
          tmem_st32(tP + lane_base + 32u, reinterpret_cast<const float *>(pw + 32));
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar + B_PFULL);
          if (wwarp) {
            // window rows: their final probabilities (the same exp2(s c - m) as P, from
            // the scores read again), summed per key; then the score buffer is released
            const float nm = -m;
#pragma unroll 1
            for (int ch = 0; ch < KT / 32; ++ch) {
              float t[32];
              tmem_ld32(tmem + lane_base + (uint32_t)(sbf * 128 + ch * 32), t);
              tmem_wait_ld();
              const int key0 = kt * KT + ch * 32;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                t[i] = (wrow && key0 + i <= row) ? ex2(fmaf(t[i], p.c, nm)) * inv_z : 0.f;
              const float vsum = transpose_reduce32(t, lane);
              const int key = key0 + lane;
              if (key < p.L && vsum != 0.f) atomicAdd(p.votes + (size_t)ukv * p.L + key, vsum);
            }
            release(sbf);
          }
        }
        ++pc;
      }
      // the job's output rows: O / l in bf16, then O is free for the next job; and the
      // row's log-sum-exp, ln 2 (m + log2 l) (m and l are in the log2 domain of s c)
      if (ok && valid && p.lse)
        p.lse[(size_t)J.uq * p.L + row] = l > 0.f ? 0.6931471805599453f * (m + lg2(l)) : -INFINITY;
      ok = __all_sync(0xffffffffu, ok && ab.wait(bar + B_PDONE, (pc - 1) & 1));
      if (ok) {
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        __nv_bfloat16 *orow = p.o + ((size_t)J.uq * p.L + row) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tmem_ld32(tO + lane_base + (uint32_t)c0, o);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint4 w;
              w.x = pack_bf16(o[c8 * 8 + 0] * inv, o[c8 * 8 + 1] * inv);
              w.y = pack_bf16(o[c8 * 8 + 2] * inv, o[c8 * 8 + 3] * inv);
              w.z = pack_bf16(o[c8 * 8 + 4] * inv, o[c8 * 8 + 5] * inv);
              w.w = pack_bf16(o[c8 * 8 + 6] * inv, o[c8 * 8 + 7] * inv);
              *reinterpret_cast<uint4 *>(orow + c0 + c8 * 8) = w;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar + B_OFREE);
      }
    }
  }

  // ---------------------------------- teardown ----------------------------------
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}


template <int D>
cudaError_t launch_t(const Ctx &c, const PrefillArgs &a, PreP p) {
  static bool attr[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               PGeo<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  CUtensorMap tq, tk, tv;
  const uint64_t ukv = (uint64_t)a.units_q / a.G;
  if (!encode_rows_map(&tq, a.q, (uint64_t)a.units_q * a.L, D, ROWS)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&tk, a.k, ukv * a.L, D, KT)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&tv, a.v, ukv * a.L, D, KT)) return cudaErrorInvalidValue;
  const long long jobs = (long long)a.units_q * p.nqt;
  const int grid = (int)(jobs < c.num_sms ? jobs : c.num_sms);
  prefill_kernel<D><<<grid, NTH, PGeo<D>::SMEM, c.stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const Ctx &c, const PrefillArgs &a) {
  if (a.units_q < 1 || a.G < 1 || a.units_q % a.G || a.L < 1 || (a.D != 64 && a.D != 128))
    return cudaErrorInvalidValue;
  PreP p;
  p.q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
  p.o = reinterpret_cast<__nv_bfloat16 *>(a.o);
  p.votes = a.votes;
  p.lse = a.lse;
  p.L = a.L;
  p.G = a.G;
  p.Wq = a.Wq;
  p.uq = a.units_q;
  p.nqt = (a.L + ROWS - 1) / ROWS;
  p.c = (float)(1.4426950408889634 / sqrt((double)a.D));
  p.status = c.status;
  p.timeout = c.timeout_ns;
  if (a.votes) {
    const cudaError_t e = cudaMemsetAsync(a.votes, 0, (size_t)(a.units_q / a.G) * a.L * sizeof(float),
                                          c.stream);
    if (e != cudaSuccess) return e;
  }
  if (a.D == 128) return launch_t<128>(c, a, p);
  return launch_t<64>(c, a, p);
}

}  // namespace kvc
