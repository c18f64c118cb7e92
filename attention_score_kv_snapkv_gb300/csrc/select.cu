// SnapKV steps 3-4 (SnapKV article, 処理の流れ steps 3 and 4): 1D pooling of the vote
// over the prefix candidates (max-pool, or the window average as the pooling variant),
// per-head top-k (equal pooled votes: lower position first), then the gather of the
// kept prefix rows and the kept window into the compact cache.  The same code cuts
// H2O's prompt to heavy hitters + recent window (pool 1).
//
// pool_topk_kernel: one CTA (512 threads, two per SM) per unit.
//   phase 0  pooled vote u_j = max(v[j-h .. j+h]) (cut at the candidate range; or the
//            sum of that window / (2h + 1), zeros past the ends, for average pooling) turned
//            into an order-preserving uint32 key; the votes are staged through shared
//            memory (16-byte loads where the row is aligned);
//   phase 1  radix select of the k-th largest key;
//   phase 2  stream compaction in position order: keys above the threshold, and the
//            first `need` keys equal to it (exact lower-position tie rule), written as
//            ascending positions (per-thread runs, one block-wide scan).
//   Pool kernel 7 with at most 32 candidates per thread (the usual SnapKV setting) keeps
//   each thread's 32 keys in registers and selects with three digits (11, 11, 10 bits)
//   over one shared histogram -- in pool_topk_gather_kernel, which then gathers the
//   unit's rows itself; longer prompts with pool kernel 7 go in chunks of that size
//   (pool_topk_chunk_kernel, then topk_merge_kernel, which gathers); other pool sizes
//   keep the keys in shared (else global) memory and select with four 8-bit digits over
//   per-warp histograms.
// gather_kernel: 16-byte vectorised copy of the kept K/V rows, positions, scores (after
//   pool_topk_kernel, or alone when every position is kept).
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int NT = 512;          // threads of pool_topk_kernel (two CTAs per SM)
constexpr int NWARP = NT / 32;
constexpr int NBIN = 256;        // radix digit of 8 bits, four passes
constexpr int CHUNK = 4096;      // pooling staging floats (aliases the histograms)
constexpr int SMEM_KEYS_MAX = 48 * 1024;  // candidates kept in shared memory

constexpr int RUN = 32;          // positions per thread in the kernel-7 pooling path
constexpr int CHUNK_C = NT * RUN;  // candidates per CTA of the chunked path
constexpr int RUN2 = 16;         // candidates per thread in the merge of the chunked path

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct TopkP {
  const float *votes;  // [U, L]
  int L, n_cand, k, half;  // half = (pool kernel - 1) / 2
  int avg;             // 1: window average (sum / (2 half + 1), zeros past the ends), 0: max
  int32_t *sel;        // [U, cap] output positions
  int cap;
  uint32_t *kglobal;   // [U, n_cand] keys when they do not fit in shared memory
  // chunked path (long prompts): each chunk's local top-k, positions and keys
  int nchunks;         // chunks of CHUNK_C candidates per unit
  int32_t *cpos;       // [U, nchunks, cap]
  uint32_t *ckey;      // [U, nchunks, cap]
};

// shared memory (32-bit words): per-warp histograms [NWARP][NBIN] (the pooling stage
// buffer while pooling), merged histogram [NBIN], misc [128], then the keys
constexpr int SM_HIST = 0;
constexpr int SM_TOT = NWARP * NBIN;
constexpr int SM_MISC = SM_TOT + NBIN;
constexpr int SM_KEYS = SM_MISC + 128;
static_assert(NWARP * NBIN >= CHUNK, "the pooling stage aliases the histograms");
// Keys are stored with one pad word per 32 (key j at kidx(j)): a warp reading 32
// consecutive keys and a thread writing its run of 32 are both free of bank conflicts.
__host__ __device__ constexpr int kidx(int j) { return j + (j >> 5); }
// words of the key region: the padded keys, or the padded staging of the votes with a
// halo of 3 on both sides
__host__ __device__ constexpr int key_words(int n) { return n + 6 + (n + 6) / 32 + 1; }

// Fast path (pool kernel 7, candidates fit one run of RUN per thread): the keys stay in
// registers and the radix select uses three digits (bits 31-21, 20-10, 9-0) over one
// shared histogram of NB bins.  misc words used: [0] bin found, [1] keys still to take
// from it, [8, 8 + NWARP) warp totals of the bin search, [32, 32 + NWARP) warp totals of
// the compaction scan.
constexpr int NB = 2048;
constexpr int M_BIN = 0, M_NEED = 1, M_WSUM = 8, M_CSUM = 32;
static_assert(NWARP * NBIN >= NB, "the fast path's histogram aliases the per-warp histograms");

// Bin search over a histogram of PER * NT bins: finds the bin b holding the need-th largest
// key (the bins above b hold fewer than `need` keys, b and those above at least `need`;
// 1 <= need <= the histogram's total) and writes misc[M_BIN] = b, misc[M_NEED] = need minus
// the keys above b.  Thread t owns bins [t PER, (t + 1) PER); suffix sums run over the
// lanes of a warp, then over the warps.  Ends synchronised.
template <int PER>
__device__ __forceinline__ void find_bin(const uint32_t *hist, int *misc, int need) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t own[PER], s = 0;
#pragma unroll
  for (int b = 0; b < PER; ++b) {
    own[b] = hist[tid * PER + b];
    s += own[b];
  }
  uint32_t incl = s;  // keys in the bins of this lane and every higher lane of the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += t;
  }
  if (lane == 0) misc[M_WSUM + warp] = (int)incl;
  __syncthreads();
  uint32_t above = incl - s;
  for (int w = warp + 1; w < NWARP; ++w) above += (uint32_t)misc[M_WSUM + w];
  if (above < (uint32_t)need && (uint32_t)need <= above + s) {
    uint32_t acc = above;
#pragma unroll
    for (int b = PER - 1; b >= 0; --b) {
      if (acc + own[b] >= (uint32_t)need) {
        misc[M_BIN] = tid * PER + b;
        misc[M_NEED] = need - (int)acc;
        break;
      }
      acc += own[b];
    }
  }
  __syncthreads();
}

// The pool-kernel-7 (or pool-kernel-1: nopool) path with each thread's keys in registers:
// pooled keys of the candidates [c0, c0 + nc) of a unit whose votes v hold nall candidates
// (the windows read up to three positions beyond the range where those exist, else the
// padding), then the
// positions of the k largest (equal keys: lower position first), ascending, into
// sel_out[0..k) and, with key_out, their keys beside them.  nc <= NT * RUN, 1 <= k <= nc.
// Shared memory: the histogram region, misc, and key_words(nc) words at `stage`.
__device__ __forceinline__ void select_run(const float *v, int c0, int nc, int nall, int k,
                                           bool avg, bool nopool, int32_t *sel_out,
                                           uint32_t *key_out, uint32_t *sm, uint32_t *stage,
                                           int *misc) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float pad = avg ? 0.f : -INFINITY;  // value beyond both ends of the candidates
  const float inv = 1.f / 7.f;
  // pool kernel 7, one run of 32 consecutive positions per thread: the votes go to
  // shared memory with one pad word per 32 (a thread's run is then conflict-free
  // across the warp); the run and its halo are read into registers and the window
  // maxima (or sums) formed there.  Staged index jj holds position jj - 3.
  float *vs = reinterpret_cast<float *>(stage);
  const float *vc = v + c0;
  if ((reinterpret_cast<uintptr_t>(vc) & 15u) == 0) {
    // 16-byte loads, all of a thread's in flight together
    const int n4 = nc >> 2;
    const float4 *v4 = reinterpret_cast<const float4 *>(vc);
    for (int i1 = tid; i1 < n4; i1 += 8 * NT) {
      float4 t8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = i1 + e * NT;
        t8[e] = i < n4 ? __ldg(v4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int i = i1 + e * NT;
        if (i < n4) {
          const int jj = 4 * i + 3;
          vs[kidx(jj)] = t8[e].x;
          vs[kidx(jj + 1)] = t8[e].y;
          vs[kidx(jj + 2)] = t8[e].z;
          vs[kidx(jj + 3)] = t8[e].w;
        }
      }
    }
    if (tid < 3) {  // the halos: three positions below and above the range
      const int lo = c0 - 3 + tid, hi = c0 + nc + tid;
      vs[kidx(tid)] = lo >= 0 ? __ldg(v + lo) : pad;
      vs[kidx(nc + 3 + tid)] = hi < nall ? __ldg(v + hi) : pad;
    } else if (tid < 3 + (nc & 3)) {  // the last nc % 4 candidates
      const int q = (nc & ~3) + tid - 3;
      vs[kidx(q + 3)] = __ldg(vc + q);
    }
  } else {
    // eight loads in flight per thread before the stores
    for (int j1 = tid; j1 < nc + 6; j1 += 8 * NT) {
      float t8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int q = c0 + j1 + e * NT - 3;  // the position staged at index j1 + e NT
        t8[e] = (j1 + e * NT < nc + 6 && q >= 0 && q < nall) ? __ldg(v + q) : pad;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = j1 + e * NT;
        if (j < nc + 6) vs[kidx(j)] = t8[e];
      }
    }
  }
  uint32_t *hist = sm + SM_HIST;
  for (int b = tid; b < NB; b += NT) hist[b] = 0;
  __syncthreads();
  const int j0 = tid * RUN;
  uint32_t key[RUN];  // this thread's pooled keys (positions j0 ..), 0 past the candidates
  {
    float w[RUN + 6];
#pragma unroll
    for (int i = 0; i < RUN + 6; ++i) {
      const int jj = j0 + i;  // staged index of position j0 + i - 3
      w[i] = jj < nc + 6 ? vs[kidx(jj)] : pad;
    }
#pragma unroll
    for (int i = 0; i < RUN; ++i) {
      const float m = nopool ? w[i + 3]
                      : avg ? (((((w[i] + w[i + 1]) + w[i + 2]) + w[i + 3]) + w[i + 4]) + w[i + 5] + w[i + 6]) * inv
                            : fmax3(fmax3(w[i], w[i + 1], w[i + 2]), fmax3(w[i + 3], w[i + 4], w[i + 5]), w[i + 6]);
      key[i] = j0 + i < nc ? order_key(m) : 0u;
    }
  }
  // radix pass 0 (bits 31-21): neighbouring pooled values mostly share their top digit,
  // so a thread adds each run of equal digits with one shared atomic
  {
    uint32_t cur = 0xffffffffu, cnt = 0;
#pragma unroll
    for (int i = 0; i < RUN; ++i) {
      if (j0 + i < nc) {
        const uint32_t b = key[i] >> 21;
        if (b != cur) {
          if (cnt) atomicAdd(&hist[cur], cnt);
          cur = b;
          cnt = 0;
        }
        ++cnt;
      }
    }
    if (cnt) atomicAdd(&hist[cur], cnt);
  }
  __syncthreads();
  find_bin<NB / NT>(hist, misc, k);
  const uint32_t b0 = (uint32_t)misc[M_BIN];
  int need = misc[M_NEED];
#pragma unroll
  for (int b = 0; b < NB / NT; ++b) hist[tid * (NB / NT) + b] = 0;  // own bins (read above)
  __syncthreads();
  // radix pass 1 (bits 20-10) over the keys of bucket b0
#pragma unroll
  for (int i = 0; i < RUN; ++i)
    if (j0 + i < nc && (key[i] >> 21) == b0) atomicAdd(&hist[(key[i] >> 10) & (NB - 1)], 1u);
  __syncthreads();
  find_bin<NB / NT>(hist, misc, need);
  const uint32_t pre = (b0 << 11) | (uint32_t)misc[M_BIN];  // key >> 10 of the bucket
  need = misc[M_NEED];
#pragma unroll
  for (int b = 0; b < NB / NT; ++b) hist[tid * (NB / NT) + b] = 0;
  __syncthreads();
  // radix pass 2 (bits 9-0)
#pragma unroll
  for (int i = 0; i < RUN; ++i)
    if (j0 + i < nc && (key[i] >> 10) == pre) atomicAdd(&hist[key[i] & 1023u], 1u);
  __syncthreads();
  find_bin<1024 / NT>(hist, misc, need);
  const uint32_t T = (pre << 10) | (uint32_t)misc[M_BIN];
  need = misc[M_NEED];
  // compaction in position order: counts above / equal to the threshold, a block-wide
  // exclusive scan, then each thread writes its chosen positions (ties: the first
  // `need` equal keys by position)
  // this thread's keys above and equal to the threshold, as bit masks over its run
  uint32_t gtm = 0u, eqm = 0u;
#pragma unroll
  for (int i = 0; i < RUN; ++i) {
    const bool valid = j0 + i < nc;
    gtm |= (valid && key[i] > T) ? (1u << i) : 0u;
    eqm |= (valid && key[i] == T) ? (1u << i) : 0u;
  }
  // keys for key_out are read back by position below: staged where the votes were (every
  // thread has finished reading the votes: barriers have passed since)
  if (key_out) {
#pragma unroll
    for (int i = 0; i < RUN; ++i)
      if (j0 + i < nc) stage[kidx(j0 + i)] = key[i];
  }
  const int gt = __popc(gtm), eq = __popc(eqm);
  const int packed = gt | (eq << 16);
  int incl = packed;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) misc[M_CSUM + warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w2 = 0; w2 < warp; ++w2) wbase += misc[M_CSUM + w2];
  const int excl = wbase + incl - packed;
  const int eq_before = excl >> 16;
  // the taken keys: every key above the threshold, and of the equal ones the first
  // `need` by position across the CTA, i.e. this thread's first need - eq_before
  uint32_t m = gtm;
  for (int t = max(0, min(eq, need - eq_before)); t > 0; --t) {
    const uint32_t low = eqm & (0u - eqm);
    m |= low;
    eqm ^= low;
  }
  int out = (excl & 0xffff) + min(eq_before, need);
  while (m) {  // ascending positions: lowest bit first
    const int i = __ffs(m) - 1;
    m &= m - 1;
    if (out < k) {
      sel_out[out] = c0 + j0 + i;
      if (key_out) key_out[out] = stage[kidx(j0 + i)];
    }
    ++out;
  }
}

__global__ void __launch_bounds__(NT, 2) pool_topk_kernel(const TopkP p) {
  // Programmatic dependent launch: the gather kernel may start launching (its CTAs take
  // SM slots as these exit, and wait until this grid has completed); this grid waits for
  // the kernel that wrote the votes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint32_t sm[];
  uint32_t *tot = sm + SM_TOT;
  int *misc = reinterpret_cast<int *>(sm + SM_MISC);  // [0] prefix, [1] need, [2..] warp eq, [2+NWARP..] warp gt
  const int u = blockIdx.x;
  const int n = p.n_cand;
  const bool in_smem = n <= SMEM_KEYS_MAX;
  uint32_t *kb = in_smem ? sm + SM_KEYS : p.kglobal + (size_t)u * key_words(n);
  const float *v = p.votes + (size_t)u * p.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = p.half;
  const bool avg = p.avg != 0;                  // CTA-uniform
  const float pad = avg ? 0.f : -INFINITY;      // value beyond both ends of the candidates
  const float inv = 1.f / (float)(2 * h + 1);

  // phase 0: pooled keys u_j = max(v[j-h .. j+h]) cut at the candidate range (or the
  // window average with zero padding).  The
  // votes are staged through shared memory (coalesced, read once from L2): all of them
  // at once into the key array when it is in shared memory (each thread keeps its
  // pooled values in registers until every window has been read), else in chunks.
  // (pool kernel 7 over at most NT * RUN candidates runs in pool_topk_gather_kernel)
  if (2 * h < CHUNK / 2) {
    float *stage = reinterpret_cast<float *>(sm + SM_HIST);
    const int step = CHUNK - 2 * h;
    for (int c0 = 0; c0 < n; c0 += step) {
      const int lo = c0 - h;
      for (int i1 = tid; i1 < CHUNK; i1 += 8 * NT) {
        float t8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = lo + i1 + e * NT;
          t8[e] = (i1 + e * NT < CHUNK && j >= 0 && j < n) ? __ldg(v + j) : pad;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (i1 + e * NT < CHUNK) stage[i1 + e * NT] = t8[e];
      }
      __syncthreads();
      const int cnt = min(step, n - c0);
      for (int i = tid; i < cnt; i += NT) {
        float m = stage[i];
        if (avg) {
          for (int t = 1; t <= 2 * h; ++t) m += stage[i + t];
          m *= inv;
        } else {
          for (int t = 1; t <= 2 * h; ++t) m = fmaxf(m, stage[i + t]);
        }
        kb[kidx(c0 + i)] = order_key(m);
      }
      __syncthreads();
    }
  } else {  // very wide pooling kernels: direct loads
    for (int j = tid; j < n; j += NT) {
      const int lo = max(0, j - h), hi = min(n - 1, j + h);
      float m = v[lo];
      if (avg) {  // the zeros past the ends add nothing
        for (int t = lo + 1; t <= hi; ++t) m += v[t];
        m *= inv;
      } else {
        for (int t = lo + 1; t <= hi; ++t) m = fmaxf(m, v[t]);
      }
      kb[kidx(j)] = order_key(m);
    }
  }
  if (tid == 0) {
    misc[0] = 0;      // prefix of the threshold key
    misc[1] = p.k;    // keys still to take from the current bucket
  }
  __syncthreads();

  // phase 1: radix select of the k-th largest key, four 8-bit digits from the top.
  // Each warp counts into its own histogram (no contention between warps; within a
  // warp, one shared atomic per distinct bin), then the histograms are merged.
  uint32_t mask_hi = 0;
  uint32_t *whist = sm + SM_HIST + warp * NBIN;
#pragma unroll 1
  for (int d = 0; d < 4; ++d) {
    const int sh = 24 - 8 * d;
    for (int b = lane; b < NBIN; b += 32) whist[b] = 0;
    __syncwarp();
    const uint32_t prefix = (uint32_t)misc[0];
    if (d == 0) {
      // the top digit (sign and high exponent bits) puts most keys into a few bins:
      // one atomic per distinct bin of the warp
      for (int j1 = warp * 32; j1 < n; j1 += 8 * NT) {  // eight keys in flight per thread
        uint32_t key8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = j1 + e * NT + lane;
          key8[e] = j < n ? kb[kidx(j)] : 0u;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = j1 + e * NT + lane;
          const uint32_t vm = __ballot_sync(0xffffffffu, j < n);
          if (j < n) {
            const uint32_t bin = key8[e] >> sh;
            const uint32_t grp = __match_any_sync(vm, bin);
            if (lane == __ffs(grp) - 1) atomicAdd(&whist[bin], (uint32_t)__popc(grp));
          }
        }
      }
    } else {
      // lower digits of the keys left in the bucket: spread bins, plain atomics
      // (eight keys in flight per thread: the keys may live in global memory)
      for (int j1 = warp * 32 + lane; j1 < n; j1 += 8 * NT) {
        uint32_t key8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) key8[e] = j1 + e * NT < n ? kb[kidx(j1 + e * NT)] : ~prefix;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (j1 + e * NT < n && (key8[e] & mask_hi) == prefix)
            atomicAdd(&whist[(key8[e] >> sh) & (NBIN - 1)], 1u);
      }
    }
    __syncthreads();
    for (int b = tid; b < NBIN; b += NT) {
      uint32_t s = 0;
#pragma unroll 4
      for (int w = 0; w < NWARP; ++w) s += sm[SM_HIST + w * NBIN + b];
      tot[b] = s;
    }
    __syncthreads();
    if (warp == 0) {
      const int need = misc[1];
      constexpr int per = NBIN / 32;
      // lane l owns bins [l*per, (l+1)*per); sum, then suffix sums from the top lane
      uint32_t s = 0;
#pragma unroll
      for (int b = 0; b < per; ++b) s += tot[lane * per + b];
      uint32_t incl = s;  // keys in bins owned by this lane and every higher lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += t;
      }
      const uint32_t above = incl - s;  // keys in bins owned by higher lanes
      const bool mine = above < (uint32_t)need && (uint32_t)need <= above + s;
      if (mine) {
        uint32_t acc = above;
        for (int b = per - 1; b >= 0; --b) {
          const uint32_t hb = tot[lane * per + b];
          if (acc + hb >= (uint32_t)need) {
            misc[0] = (int)(prefix | ((uint32_t)(lane * per + b) << sh));
            misc[1] = need - (int)acc;
            break;
          }
          acc += hb;
        }
      }
    }
    mask_hi |= (uint32_t)(NBIN - 1) << sh;
    __syncthreads();
  }
  const uint32_t T = (uint32_t)misc[0];
  const int need = misc[1];

  // phase 2: compaction in position order.  Positions go in super-chunks of NT * RUN;
  // within one, thread t owns the run [t*RUN, (t+1)*RUN): it counts its keys above and
  // equal to the threshold, a block-wide exclusive scan gives its output offset, and it
  // writes its chosen positions (ties: the first `need` equal keys by position).
  int32_t *sel = p.sel + (size_t)u * p.cap;
  int *wsum = misc + 2;  // per-warp totals of the packed counts
  int gt_base = 0, eq_base = 0;
  for (int c0 = 0; c0 < n; c0 += NT * RUN) {
    const int j0 = c0 + tid * RUN;
    int gt = 0, eq = 0;
#pragma unroll 8
    for (int i = 0; i < RUN; ++i) {
      const int j = j0 + i;
      const uint32_t key = j < n ? kb[kidx(j)] : 0u;
      gt += (j < n && key > T) ? 1 : 0;
      eq += (j < n && key == T) ? 1 : 0;
    }
    // exclusive scan of (gt | eq << 16) over the block
    const int packed = gt | (eq << 16);
    int incl = packed;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int wbase = 0, total = 0;
    for (int w2 = 0; w2 < NWARP; ++w2) {
      const int x = wsum[w2];
      if (w2 < warp) wbase += x;
      total += x;
    }
    const int excl = wbase + incl - packed;
    int gt_before = gt_base + (excl & 0xffff), eq_before = eq_base + (excl >> 16);
    if (gt + eq > 0) {
      int out = gt_before + min(eq_before, need);
#pragma unroll 8
      for (int i = 0; i < RUN; ++i) {
        const int j = j0 + i;
        const uint32_t key = j < n ? kb[kidx(j)] : 0u;
        const bool take = j < n && (key > T || (key == T && eq_before++ < need));
        if (take) {
          if (out < p.k) sel[out] = j;
          ++out;
        }
      }
    }
    gt_base += total & 0xffff;
    eq_base += total >> 16;
    __syncthreads();  // wsum is rewritten by the next super-chunk
  }
}

struct GatherP {
  const int32_t *sel;      // [U, cap] chosen prefix positions (first k)
  const float *votes;      // [U, L] or null
  const uint4 *k, *v;      // [U, L, D]
  uint4 *ko, *vo;          // [U, cap, D]
  int32_t *pos_out;        // [U, cap]
  int32_t *n_valid_out;    // [U]
  float *kept;             // [U, cap] or null
  int L, cap, k_pick, n_keep, keep_window, identity, row_vecs;  // row_vecs = D / 8
  uint32_t *status;
};

// grid (U, ceil(cap / 32)); 256 threads; each CTA fills 32 rows of one unit.
__global__ void __launch_bounds__(256) gather_kernel(const GatherP p) {
  // programmatic dependent launch: wait for the kernel that wrote the positions / votes
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int u = blockIdx.x;  // units on x: more than 65535 of them fit
  const int r0 = blockIdx.y * 32;
  __shared__ int spos[32];
  if (threadIdx.x < 32) {
    const int s = r0 + threadIdx.x;
    int pos = -1;
    if (s < p.n_keep) {
      if (p.identity) pos = s;
      else if (s < p.k_pick) pos = p.sel[(size_t)u * p.cap + s];
      else pos = p.L - p.keep_window + (s - p.k_pick);
      if (pos < 0 || pos >= p.L) {  // never expected: keep every access in bounds
        set_status(p.status, KVC_DEV_BAD_STATE);
        pos = -1;
      }
    }
    spos[threadIdx.x] = pos;
    if (s < p.cap) {
      p.pos_out[(size_t)u * p.cap + s] = pos;
      if (p.kept) p.kept[(size_t)u * p.cap + s] = pos >= 0 ? p.votes[(size_t)u * p.L + pos] : 0.f;
    }
    if (blockIdx.y == 0 && threadIdx.x == 0) p.n_valid_out[u] = p.n_keep;
  }
  __syncthreads();
  const int rv = p.row_vecs;
  for (int e = threadIdx.x; e < 32 * rv; e += 256) {
    const int r = e / rv, c = e - r * rv;
    const int pos = spos[r];
    if (pos < 0) continue;
    const size_t src = ((size_t)u * p.L + pos) * rv + c;
    const size_t dst = ((size_t)u * p.cap + r0 + r) * rv + c;
    const uint4 kv = __ldg(p.k + src);
    const uint4 vv = __ldg(p.v + src);
    p.ko[dst] = kv;
    p.vo[dst] = vv;
  }
}

// The gather of one unit by a whole CTA, from its chosen positions spos[0..k_pick) (shared
// memory): every cache row's position (-1 past n_keep), the kept scores, n_valid, and the
// kept K/V rows in 16-byte pieces with eight loads in flight per thread.
__device__ __forceinline__ void gather_unit(const GatherP &gp, int u, const int32_t *spos) {
  const int tid = threadIdx.x;
  // positions of every cache row (-1 past n_keep), the kept scores, n_valid
  for (int r = tid; r < gp.cap; r += NT) {
    int pos = -1;
    if (r < gp.n_keep) {
      pos = r < gp.k_pick ? spos[r] : gp.L - gp.keep_window + (r - gp.k_pick);
      if (pos < 0 || pos >= gp.L) {  // never expected: keep every access in bounds
        set_status(gp.status, KVC_DEV_BAD_STATE);
        pos = -1;
      }
    }
    gp.pos_out[(size_t)u * gp.cap + r] = pos;
    if (gp.kept) gp.kept[(size_t)u * gp.cap + r] = pos >= 0 ? gp.votes[(size_t)u * gp.L + pos] : 0.f;
  }
  if (tid == 0) gp.n_valid_out[u] = gp.n_keep;
  // the kept rows: 16-byte pieces, eight loads in flight per thread
  const int rv = gp.row_vecs, rvs = rv == 16 ? 4 : 3;  // D / 8 = 16 or 8 pieces a row
  const int total = gp.n_keep * rv;
  for (int e0 = tid; e0 < total; e0 += 4 * NT) {
    uint4 kk[4], vv[4];
    size_t dst[4];
    bool ok[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + j * NT;
      ok[j] = e < total;
      dst[j] = 0;
      if (ok[j]) {
        const int r = e >> rvs, c = e & (rv - 1);
        const int pos = r < gp.k_pick ? spos[r] : gp.L - gp.keep_window + (r - gp.k_pick);
        ok[j] = pos >= 0 && pos < gp.L;
        if (ok[j]) {
          const size_t src = ((size_t)u * gp.L + pos) * rv + c;
          kk[j] = __ldg(gp.k + src);
          vv[j] = __ldg(gp.v + src);
          dst[j] = ((size_t)u * gp.cap + r) * rv + c;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (ok[j]) {
        gp.ko[dst[j]] = kk[j];
        gp.vo[dst[j]] = vv[j];
      }
  }
}

// Chunked path for long prompts (pool kernel 7): the global top-k (equal keys: lower
// position first) lies inside the union of each chunk's local top-k taken with the same
// rule, since restricted to one chunk it is a prefix of that chunk's order.  Kernel 1:
// one CTA per (chunk of CHUNK_C candidates, unit) pools its range (the windows read the
// neighbouring chunks' votes) and writes its local top-k, ascending, with their keys.
// Kernel 2: one CTA per unit selects the top k of those candidates, which are in position
// order chunk after chunk, and gathers the unit's kept rows (gather_unit).
__global__ void __launch_bounds__(NT, 2) pool_topk_chunk_kernel(const TopkP p) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint32_t sm[];
  int *misc = reinterpret_cast<int *>(sm + SM_MISC);
  const int u = blockIdx.x, c = blockIdx.y;  // units on x: more than 65535 of them fit
  const int c0 = c * CHUNK_C;
  const int nc = min(CHUNK_C, p.n_cand - c0);
  const size_t o = ((size_t)u * p.nchunks + c) * p.cap;
  select_run(p.votes + (size_t)u * p.L, c0, nc, p.n_cand, min(p.k, nc), p.avg != 0, p.half == 0,
             p.cpos + o,
             p.ckey + o, sm, sm + SM_KEYS, misc);
}

__global__ void __launch_bounds__(NT, 2) topk_merge_kernel(const TopkP p, const GatherP gp) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint32_t sm[];
  int *misc = reinterpret_cast<int *>(sm + SM_MISC);
  uint32_t *hist = sm + SM_HIST;
  const int u = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // candidates: chunk c holds min(k, its length) of them; all chunks but the last hold k
  const int last_nc = p.n_cand - (p.nchunks - 1) * CHUNK_C;
  const int total = (p.nchunks - 1) * p.k + min(p.k, last_nc);
  const int e0 = tid * RUN2;
  uint32_t key[RUN2];
  int pos[RUN2];
#pragma unroll
  for (int i = 0; i < RUN2; ++i) {
    const int e = e0 + i;
    key[i] = 0u;
    pos[i] = -1;
    if (e < total) {
      const int c = e / p.k, ii = e - c * p.k;
      const size_t o = ((size_t)u * p.nchunks + c) * p.cap + ii;
      key[i] = p.ckey[o];
      pos[i] = p.cpos[o];
    }
  }
  for (int b = tid; b < NB; b += NT) hist[b] = 0;
  __syncthreads();
  // three radix digits (bits 31-21, 20-10, 9-0) over one shared histogram, as select_run
  {
    uint32_t cur = 0xffffffffu, cnt = 0;
#pragma unroll
    for (int i = 0; i < RUN2; ++i) {
      if (e0 + i < total) {
        const uint32_t b = key[i] >> 21;
        if (b != cur) {
          if (cnt) atomicAdd(&hist[cur], cnt);
          cur = b;
          cnt = 0;
        }
        ++cnt;
      }
    }
    if (cnt) atomicAdd(&hist[cur], cnt);
  }
  __syncthreads();
  find_bin<NB / NT>(hist, misc, p.k);
  const uint32_t b0 = (uint32_t)misc[M_BIN];
  int need = misc[M_NEED];
#pragma unroll
  for (int b = 0; b < NB / NT; ++b) hist[tid * (NB / NT) + b] = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < RUN2; ++i)
    if (e0 + i < total && (key[i] >> 21) == b0) atomicAdd(&hist[(key[i] >> 10) & (NB - 1)], 1u);
  __syncthreads();
  find_bin<NB / NT>(hist, misc, need);
  const uint32_t pre = (b0 << 11) | (uint32_t)misc[M_BIN];
  need = misc[M_NEED];
#pragma unroll
  for (int b = 0; b < NB / NT; ++b) hist[tid * (NB / NT) + b] = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < RUN2; ++i)
    if (e0 + i < total && (key[i] >> 10) == pre) atomicAdd(&hist[key[i] & 1023u], 1u);
  __syncthreads();
  find_bin<1024 / NT>(hist, misc, need);
  const uint32_t T = (pre << 10) | (uint32_t)misc[M_BIN];
  need = misc[M_NEED];
  // compaction in candidate (= position) order, ties: the first `need` equal keys
  int gt = 0, eq = 0;
#pragma unroll
  for (int i = 0; i < RUN2; ++i) {
    gt += (e0 + i < total && key[i] > T) ? 1 : 0;
    eq += (e0 + i < total && key[i] == T) ? 1 : 0;
  }
  const int packed = gt | (eq << 16);
  int incl = packed;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) misc[M_CSUM + warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int w2 = 0; w2 < warp; ++w2) wbase += misc[M_CSUM + w2];
  const int excl = wbase + incl - packed;
  int eq_before = excl >> 16;
  // the chosen positions go to shared memory (the histogram region: k <= NWARP * NBIN
  // words), then the CTA gathers the unit's rows
  int32_t *spos = reinterpret_cast<int32_t *>(hist);
  if (gt + eq > 0) {
    int out = (excl & 0xffff) + min(eq_before, need);
#pragma unroll
    for (int i = 0; i < RUN2; ++i) {  // branch-free: predicated stores
      const bool valid = e0 + i < total;
      const bool eqT = valid && key[i] == T;
      const bool take = (valid && key[i] > T) || (eqT && eq_before < need);
      eq_before += eqT ? 1 : 0;
      if (take && out < p.k) spos[out] = pos[i];
      out += take ? 1 : 0;
    }
  }
  __syncthreads();
  gather_unit(gp, u, spos);
}

// The short-prompt path (pool kernel 7, candidates in registers) with the gather fused in:
// one CTA per unit selects its positions into shared memory (where the votes were staged)
// and then copies the unit's kept K/V rows itself, so the copies of early units overlap
// the selection of later ones instead of waiting for a separate gather launch.
__global__ void __launch_bounds__(NT, 2) pool_topk_gather_kernel(const TopkP p, const GatherP gp) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ uint32_t sm[];
  int *misc = reinterpret_cast<int *>(sm + SM_MISC);
  uint32_t *kb = sm + SM_KEYS;
  int32_t *spos = reinterpret_cast<int32_t *>(kb);  // the chosen positions [k]
  const int u = blockIdx.x;
  select_run(p.votes + (size_t)u * p.L, 0, p.n_cand, p.n_cand, p.k, p.avg != 0, p.half == 0, spos,
             nullptr, sm, kb, misc);
  __syncthreads();
  gather_unit(gp, u, spos);
}

bool g_topk_attr[64];
bool g_fused_attr[64];
bool g_chunk_attr[64];

}  // namespace

// The chunked path's candidates after the selected positions and the keys.
static size_t chunk_ws_offset(int units, int n, int cap) {
  size_t b = (size_t)units * cap * sizeof(int32_t);
  if (n > SMEM_KEYS_MAX) b += (size_t)units * key_words(n) * sizeof(uint32_t);
  return (b + 255) & ~(size_t)255;
}

size_t select_ws_bytes(int units, int L, int keep_window, int cap) {
  const int n = L > keep_window ? L - keep_window : 0;
  size_t b = chunk_ws_offset(units, n, cap);  // selected positions (and keys)
  if (n > CHUNK_C)                            // the chunked path's candidates
    b += (size_t)units * ((n + CHUNK_C - 1) / CHUNK_C) * cap * (sizeof(int32_t) + sizeof(uint32_t));
  return (b + 255) & ~(size_t)255;
}

cudaError_t launch_select_gather(const Ctx &c, const SelectArgs &a) {
  const int n_cand = a.L - a.keep_window;
  const int n_keep = a.identity ? a.L : a.budget;
  const int k_pick = a.identity ? 0 : a.budget - a.keep_window;
  GatherP gp;
  gp.sel = a.sel_ws;
  gp.votes = a.votes;
  gp.k = reinterpret_cast<const uint4 *>(a.k);
  gp.v = reinterpret_cast<const uint4 *>(a.v);
  gp.ko = reinterpret_cast<uint4 *>(a.k_out);
  gp.vo = reinterpret_cast<uint4 *>(a.v_out);
  gp.pos_out = a.pos_out;
  gp.n_valid_out = a.n_valid_out;
  gp.kept = a.kept_scores;
  gp.L = a.L;
  gp.cap = a.cap;
  gp.k_pick = k_pick;
  gp.n_keep = n_keep;
  gp.keep_window = a.keep_window;
  gp.identity = a.identity;
  gp.row_vecs = a.D / 8;
  gp.status = c.status;
  if (!a.identity && k_pick > 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int smem = SM_KEYS * 4 + (n_cand <= SMEM_KEYS_MAX ? key_words(n_cand) * 4 : 0);
    if (dev < 64 && !g_topk_attr[dev]) {
      cudaError_t e = cudaFuncSetAttribute(pool_topk_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (SM_KEYS + key_words(SMEM_KEYS_MAX)) * 4);
      if (e != cudaSuccess) return e;
      g_topk_attr[dev] = true;
    }
    TopkP tp;
    tp.votes = a.votes;
    tp.L = a.L;
    tp.n_cand = n_cand;
    tp.k = k_pick;
    tp.half = (a.pool_kernel - 1) / 2;
    tp.avg = a.pool_avg;
    tp.sel = a.sel_ws;
    tp.cap = a.cap;
    tp.kglobal = reinterpret_cast<uint32_t *>(a.sel_ws + (size_t)a.units * a.cap);
    tp.nchunks = (n_cand + CHUNK_C - 1) / CHUNK_C;
    uint8_t *cbase = reinterpret_cast<uint8_t *>(a.sel_ws) + chunk_ws_offset(a.units, n_cand, a.cap);
    tp.cpos = reinterpret_cast<int32_t *>(cbase);
    tp.ckey = reinterpret_cast<uint32_t *>(cbase + (size_t)a.units * tp.nchunks * a.cap * sizeof(int32_t));
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NT);
    cfg.stream = c.stream;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    // long prompts with pool kernel 7: the chunked path when the chunks' candidates fit
    // the merge's registers
    const bool reg_pool = tp.half == 3 || tp.half == 0;  // pool kernel 7 or 1
    const bool chunked = reg_pool && n_cand > CHUNK_C && tp.nchunks * k_pick <= NT * RUN2;
    // short prompts with pool kernel 7 or 1: selection and gather in one kernel
    const bool fused = reg_pool && n_cand <= CHUNK_C && (a.D == 64 || a.D == 128);
    if (fused) {
      if (dev < 64 && !g_fused_attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(pool_topk_gather_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (SM_KEYS + key_words(CHUNK_C)) * 4);
        if (e != cudaSuccess) return e;
        g_fused_attr[dev] = true;
      }
      cfg.gridDim = dim3((unsigned)a.units);
      cfg.dynamicSmemBytes = (size_t)smem;
      return cudaLaunchKernelEx(&cfg, pool_topk_gather_kernel, tp, gp);
    }
    if (chunked) {
      if (dev < 64 && !g_chunk_attr[dev]) {
        cudaError_t e = cudaFuncSetAttribute(pool_topk_chunk_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (SM_KEYS + key_words(CHUNK_C)) * 4);
        if (e != cudaSuccess) return e;
        g_chunk_attr[dev] = true;
      }
      cfg.gridDim = dim3((unsigned)a.units, (unsigned)tp.nchunks);
      cfg.dynamicSmemBytes = (size_t)(SM_KEYS + key_words(CHUNK_C)) * 4;
      cudaError_t e = cudaLaunchKernelEx(&cfg, pool_topk_chunk_kernel, tp);
      if (e != cudaSuccess) return e;
      cfg.gridDim = dim3((unsigned)a.units);
      cfg.dynamicSmemBytes = (size_t)SM_KEYS * 4;
      return cudaLaunchKernelEx(&cfg, topk_merge_kernel, tp, gp);  // with the gather
    } else {
      cfg.gridDim = dim3((unsigned)a.units);
      cfg.dynamicSmemBytes = (size_t)smem;
      cudaError_t e = cudaLaunchKernelEx(&cfg, pool_topk_kernel, tp);
      if (e != cudaSuccess) return e;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.units, (unsigned)((a.cap + 31) / 32));
  cfg.blockDim = dim3(256);
  cfg.stream = c.stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_kernel, gp);
}

}  // namespace kvc
