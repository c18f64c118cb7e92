// SnapKV steps 3-4 (SnapKV article, 処理の流れ steps 3 and 4): 1D max-pool of the vote
// over the prefix candidates, per-head top-k (equal pooled votes: lower position
// first), then the gather of the kept prefix rows and the kept window into the compact
// cache.  The same code cuts H2O's prompt to heavy hitters + recent window (pool 1).
//
// pool_topk_kernel: one CTA (1024 threads) per unit.
//   phase 0  pooled vote u_j = max(v[j-h .. j+h]) (cut at the candidate range) turned
//            into an order-preserving uint32 key, kept in shared memory (global
//            workspace when the candidate range does not fit);
//   phase 1  radix select of the k-th largest key: three histogram passes over the
//            11 + 11 + 10 key bits, each narrowing the bucket that holds it;
//   phase 2  stream compaction in position order: keys above the threshold, and the
//            first `need` keys equal to it (exact lower-position tie rule), written as
//            ascending positions.
// gather_kernel: 16-byte vectorised copy of the kept K/V rows, positions, scores.
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int NT = 1024;        // threads of pool_topk_kernel
constexpr int NWARP = NT / 32;
constexpr int SMEM_KEYS_MAX = 50 * 1024;  // candidates kept in shared memory

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct TopkP {
  const float *votes;  // [U, L]
  int L, n_cand, k, half;  // half = (pool kernel - 1) / 2
  int32_t *sel;        // [U, cap] output positions
  int cap;
  uint32_t *kglobal;   // [U, n_cand] keys when they do not fit in shared memory
};

__global__ void __launch_bounds__(NT, 1) pool_topk_kernel(const TopkP p) {
  extern __shared__ uint32_t sm[];
  uint32_t *hist = sm;                 // 2048 bins
  int *misc = reinterpret_cast<int *>(sm + 2048);   // [0] prefix, [1] need, [2..33] warp eq, [34..65] warp take
  uint32_t *keys = sm + 2048 + 128;    // n_cand keys (shared path)
  const int u = blockIdx.x;
  const int n = p.n_cand;
  const bool in_smem = n <= SMEM_KEYS_MAX;
  uint32_t *kb = in_smem ? keys : p.kglobal + (size_t)u * n;
  const float *v = p.votes + (size_t)u * p.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // phase 0: pooled keys
  for (int j = tid; j < n; j += NT) {
    const int lo = max(0, j - p.half), hi = min(n - 1, j + p.half);
    float m = v[lo];
    for (int t = lo + 1; t <= hi; ++t) m = fmaxf(m, v[t]);
    kb[j] = order_key(m);
  }
  if (tid == 0) {
    misc[0] = 0;      // prefix of the threshold key
    misc[1] = p.k;    // keys still to take from the current bucket
  }
  __syncthreads();

  // phase 1: radix select of the k-th largest key
  uint32_t mask_hi = 0;
  const int shifts[3] = {21, 10, 0};
  const int widths[3] = {11, 11, 10};
#pragma unroll 1
  for (int d = 0; d < 3; ++d) {
    const int sh = shifts[d], w = widths[d], nb = 1 << w;
    for (int i = tid; i < nb; i += NT) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = (uint32_t)misc[0];
    // warp-aggregated counting: one shared atomic per distinct bin per warp (the first
    // digit puts most keys into a handful of bins)
    for (int j0 = warp * 32; j0 < n; j0 += NT) {
      const int j = j0 + lane;
      const uint32_t key = j < n ? kb[j] : 0u;
      const bool valid = j < n && (key & mask_hi) == prefix;
      const uint32_t vm = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t bin = (key >> sh) & (nb - 1);
        const uint32_t grp = __match_any_sync(vm, bin);
        if (lane == __ffs(grp) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(grp));
      }
    }
    __syncthreads();
    if (warp == 0) {
      const int need = misc[1];
      const int per = nb / 32;
      // lane l owns bins [l*per, (l+1)*per); sum, then suffix sums from the top lane
      uint32_t s = 0;
      for (int b = 0; b < per; ++b) s += hist[lane * per + b];
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
          const uint32_t h = hist[lane * per + b];
          if (acc + h >= (uint32_t)need) {
            misc[0] = (int)(prefix | ((uint32_t)(lane * per + b) << sh));
            misc[1] = need - (int)acc;
            break;
          }
          acc += h;
        }
      }
    }
    mask_hi |= (uint32_t)(nb - 1) << sh;
    __syncthreads();
  }
  const uint32_t T = (uint32_t)misc[0];
  const int need = misc[1];

  // phase 2: compaction in position order; warp w owns positions [w*blk, (w+1)*blk)
  const int blk = ((n + NWARP - 1) / NWARP + 31) & ~31;
  const int b0 = warp * blk, b1 = min(n, b0 + blk);
  int eq_cnt = 0, gt_cnt = 0;
  for (int j0 = b0; j0 < b1; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t key = j < b1 ? kb[j] : 0u;
    eq_cnt += __popc(__ballot_sync(0xffffffffu, j < b1 && key == T));
    gt_cnt += __popc(__ballot_sync(0xffffffffu, j < b1 && key > T));
  }
  if (lane == 0) {
    misc[2 + warp] = eq_cnt;
    misc[34 + warp] = gt_cnt;
  }
  __syncthreads();
  int eq_base = 0, out_base = 0;
  for (int w2 = 0; w2 < warp; ++w2) {
    const int e = misc[2 + w2], g = misc[34 + w2];
    const int take_eq = max(0, min(e, need - eq_base));
    out_base += g + take_eq;
    eq_base += e;
  }
  int32_t *sel = p.sel + (size_t)u * p.cap;
  const uint32_t lt = (1u << lane) - 1u;
  for (int j0 = b0; j0 < b1; j0 += 32) {
    const int j = j0 + lane;
    const uint32_t key = j < b1 ? kb[j] : 0u;
    const bool eq = j < b1 && key == T, gt = j < b1 && key > T;
    const uint32_t eqm = __ballot_sync(0xffffffffu, eq);
    const int rank = eq_base + __popc(eqm & lt);
    const bool take = gt || (eq && rank < need);
    const uint32_t tm = __ballot_sync(0xffffffffu, take);
    const int slot = out_base + __popc(tm & lt);
    if (take && slot < p.k) sel[slot] = j;
    eq_base += __popc(eqm);
    out_base += __popc(tm);
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

// grid (ceil(cap / 32), U); 256 threads; each CTA fills 32 rows of one unit.
__global__ void __launch_bounds__(256) gather_kernel(const GatherP p) {
  const int u = blockIdx.y;
  const int r0 = blockIdx.x * 32;
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
    if (blockIdx.x == 0 && threadIdx.x == 0) p.n_valid_out[u] = p.n_keep;
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

bool g_topk_attr[64];

}  // namespace

size_t select_ws_bytes(int units, int L, int keep_window, int cap) {
  const size_t n = (size_t)(L > keep_window ? L - keep_window : 0);
  size_t b = (size_t)units * cap * sizeof(int32_t);               // selected positions
  if (n > (size_t)SMEM_KEYS_MAX) b += (size_t)units * n * sizeof(uint32_t);  // keys
  return (b + 255) & ~(size_t)255;
}

cudaError_t launch_select_gather(const Ctx &c, const SelectArgs &a) {
  const int n_cand = a.L - a.keep_window;
  const int n_keep = a.identity ? a.L : a.budget;
  const int k_pick = a.identity ? 0 : a.budget - a.keep_window;
  if (!a.identity && k_pick > 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int smem = (2048 + 128) * 4 + (n_cand <= SMEM_KEYS_MAX ? n_cand * 4 : 0);
    if (dev < 64 && !g_topk_attr[dev]) {
      cudaError_t e = cudaFuncSetAttribute(pool_topk_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (2048 + 128 + SMEM_KEYS_MAX) * 4);
      if (e != cudaSuccess) return e;
      g_topk_attr[dev] = true;
    }
    TopkP tp;
    tp.votes = a.votes;
    tp.L = a.L;
    tp.n_cand = n_cand;
    tp.k = k_pick;
    tp.half = (a.pool_kernel - 1) / 2;
    tp.sel = a.sel_ws;
    tp.cap = a.cap;
    tp.kglobal = reinterpret_cast<uint32_t *>(a.sel_ws + (size_t)a.units * a.cap);
    pool_topk_kernel<<<a.units, NT, smem, c.stream>>>(tp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
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
  dim3 grid((a.cap + 31) / 32, a.units);
  gather_kernel<<<grid, 256, 0, c.stream>>>(gp);
  return cudaGetLastError();
}

}  // namespace kvc
