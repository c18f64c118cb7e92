// H2O decode step (H2O article, 処理の流れ: every decode step's attention over the
// cache updates each cached token's cumulative score; over budget, heavy hitters and
// the recent window are kept and the rest is evicted; 何を残すのか: heavy hitters +
// recent tokens).
//
// One CTA per (layer, batch, KV head) unit, one pass over the cache:
//   1. logits of the G query heads against every live row (the new token's row comes
//      straight from k_new, so nothing waits on its write);
//   2. exact softmax normaliser per head (block reduction);
//   3. o = P.V, merged over the 8 warps;
//   4. score[e] += sum_g p_g[e] (the new entry starts from 0);
//   5. if the unit now holds every slot: evict the smallest score among positions
//      <= t - n_recent, the higher position on exact ties; its slot becomes free.
// The step is HBM-bound: each live K and V row is read once (plus 12 bytes of score
// and position per entry).  Rows are read as 16-byte chunks, D/8 lanes per row, four
// loads in flight per lane, so a CTA keeps about 16 KB of each phase's rows in flight.
//
// Split step (few units, or more slots than one CTA's shared memory holds): the
// unit's live rows are cut into nsplit ranges, one CTA each.  A CTA forms its rows'
// logits (also written to the state's scratch), a partial softmax (max, normaliser) per
// head and the partial o = sum exp(logit - max) v, and publishes them; the last of the
// unit's CTAs to finish (arrival counter, no waiting) merges the output, adds every
// entry's probability to its score, evicts, writes the new token's row and resets the
// counter.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int NT = 256;
constexpr int NW = NT / 32;

struct H2OP {
  const __nv_bfloat16 *q, *k_new, *v_new;
  __nv_bfloat16 *k, *v;
  float *score;
  int32_t *pos, *n_used, *free_slot;
  __nv_bfloat16 *out;
  int32_t *evicted;
  int slots, n_recent, t;
  float c;  // log2(e)/sqrt(D)
  uint32_t *status;
};

template <int D, int G>
__global__ void __launch_bounds__(NT) h2o_step_kernel(const H2OP p) {
  extern __shared__ float hs[];
  float *qs = hs;                         // [G][D]
  float *lg = qs + G * D;                 // [G][slots]: logits, then probabilities
  float *red = lg + G * p.slots;          // [NW][G][D]
  __shared__ float wred[NW][G];
  __shared__ float gstat[2][G];           // max, sum
  __shared__ float es[NW];
  __shared__ int ep[NW], eslot[NW];

  const int u = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.slots;
  const int f = p.free_slot[u], nu = p.n_used[u];
  if (f < 0 || f >= S || nu < 0 || nu >= S || (nu < S - 1 && f != nu)) {
    if (tid == 0) set_status(p.status, KVC_DEV_BAD_STATE);
    return;
  }
  const int count = nu + 1;  // live rows 0..count-1, the new token at slot f
  const size_t rowbase = (size_t)u * S;

  for (int e = tid; e < G * D; e += NT)
    qs[e] = __bfloat162float(p.q[(size_t)u * G * D + e]) * p.c;
  __syncthreads();

  // 1. logits.  D/8 lanes per row, each with one 16-byte chunk (8 head dims), so a warp
  // load covers 32/(D/8) rows; four such loads are in flight per lane before any is used.
  constexpr int LPR = D / 8;     // lanes per row
  constexpr int RPL = 32 / LPR;  // rows per warp load
  constexpr int NB = 4;          // loads in flight per lane
  const int sub = lane / LPR, ch = lane % LPR;
  float qreg[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < 8; ++d) qreg[g][d] = qs[g * D + ch * 8 + d];
  for (int e0 = warp * RPL; e0 < count; e0 += NB * NW * RPL) {
    uint4 kw[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int e = e0 + i * NW * RPL + sub;
      if (e < count) {
        const __nv_bfloat16 *src = (e == f) ? p.k_new + (size_t)u * D : p.k + (rowbase + e) * D;
        kw[i] = *reinterpret_cast<const uint4 *>(src + ch * 8);
      }
    }
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int e = e0 + i * NW * RPL + sub;
      const float kf[8] = {bf_lo(kw[i].x), bf_hi(kw[i].x), bf_lo(kw[i].y), bf_hi(kw[i].y),
                           bf_lo(kw[i].z), bf_hi(kw[i].z), bf_lo(kw[i].w), bf_hi(kw[i].w)};
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
#pragma unroll
        for (int d = 0; d < 8; ++d) a = fmaf(qreg[g][d], kf[d], a);
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (ch == 0 && e < count) lg[g * S + e] = a;
      }
    }
  }
  __syncthreads();

  // 2. per-head max and normaliser
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float mx = -INFINITY;
    for (int e = tid; e < count; e += NT) mx = fmaxf(mx, lg[g * S + e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) wred[warp][g] = mx;
  }
  __syncthreads();
  if (tid < G) {
    float mx = -INFINITY;
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, wred[w][tid]);
    gstat[0][tid] = mx;
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float M = gstat[0][g];
    float sm = 0.f;
    for (int e = tid; e < count; e += NT) {
      const float x = ex2(lg[g * S + e] - M);
      lg[g * S + e] = x;
      sm += x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    if (lane == 0) wred[warp][g] = sm;
  }
  __syncthreads();
  if (tid < G) {
    float sm = 0.f;
    for (int w = 0; w < NW; ++w) sm += wred[w][tid];
    gstat[1][tid] = 1.f / sm;
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float inv = gstat[1][g];
    for (int e = tid; e < count; e += NT) lg[g * S + e] *= inv;
  }
  __syncthreads();

  // 3. o = P.V with the same row layout (lane: one row, 8 head dims); the RPL rows of a
  // warp load are summed by shuffles at the end
  float o[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < 8; ++d) o[g][d] = 0.f;
  for (int e0 = warp * RPL; e0 < count; e0 += NB * NW * RPL) {
    uint4 vw[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int e = e0 + i * NW * RPL + sub;
      if (e < count) {
        const __nv_bfloat16 *src = (e == f) ? p.v_new + (size_t)u * D : p.v + (rowbase + e) * D;
        vw[i] = *reinterpret_cast<const uint4 *>(src + ch * 8);
      }
    }
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int e = e0 + i * NW * RPL + sub;
      if (e < count) {
        const float vf[8] = {bf_lo(vw[i].x), bf_hi(vw[i].x), bf_lo(vw[i].y), bf_hi(vw[i].y),
                             bf_lo(vw[i].z), bf_hi(vw[i].z), bf_lo(vw[i].w), bf_hi(vw[i].w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pe = lg[g * S + e];
#pragma unroll
          for (int d = 0; d < 8; ++d) o[g][d] = fmaf(pe, vf[d], o[g][d]);
        }
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < 8; ++d) {
#pragma unroll
      for (int o2 = LPR; o2 < 32; o2 <<= 1) o[g][d] += __shfl_xor_sync(0xffffffffu, o[g][d], o2);
    }
  if (sub == 0)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int d = 0; d < 8; ++d) red[(warp * G + g) * D + ch * 8 + d] = o[g][d];

  // 4. scores; 5. eviction candidates (per-thread best, then block reduction)
  float best_s = INFINITY;
  int best_p = -1, best_e = -1;
  const int thresh = p.t - p.n_recent;
  for (int e = tid; e < count; e += NT) {
    float add = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) add += lg[g * S + e];
    const float sc = (e == f ? 0.f : p.score[rowbase + e]) + add;
    p.score[rowbase + e] = sc;
    const int ps = (e == f) ? p.t : p.pos[rowbase + e];
    if (count == S && ps <= thresh) {
      if (sc < best_s || (sc == best_s && ps > best_p)) {
        best_s = sc;
        best_p = ps;
        best_e = e;
      }
    }
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += NT) {
    const int g = e / D, d = e - g * D;
    float a = 0.f;
    for (int w = 0; w < NW; ++w) a += red[(w * G + g) * D + d];
    p.out[(size_t)u * G * D + e] = __float2bfloat16(a);
  }
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, best_s, o2);
    const int p2 = __shfl_xor_sync(0xffffffffu, best_p, o2);
    const int e2 = __shfl_xor_sync(0xffffffffu, best_e, o2);
    if (e2 >= 0 && (best_e < 0 || s2 < best_s || (s2 == best_s && p2 > best_p))) {
      best_s = s2;
      best_p = p2;
      best_e = e2;
    }
  }
  if (lane == 0) {
    es[warp] = best_s;
    ep[warp] = best_p;
    eslot[warp] = best_e;
  }
  // new token's row
  for (int e = tid; e < D / 8; e += NT) {
    reinterpret_cast<uint4 *>(p.k + (rowbase + f) * D)[e] =
        reinterpret_cast<const uint4 *>(p.k_new + (size_t)u * D)[e];
    reinterpret_cast<uint4 *>(p.v + (rowbase + f) * D)[e] =
        reinterpret_cast<const uint4 *>(p.v_new + (size_t)u * D)[e];
  }
  __syncthreads();
  if (tid == 0) {
    p.pos[rowbase + f] = p.t;
    int victim = -1, vpos = -1;
    float vs = INFINITY;
    for (int w = 0; w < NW; ++w) {
      if (eslot[w] < 0) continue;
      if (victim < 0 || es[w] < vs || (es[w] == vs && ep[w] > vpos)) {
        victim = eslot[w];
        vpos = ep[w];
        vs = es[w];
      }
    }
    if (count == S) {
      if (victim < 0) {  // cannot happen with n_recent < S; keep the state consistent
        set_status(p.status, KVC_DEV_BAD_STATE);
        victim = f == 0 ? 1 % S : 0;
        vpos = p.pos[rowbase + victim];
      }
      p.free_slot[u] = victim;
      p.n_used[u] = S - 1;
      if (p.evicted) p.evicted[u] = vpos;
    } else {
      p.free_slot[u] = count;
      p.n_used[u] = count;
      if (p.evicted) p.evicted[u] = -1;
    }
  }
}

__global__ void h2o_init_kernel(int32_t *n_used, int32_t *free_slot, const int32_t *n_valid,
                                int units) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u < units) {
    n_used[u] = n_valid[u];
    free_slot[u] = n_valid[u];
  }
}

struct H2OSplitP {
  H2OP b;
  int nsplit, chunk;   // CTAs per unit; rows per CTA at most
  int *cnt;            // [U] arrival counters (zero between calls)
  float *logit;        // [U][G][slots] scaled logits (log2 domain)
  float2 *part_ml;     // [U][nsplit][G] (max, normaliser) of each range
  float *part_o;       // [U][nsplit][G][D] unnormalised o of each range
};

template <int D, int G>
__global__ void __launch_bounds__(NT) h2o_split_kernel(const H2OSplitP sp) {
  const H2OP &p = sp.b;
  extern __shared__ float hs[];
  float *qs = hs;                         // [G][D]
  float *lg = qs + G * D;                 // [G][chunk]: this range's logits, then exp
  float *red = lg + G * sp.chunk;         // [NW][G][D]
  __shared__ float wred[NW][G];
  __shared__ float gstat[2][G];           // max, 1/sum (merged)
  __shared__ float es[NW];
  __shared__ int ep[NW], eslot[NW];
  __shared__ int last;

  const int u = blockIdx.x / sp.nsplit, r = blockIdx.x - u * sp.nsplit;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.slots;
  const int f = p.free_slot[u], nu = p.n_used[u];
  if (f < 0 || f >= S || nu < 0 || nu >= S || (nu < S - 1 && f != nu)) {
    if (tid == 0 && r == 0) set_status(p.status, KVC_DEV_BAD_STATE);
    return;  // every CTA of the unit sees the same state: none counts in
  }
  const int count = nu + 1;
  const int e0 = (int)(((long long)r * count) / sp.nsplit);
  const int e1 = (int)(((long long)(r + 1) * count) / sp.nsplit);
  const size_t rowbase = (size_t)u * S;
  float *glog = sp.logit + (size_t)u * G * S;

  for (int e = tid; e < G * D; e += NT)
    qs[e] = __bfloat162float(p.q[(size_t)u * G * D + e]) * p.c;
  __syncthreads();

  // 1. logits of rows e0..e1-1 (layout as in h2o_step_kernel; eight loads in flight per
  // lane when the query registers leave room)
  constexpr int LPR = D / 8, RPL = 32 / LPR, NB = G <= 2 ? 8 : 4;
  const int sub = lane / LPR, ch = lane % LPR;
  float qreg[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < 8; ++d) qreg[g][d] = qs[g * D + ch * 8 + d];
  for (int b0 = e0 + warp * RPL; b0 < e1; b0 += NB * NW * RPL) {
    uint4 kw[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int e = b0 + i * NW * RPL + sub;
      if (e < e1) {
        const __nv_bfloat16 *src = (e == f) ? p.k_new + (size_t)u * D : p.k + (rowbase + e) * D;
        kw[i] = *reinterpret_cast<const uint4 *>(src + ch * 8);
      }
    }
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int e = b0 + i * NW * RPL + sub;
      const float kf[8] = {bf_lo(kw[i].x), bf_hi(kw[i].x), bf_lo(kw[i].y), bf_hi(kw[i].y),
                           bf_lo(kw[i].z), bf_hi(kw[i].z), bf_lo(kw[i].w), bf_hi(kw[i].w)};
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
#pragma unroll
        for (int d = 0; d < 8; ++d) a = fmaf(qreg[g][d], kf[d], a);
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (ch == 0 && e < e1) {
          lg[g * sp.chunk + (e - e0)] = a;
          glog[(size_t)g * S + e] = a;
        }
      }
    }
  }
  __syncthreads();

  // 2. this range's max and normaliser per head
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float mx = -INFINITY;
    for (int e = tid; e < e1 - e0; e += NT) mx = fmaxf(mx, lg[g * sp.chunk + e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) wred[warp][g] = mx;
  }
  __syncthreads();
  if (tid < G) {
    float mx = -INFINITY;
    for (int w = 0; w < NW; ++w) mx = fmaxf(mx, wred[w][tid]);
    gstat[0][tid] = mx;
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float M = gstat[0][g];
    float sm = 0.f;
    for (int e = tid; e < e1 - e0; e += NT) {
      const float x = M == -INFINITY ? 0.f : ex2(lg[g * sp.chunk + e] - M);
      lg[g * sp.chunk + e] = x;
      sm += x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    if (lane == 0) wred[warp][g] = sm;
  }
  __syncthreads();
  if (tid < G) {
    float sm = 0.f;
    for (int w = 0; w < NW; ++w) sm += wred[w][tid];
    sp.part_ml[((size_t)u * sp.nsplit + r) * G + tid] = make_float2(gstat[0][tid], sm);
  }

  // 3. partial o = sum over the range of exp(logit - max) . v
  float o[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < 8; ++d) o[g][d] = 0.f;
  for (int b0 = e0 + warp * RPL; b0 < e1; b0 += NB * NW * RPL) {
    uint4 vw[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int e = b0 + i * NW * RPL + sub;
      if (e < e1) {
        const __nv_bfloat16 *src = (e == f) ? p.v_new + (size_t)u * D : p.v + (rowbase + e) * D;
        vw[i] = *reinterpret_cast<const uint4 *>(src + ch * 8);
      }
    }
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int e = b0 + i * NW * RPL + sub;
      if (e < e1) {
        const float vf[8] = {bf_lo(vw[i].x), bf_hi(vw[i].x), bf_lo(vw[i].y), bf_hi(vw[i].y),
                             bf_lo(vw[i].z), bf_hi(vw[i].z), bf_lo(vw[i].w), bf_hi(vw[i].w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pe = lg[g * sp.chunk + (e - e0)];
#pragma unroll
          for (int d = 0; d < 8; ++d) o[g][d] = fmaf(pe, vf[d], o[g][d]);
        }
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < 8; ++d) {
#pragma unroll
      for (int o2 = LPR; o2 < 32; o2 <<= 1) o[g][d] += __shfl_xor_sync(0xffffffffu, o[g][d], o2);
    }
  if (sub == 0)
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int d = 0; d < 8; ++d) red[(warp * G + g) * D + ch * 8 + d] = o[g][d];
  __syncthreads();
  for (int e = tid; e < G * D; e += NT) {
    float a = 0.f;
    for (int w = 0; w < NW; ++w) a += red[w * G * D + e];
    sp.part_o[((size_t)u * sp.nsplit + r) * G * D + e] = a;
  }

  // the last CTA of the unit to get here does the rest
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(&sp.cnt[u], 1) == sp.nsplit - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();

  // 4. merged (max, 1/normaliser) per head and the output
  if (tid < G) {
    float M = -INFINITY;
    for (int q = 0; q < sp.nsplit; ++q)
      M = fmaxf(M, __ldcg(sp.part_ml + ((size_t)u * sp.nsplit + q) * G + tid).x);
    float L = 0.f;
    for (int q = 0; q < sp.nsplit; ++q) {
      const float2 ml = __ldcg(sp.part_ml + ((size_t)u * sp.nsplit + q) * G + tid);
      L += ml.x == -INFINITY ? 0.f : ml.y * ex2(ml.x - M);
    }
    gstat[0][tid] = M;
    gstat[1][tid] = 1.f / L;
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += NT) {
    const int g = e / D;
    float a = 0.f;
    for (int q = 0; q < sp.nsplit; ++q) {
      const float2 ml = __ldcg(sp.part_ml + ((size_t)u * sp.nsplit + q) * G + g);
      if (ml.x != -INFINITY)
        a += __ldcg(sp.part_o + ((size_t)u * sp.nsplit + q) * G * D + e) * ex2(ml.x - gstat[0][g]);
    }
    p.out[(size_t)u * G * D + e] = __float2bfloat16(a * gstat[1][g]);
  }

  // 5. scores and the eviction candidate (as in h2o_step_kernel)
  float best_s = INFINITY;
  int best_p = -1, best_e = -1;
  const int thresh = p.t - p.n_recent;
  for (int e = tid; e < count; e += NT) {
    float add = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) add += ex2(__ldcg(glog + (size_t)g * S + e) - gstat[0][g]) * gstat[1][g];
    const float sc = (e == f ? 0.f : p.score[rowbase + e]) + add;
    p.score[rowbase + e] = sc;
    const int ps = (e == f) ? p.t : p.pos[rowbase + e];
    if (count == S && ps <= thresh) {
      if (sc < best_s || (sc == best_s && ps > best_p)) {
        best_s = sc;
        best_p = ps;
        best_e = e;
      }
    }
  }
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, best_s, o2);
    const int p2 = __shfl_xor_sync(0xffffffffu, best_p, o2);
    const int e2 = __shfl_xor_sync(0xffffffffu, best_e, o2);
    if (e2 >= 0 && (best_e < 0 || s2 < best_s || (s2 == best_s && p2 > best_p))) {
      best_s = s2;
      best_p = p2;
      best_e = e2;
    }
  }
  if (lane == 0) {
    es[warp] = best_s;
    ep[warp] = best_p;
    eslot[warp] = best_e;
  }
  for (int e = tid; e < D / 8; e += NT) {
    reinterpret_cast<uint4 *>(p.k + (rowbase + f) * D)[e] =
        reinterpret_cast<const uint4 *>(p.k_new + (size_t)u * D)[e];
    reinterpret_cast<uint4 *>(p.v + (rowbase + f) * D)[e] =
        reinterpret_cast<const uint4 *>(p.v_new + (size_t)u * D)[e];
  }
  __syncthreads();
  if (tid == 0) {
    p.pos[rowbase + f] = p.t;
    int victim = -1, vpos = -1;
    float vs = INFINITY;
    for (int w = 0; w < NW; ++w) {
      if (eslot[w] < 0) continue;
      if (victim < 0 || es[w] < vs || (es[w] == vs && ep[w] > vpos)) {
        victim = eslot[w];
        vpos = ep[w];
        vs = es[w];
      }
    }
    if (count == S) {
      if (victim < 0) {  // cannot happen with n_recent < S; keep the state consistent
        set_status(p.status, KVC_DEV_BAD_STATE);
        victim = f == 0 ? 1 % S : 0;
        vpos = p.pos[rowbase + victim];
      }
      p.free_slot[u] = victim;
      p.n_used[u] = S - 1;
      if (p.evicted) p.evicted[u] = vpos;
    } else {
      p.free_slot[u] = count;
      p.n_used[u] = count;
      if (p.evicted) p.evicted[u] = -1;
    }
    sp.cnt[u] = 0;
  }
}

template <int D, int G>
cudaError_t launch_split_t(const Ctx &c, const H2OArgs &a, const H2OSplitP &sp) {
  const size_t smem = ((size_t)G * D + (size_t)G * sp.chunk + (size_t)NW * G * D) * sizeof(float);
  static bool attr[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(h2o_split_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  h2o_split_kernel<D, G><<<(unsigned)((long long)a.units * sp.nsplit), NT, smem, c.stream>>>(sp);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_t(const Ctx &c, const H2OArgs &a, const H2OP &p) {
  const size_t smem = ((size_t)G * D + (size_t)G * a.slots + (size_t)NW * G * D) * sizeof(float);
  static bool attr[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(h2o_step_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  h2o_step_kernel<D, G><<<a.units, NT, smem, c.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

H2OSplitPlan plan_h2o_split(long long units, int G, int D, int slots, int num_sms) {
  H2OSplitPlan pl;
  const int nsm = num_sms > 0 ? num_sms : 1;
  // enough CTAs for eight per SM, at least 64 rows each, and few enough rows per CTA
  // that its logits fit shared memory next to the query and the reduction buffers
  long long want = (8LL * nsm + units - 1) / units;
  const long long by_rows = (slots + 63) / 64;
  if (want > by_rows) want = by_rows;
  const long long cap_rows = (200 * 1024 / 4 - 9LL * G * D) / G;  // logits per CTA that fit
  const long long need = cap_rows > 0 ? (slots + cap_rows - 1) / cap_rows : (1LL << 30);
  if (want < need) want = need;
  if (want < 1) want = 1;
  pl.nsplit = (int)want;
  pl.chunk = (slots + pl.nsplit - 1) / pl.nsplit;
  pl.feasible = cap_rows > 0 && pl.chunk <= cap_rows && units * pl.nsplit <= 0x7fffffffLL;
  size_t b = ((size_t)units * sizeof(int) + 255) & ~(size_t)255;                // counters
  b += ((size_t)units * G * slots * sizeof(float) + 255) & ~(size_t)255;        // logits
  b += ((size_t)units * pl.nsplit * G * sizeof(float2) + 255) & ~(size_t)255;   // (max, sum)
  b += ((size_t)units * pl.nsplit * G * D * sizeof(float) + 255) & ~(size_t)255;  // partial o
  pl.scratch_bytes = b;
  return pl;
}

bool h2o_single_fits(int G, int D, long long slots) {
  return ((size_t)G * D + (size_t)G * slots + (size_t)NW * G * D) * sizeof(float) <= 200 * 1024;
}

cudaError_t launch_h2o_step(const Ctx &c, const H2OArgs &a) {
  H2OP p;
  p.q = reinterpret_cast<const __nv_bfloat16 *>(a.q);
  p.k_new = reinterpret_cast<const __nv_bfloat16 *>(a.k_new);
  p.v_new = reinterpret_cast<const __nv_bfloat16 *>(a.v_new);
  p.k = reinterpret_cast<__nv_bfloat16 *>(a.k);
  p.v = reinterpret_cast<__nv_bfloat16 *>(a.v);
  p.score = a.score;
  p.pos = a.pos;
  p.n_used = a.n_used;
  p.free_slot = a.free_slot;
  p.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
  p.evicted = a.evicted;
  p.slots = a.slots;
  p.n_recent = a.n_recent;
  p.t = a.t;
  p.c = (float)(1.4426950408889634 / sqrt((double)a.D));
  p.status = c.status;
  if (a.split) {
    const H2OSplitPlan pl = plan_h2o_split(a.units, a.G, a.D, a.slots, c.num_sms);
    H2OSplitP sp;
    sp.b = p;
    sp.nsplit = pl.nsplit;
    sp.chunk = pl.chunk;
    uint8_t *w = reinterpret_cast<uint8_t *>(a.scratch);
    size_t off = 0;
    sp.cnt = reinterpret_cast<int *>(w + off);
    off += ((size_t)a.units * sizeof(int) + 255) & ~(size_t)255;
    sp.logit = reinterpret_cast<float *>(w + off);
    off += ((size_t)a.units * a.G * a.slots * sizeof(float) + 255) & ~(size_t)255;
    sp.part_ml = reinterpret_cast<float2 *>(w + off);
    off += ((size_t)a.units * pl.nsplit * a.G * sizeof(float2) + 255) & ~(size_t)255;
    sp.part_o = reinterpret_cast<float *>(w + off);
#define KVC_H2OS(DD, GG) \
  if (a.D == DD && a.G == GG) return launch_split_t<DD, GG>(c, a, sp);
    KVC_H2OS(128, 1) KVC_H2OS(128, 2) KVC_H2OS(128, 3) KVC_H2OS(128, 4)
    KVC_H2OS(128, 5) KVC_H2OS(128, 6) KVC_H2OS(128, 7) KVC_H2OS(128, 8)
    KVC_H2OS(64, 1) KVC_H2OS(64, 2) KVC_H2OS(64, 3) KVC_H2OS(64, 4)
    KVC_H2OS(64, 5) KVC_H2OS(64, 6) KVC_H2OS(64, 7) KVC_H2OS(64, 8)
#undef KVC_H2OS
    return cudaErrorInvalidValue;
  }
#define KVC_H2O(DD, GG) \
  if (a.D == DD && a.G == GG) return launch_t<DD, GG>(c, a, p);
  KVC_H2O(128, 1) KVC_H2O(128, 2) KVC_H2O(128, 3) KVC_H2O(128, 4)
  KVC_H2O(128, 5) KVC_H2O(128, 6) KVC_H2O(128, 7) KVC_H2O(128, 8)
  KVC_H2O(64, 1) KVC_H2O(64, 2) KVC_H2O(64, 3) KVC_H2O(64, 4)
  KVC_H2O(64, 5) KVC_H2O(64, 6) KVC_H2O(64, 7) KVC_H2O(64, 8)
#undef KVC_H2O
  return cudaErrorInvalidValue;
}

cudaError_t launch_h2o_init_state(const Ctx &c, int32_t *pos, int32_t *n_used,
                                  int32_t *free_slot, const int32_t *n_valid, int units,
                                  int slots) {
  (void)pos;
  (void)slots;
  h2o_init_kernel<<<(units + 255) / 256, 256, 0, c.stream>>>(n_used, free_slot, n_valid, units);
  return cudaGetLastError();
}

}  // namespace kvc
