// Decode attention over a compact (SnapKV) or sink + ring (StreamingLLM) cache: for
// each query head of each (layer, batch, KV head) unit, o = softmax(q . K_c^T / sqrt(D))
// . V_c over the unit's first n rows (SnapKV article, 推論方法: decoding reads only the
// compressed cache; StreamingLLM article, 推論の流れ: attention over sink and recent
// tokens only).  An optional append adds the step's new K/V row first (fused: the CTA
// whose tile holds the new row patches it in shared memory from k_new/v_new, and the
// unit's finishing CTA writes it to the cache, its position and the new n_valid).
//
// Design (sm_103a, HBM-bound: every cached K/V byte is read once):
// * split-K over the rows: CTA (split s, unit u) covers rows [s*C, (s+1)*C) in tiles of
//   64 rows; warp 0 streams K and V tiles into a 3-stage shared-memory ring with TMA
//   (128-byte swizzle, one mbarrier per stage), warps 1-4 compute;
// * logits: two threads per row (half a head-dim each, conflict-free reads of the
//   swizzled tile), q in shared memory pre-scaled by log2(e)/sqrt(D), fp32 FMA;
// * online softmax per warp (16 rows per tile), P.V with lanes over the head dim;
// * the four warps' states merge in shared memory; with several splits the partial
//   (m, l, o) goes to the workspace and the last CTA of the unit (atomic counter, no
//   waiting) merges all splits and writes the bf16 output, resetting the counter.
//   The counters live in a fixed 256 KB header of the workspace (one int per unit, at
//   most 65535 units) that is zero between calls, whatever the shapes of the calls.
#include <math.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int ROWS = 64;     // rows per tile
constexpr int NST = 3;       // ring depth
constexpr int NCW = 4;       // compute warps
constexpr int NTH = 32 * (NCW + 1);

template <int D, int G>
struct DGeo {
  static constexpr int KB = D / 64;
  static constexpr int KBLK = ROWS * 128;        // bytes of one k-block of a tile
  static constexpr int TB = KB * KBLK;           // bytes of one K (or V) tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = NST * TB;
  static constexpr int OFF_Q = 2 * NST * TB;     // fp32 q [G][D]
  static constexpr int OFF_RED = OFF_Q + G * D * 4;  // fp32 [NCW][G][D + 2]
  static constexpr int OFF_BAR = OFF_RED + NCW * G * (D + 2) * 4;
  static constexpr int SMEM = OFF_BAR + 128 + 1024;
  static constexpr int DV = D / 32;              // head-dim elements per lane in P.V
};

struct DecP {
  const __nv_bfloat16 *q;
  float c;                 // log2(e)/sqrt(D)
  int32_t *n_valid;        // [U] or null
  const __nv_bfloat16 *k_new, *v_new;  // [U, D] or null (append)
  __nv_bfloat16 *kc, *vc;  // the caches [U, cap, D] (append writes one row)
  int32_t *pos;            // [U, cap] or null
  int new_pos;
  int n_uniform, cap, chunk, splits;
  __nv_bfloat16 *out;
  float2 *part_ml;         // [U][S][G]
  float *part_o;           // [U][S][G][D]
  int *cnt;                // [U]
  uint32_t *status;
  unsigned long long timeout;
};

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

template <int D, int G>
__global__ void __launch_bounds__(NTH) decode_kernel(const __grid_constant__ CUtensorMap tk,
                                                     const __grid_constant__ CUtensorMap tv,
                                                     const DecP p) {
  using Gm = DGeo<D, G>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  float *qs = reinterpret_cast<float *>(smem + Gm::OFF_Q);
  float *red = reinterpret_cast<float *>(smem + Gm::OFF_RED);
  const uint32_t bar = sb + Gm::OFF_BAR;  // full[NST] at +0, empty[NST] at +32
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + 64);
  volatile int *last_flag = reinterpret_cast<volatile int *>(smem + Gm::OFF_BAR + 68);

  const int u = blockIdx.y, s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Abort ab{abort_flag, p.status, p.timeout};

  int n = p.n_valid ? p.n_valid[u] : p.n_uniform;
  if (n > p.cap || n < 0) {
    if (threadIdx.x == 0) set_status(p.status, KVC_DEV_BAD_STATE);
    n = n < 0 ? 0 : p.cap;
  }
  const int n_old = n;
  int arow = -1;  // row of the appended token, -1 if none
  if (p.k_new) {
    if (n < p.cap) {
      arow = n;
      n = n + 1;
    } else if (s == 0 && threadIdx.x == 0) {
      set_status(p.status, KVC_DEV_CACHE_FULL);
    }
  }
  const int r_begin = s * p.chunk;
  const int r_end = min(n, r_begin + p.chunk);
  const int ntiles = r_end > r_begin ? (r_end - r_begin + ROWS - 1) / ROWS : 0;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar + 8 * i, 1);
      mbar_init(bar + 32 + 8 * i, NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------------------- TMA producer ----------------------------
    if (lane == 0 && ntiles > 0) {
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int i = 0;
      for (; i < ntiles; ++i) {
        const int st = i % NST, use = i / NST;
        if (!ab.wait(bar + 32 + 8 * st, (use & 1) ^ 1)) break;
        mbar_arrive_expect_tx(bar + 8 * st, 2 * Gm::TB);
        const int row = u * p.cap + r_begin + i * ROWS;
        for (int kb = 0; kb < Gm::KB; ++kb) {
          tma_load_2d(sb + Gm::OFF_K + st * Gm::TB + kb * Gm::KBLK, &tk, kb * 64, row, bar + 8 * st);
          tma_load_2d(sb + Gm::OFF_V + st * Gm::TB + kb * Gm::KBLK, &tv, kb * 64, row, bar + 8 * st);
        }
      }
      for (int st = 0; st < NST; ++st) {  // drain
        const int cnt = i / NST + (st < i % NST ? 1 : 0);
        if (cnt > 0) mbar_wait_bounded(bar + 8 * st, (cnt - 1) & 1, p.timeout);
      }
    }
  } else {
    // ------------------------------ compute ------------------------------
    const int cw = warp - 1;                 // 0..3
    const int t = threadIdx.x - 32;          // 0..127
    // q (bf16) -> fp32 pre-scaled
    for (int e = t; e < G * D; e += 128)
      qs[e] = __bfloat162float(p.q[(size_t)u * G * D + e]) * p.c;
    named_bar(1, 128);

    const int r = t >> 1;        // row of the tile for the logit phase
    const int h = t & 1;         // which half of the head dim
    constexpr int NCH = D / 16;  // 16-byte chunks per half row
    float m[G], l[G], o[G][Gm::DV];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int d = 0; d < Gm::DV; ++d) o[g][d] = 0.f;
    }
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % NST;
      const bool got = __all_sync(0xffffffffu, ok && ab.wait(bar + 8 * st, (i / NST) & 1));
      ok = got;
      const uint8_t *ktp = smem + Gm::OFF_K + st * Gm::TB;
      const uint8_t *vtp = smem + Gm::OFF_V + st * Gm::TB;
      const int arr = arow - (r_begin + i * ROWS);  // the appended row in this tile?
      const bool patched = arow >= 0 && arr >= 0 && arr < ROWS;  // same for the whole CTA
      if (patched) {
        // every compute thread reaches this barrier, whether or not its wait succeeded
        if (got && t < 2 * (D / 8)) {
          const int which = t / (D / 8), cidx = t % (D / 8);
          const int kb = cidx >> 3, ci = cidx & 7;
          uint8_t *dst = smem + (which ? Gm::OFF_V : Gm::OFF_K) + st * Gm::TB + kb * Gm::KBLK +
                         arr * 128 + ((ci ^ (arr & 7)) << 4);
          const __nv_bfloat16 *src = (which ? p.v_new : p.k_new) + (size_t)u * D + cidx * 8;
          *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
        }
        named_bar(1, 128);
      }
      if (!got) continue;
      // ---- logits: this thread's half row ----
      float acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc[g] = 0.f;
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int cc = (D == 128) ? ((c + 4 * h) & 7) : c;      // rotation: conflict-free
        const int chunk = h * NCH + cc;                          // 16-byte chunk in the row
        const int kb = chunk >> 3, ci = chunk & 7;
        const uint4 w = *reinterpret_cast<const uint4 *>(ktp + kb * Gm::KBLK + r * 128 +
                                                          ((ci ^ (r & 7)) << 4));
        const float kf[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y),
                             bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
        const int d0 = chunk * 8;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4 *>(qs + g * D + d0);
          const float4 qb = *reinterpret_cast<const float4 *>(qs + g * D + d0 + 4);
          acc[g] = fmaf(qa.x, kf[0], acc[g]);
          acc[g] = fmaf(qa.y, kf[1], acc[g]);
          acc[g] = fmaf(qa.z, kf[2], acc[g]);
          acc[g] = fmaf(qa.w, kf[3], acc[g]);
          acc[g] = fmaf(qb.x, kf[4], acc[g]);
          acc[g] = fmaf(qb.y, kf[5], acc[g]);
          acc[g] = fmaf(qb.z, kf[6], acc[g]);
          acc[g] = fmaf(qb.w, kf[7], acc[g]);
        }
      }
      const bool rvalid = r_begin + i * ROWS + r < r_end;
      float pr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float x = acc[g] + __shfl_xor_sync(0xffffffffu, acc[g], 1);
        x = rvalid ? x : -INFINITY;
        float mx = x;
#pragma unroll
        for (int o2 = 2; o2 < 32; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float mnew = fmaxf(m[g], mx);
        float scale = 1.f, pe = 0.f;
        if (mnew != -INFINITY) {
          scale = ex2(m[g] - mnew);
          pe = ex2(x - mnew);
        }
        float ps = (h == 0) ? pe : 0.f;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o2);
        l[g] = l[g] * scale + ps;
        m[g] = mnew;
#pragma unroll
        for (int d = 0; d < Gm::DV; ++d) o[g][d] *= scale;
        pr[g] = pe;
      }
      // ---- P.V: lanes over the head dim, the warp's 16 rows ----
#pragma unroll 4
      for (int i2 = 0; i2 < 16; ++i2) {
        const int rr = cw * 16 + i2;
        float vf[Gm::DV];
        if (D == 128) {
          const int chunk = lane >> 1, kb = chunk >> 3, ci = chunk & 7;
          const uint2 w = *reinterpret_cast<const uint2 *>(vtp + kb * Gm::KBLK + rr * 128 +
                                                           ((ci ^ (rr & 7)) << 4) + (lane & 1) * 8);
          vf[0] = bf_lo(w.x);
          vf[1] = bf_hi(w.x);
          vf[2 % Gm::DV] = bf_lo(w.y);
          vf[3 % Gm::DV] = bf_hi(w.y);
        } else {
          const int ci = lane >> 2;
          const uint32_t w = *reinterpret_cast<const uint32_t *>(vtp + rr * 128 + ((ci ^ (rr & 7)) << 4) +
                                                                 (lane & 3) * 4);
          vf[0] = bf_lo(w);
          vf[1 % Gm::DV] = bf_hi(w);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pv = __shfl_sync(0xffffffffu, pr[g], 2 * i2);
#pragma unroll
          for (int d = 0; d < Gm::DV; ++d) o[g][d] = fmaf(pv, vf[d], o[g][d]);
        }
      }
      // generic-proxy writes to this stage must be ordered before the next TMA into it
      if (patched) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + 32 + 8 * st);
    }
    // ---- merge the four warps ----
    float *mine = red + cw * G * (D + 2);
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int d = 0; d < Gm::DV; ++d) mine[g * (D + 2) + lane * Gm::DV + d] = o[g][d];
      if (lane == 0) {
        mine[g * (D + 2) + D] = m[g];
        mine[g * (D + 2) + D + 1] = l[g];
      }
    }
    named_bar(1, 128);
    const bool direct = p.splits == 1;
    for (int e = t; e < G * D; e += 128) {
      const int g = e / D, d = e - g * D;
      float M = -INFINITY;
      for (int w2 = 0; w2 < NCW; ++w2) M = fmaxf(M, red[(w2 * G + g) * (D + 2) + D]);
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
        for (int w2 = 0; w2 < NCW; ++w2) {
          const float* src = red + (w2 * G + g) * (D + 2);
          const float f = ex2(src[D] - M);
          L += src[D + 1] * f;
          O += src[d] * f;
        }
      }
      if (direct) {
        p.out[(size_t)u * G * D + e] = __float2bfloat16(L > 0.f ? O / L : 0.f);
        if (e < D / 8 && arow >= 0) append_row<D>(p, u, arow, n_old, e);
      } else {
        p.part_o[(((size_t)u * p.splits + s) * G + g) * D + d] = O;
        if (d == 0) p.part_ml[((size_t)u * p.splits + s) * G + g] = make_float2(M, L);
      }
    }
    if (!direct) {
      __threadfence();
      named_bar(1, 128);
      if (t == 0) *last_flag = (atomicAdd(&p.cnt[u], 1) == p.splits - 1);
      named_bar(1, 128);
      if (*last_flag) {
        __threadfence();
        for (int e = t; e < G * D; e += 128) {
          const int g = e / D, d = e - g * D;
          float M = -INFINITY;
          for (int s2 = 0; s2 < p.splits; ++s2)
            M = fmaxf(M, __ldcg(p.part_ml + ((size_t)u * p.splits + s2) * G + g).x);
          float L = 0.f, O = 0.f;
          if (M != -INFINITY) {
            for (int s2 = 0; s2 < p.splits; ++s2) {
              const float2 ml = __ldcg(p.part_ml + ((size_t)u * p.splits + s2) * G + g);
              const float f = ex2(ml.x - M);
              L += ml.y * f;
              O += __ldcg(p.part_o + (((size_t)u * p.splits + s2) * G + g) * D + d) * f;
            }
          }
          p.out[(size_t)u * G * D + e] = __float2bfloat16(L > 0.f ? O / L : 0.f);
        }
        if (arow >= 0)
          for (int e = t; e < D / 8; e += 128) append_row<D>(p, u, arow, n_old, e);
        if (t == 0) p.cnt[u] = 0;
      }
    }
  }
}

template <int D, int G>
cudaError_t launch_t(const Ctx &c, const DecodeArgs &a, const DecP &p, dim3 grid) {
  static bool attr[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DGeo<D, G>::SMEM);
    if (e != cudaSuccess) return e;
    attr[dev] = true;
  }
  CUtensorMap tk, tv;
  if (!encode_rows_map(&tk, a.k_cache, (uint64_t)a.units * a.cap, D, ROWS)) return cudaErrorInvalidValue;
  if (!encode_rows_map(&tv, a.v_cache, (uint64_t)a.units * a.cap, D, ROWS)) return cudaErrorInvalidValue;
  decode_kernel<D, G><<<grid, NTH, DGeo<D, G>::SMEM, c.stream>>>(tk, tv, p);
  return cudaGetLastError();
}

// splits and chunk: enough CTAs to fill the GPU about twice over, chunks of whole tiles
void plan_splits(int units, int n_max, int num_sms, int *splits, int *chunk) {
  const int max_splits = n_max > 0 ? (n_max + ROWS - 1) / ROWS : 1;
  const int target = 4 * num_sms;
  int S = (target + units - 1) / units;
  if (S < 1) S = 1;
  if (S > max_splits) S = max_splits;
  int C = n_max > 0 ? (n_max + S - 1) / S : ROWS;
  C = (C + ROWS - 1) / ROWS * ROWS;
  *chunk = C;
  *splits = n_max > 0 ? (n_max + C - 1) / C : 1;
}

}  // namespace

constexpr size_t CNT_HEADER = 65536 * sizeof(int);  // per-unit counters, zero between calls

size_t decode_ws_bytes(int units, int G, int D, int cap, int num_sms) {
  const size_t smax = (size_t)(cap > 0 ? (cap + ROWS - 1) / ROWS : 1);
  size_t b = CNT_HEADER;
  b += (size_t)units * smax * G * sizeof(float2);
  b += (size_t)units * smax * G * D * sizeof(float);
  (void)num_sms;
  return (b + 255) & ~(size_t)255;
}

cudaError_t launch_decode(const Ctx &c, const DecodeArgs &a) {
  const int n_max = a.n_valid ? a.cap : a.n_uniform;
  int splits, chunk;
  plan_splits(a.units, n_max, c.num_sms, &splits, &chunk);
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
  p.chunk = chunk;
  p.splits = splits;
  p.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
  uint8_t *w = reinterpret_cast<uint8_t *>(a.ws);
  p.cnt = reinterpret_cast<int *>(w);
  p.part_ml = reinterpret_cast<float2 *>(w + CNT_HEADER);
  p.part_o = reinterpret_cast<float *>(w + CNT_HEADER + (size_t)a.units * smax * a.G * sizeof(float2));
  p.status = c.status;
  p.timeout = c.timeout_ns;
  const dim3 grid(splits, a.units);
#define KVC_DEC(DD, GG) \
  if (a.D == DD && a.G == GG) return launch_t<DD, GG>(c, a, p, grid);
  KVC_DEC(128, 1) KVC_DEC(128, 2) KVC_DEC(128, 4) KVC_DEC(128, 8)
  KVC_DEC(64, 1) KVC_DEC(64, 2) KVC_DEC(64, 4) KVC_DEC(64, 8)
#undef KVC_DEC
  return cudaErrorInvalidValue;
}

}  // namespace kvc
