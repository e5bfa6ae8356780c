// Mixture-of-experts FFN ("N7 · model/forward-parity", Thm 2: the qwen3moe
// rung): softmax routing to the k experts of largest probability, each
// expert's SwiGLU FFN on the tokens routed to it, and the sum of the expert
// outputs weighted by the routing probabilities.
//
// One call over T tokens (E experts, k per token, hidden H, expert width Ie):
//   z  = u·W_routerᵀ                       GEMM, fp32 logits [T, E]
//   route    one warp per token: softmax of z, the k largest logits (ties to
//            the lower expert), their weights and the routing margin; one CTA
//            per block of 64 tokens also counts its tokens per expert
//   scan     one CTA: per expert the prefix of the counts over the blocks,
//            then over the experts: the first sorted row of every expert
//            (group offsets) and of every (block, expert)
//   place    one CTA per block: (token, slot) -> sorted row = its (block,
//            expert) base + the number of the block's earlier tokens routed
//            to the same expert (a 64-bit token mask per expert). An expert's
//            rows are in token order, so the layout, and with it every
//            result, does not depend on scheduling
//   gather   xs[row] = u[token of row]
//   h  = act(xs·gate_eᵀ) ⊙ (xs·up_eᵀ)       grouped tcgen05 GEMM, GLU epilogue
//   ys = h·down_eᵀ                          grouped tcgen05 GEMM, fp32 [T*k, H]
//   combine  out[t] = res[t] + sum_j w[t,j] ys[pos[t,j]], j ascending
// Decode steps (few tokens, a handful of rows per expert) run the two expert
// GEMMs as a grouped split-K weight stream instead (moe_expert_gemv_kernel):
// one CTA per (active expert, 128-row weight tile, K split), the expert's rows
// the N side of tcgen05.mma, fp32 partial sums added in split order by the
// last CTA of each tile.
#include <algorithm>

#include "fk_common.cuh"
#include "fk_internal.h"
#include "fk_ops.h"
#include "fk_launch.h"

namespace fk {

namespace {

constexpr int kRouteTokens = 64;  // tokens per routing block (one 64-bit mask per expert)
constexpr int kRouteThreads = 256;
constexpr int kFusedGatherRows = 16;  // routed rows up to which the routing CTA gathers them itself
constexpr int kEPL = kMoeMaxExperts / 32;  // experts per lane

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// float -> unsigned key of the same order (negative values reversed)
FK_DEVICE uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

FK_DEVICE unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// p[e >> 5] of lane e & 31, for every lane
FK_DEVICE float prob_of(const float (&p)[kEPL], int e) {
  float pe = 0.f;
#pragma unroll
  for (int i = 0; i < kEPL; ++i)
    if (i == (e >> 5)) pe = p[i];
  return __shfl_sync(0xffffffffu, pe, e & 31);
}

// Route the tokens t_begin .. t_begin + 63 (< T) of a block: one warp per
// token; hist[e] counts the block's tokens routed to expert e.
FK_DEVICE void route_block(const float* __restrict__ z, int ld, int T, int E, int k, int norm_topk,
                           const int32_t* __restrict__ forced, int32_t* __restrict__ ids, float* __restrict__ wts,
                           float* __restrict__ margin, unsigned* dev_err, int t_begin, int* hist) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int tl = warp; tl < kRouteTokens; tl += kRouteThreads / 32) {
    const int t = t_begin + tl;
    if (t >= T) break;
    const float* zr = z + (size_t)t * ld;
    // softmax over the experts, fp32
    float v[kEPL], p[kEPL];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kEPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? zr[e] : -INFINITY;
      m = fmaxf(m, v[i]);
    }
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kEPL; ++i) {
      p[i] = lane + 32 * i < E ? expf(v[i] - m) : 0.f;
      s += p[i];
    }
    s = warp_sum(s);
    const float inv = 1.0f / s;
#pragma unroll
    for (int i = 0; i < kEPL; ++i) p[i] *= inv;
    // the k largest logits (the order of p), ties to the lower expert: keys
    // (order of z) << 32 | (~expert); 0 marks a taken or absent expert
    unsigned long long cand[kEPL];
#pragma unroll
    for (int i = 0; i < kEPL; ++i) {
      const int e = lane + 32 * i;
      cand[i] = e < E ? ((unsigned long long)order_key(v[i]) << 32) | (0xFFFFFFFFu - (uint32_t)e) : 0ull;
    }
    int my_id = 0;
    float my_p = 0.f, p_next = 0.f;
    const int rounds = k < E ? k + 1 : k;
    for (int r = 0; r < rounds; ++r) {
      unsigned long long best = 0ull;
#pragma unroll
      for (int i = 0; i < kEPL; ++i) best = cand[i] > best ? cand[i] : best;
      best = warp_max_u64(best);
      const int e = (int)(0xFFFFFFFFu - (uint32_t)(best & 0xFFFFFFFFull));
      const float pe = prob_of(p, e);
      if (lane == (e & 31)) {
#pragma unroll
        for (int i = 0; i < kEPL; ++i)
          if (i == (e >> 5)) cand[i] = 0ull;
      }
      if (r < k) {
        if (lane == r) {
          my_id = e;
          my_p = pe;
        }
      } else {
        p_next = pe;
      }
    }
    const float p_kth = __shfl_sync(0xffffffffu, my_p, k - 1);
    // forced ids: used when all k are in range and distinct
    if (forced) {
      const int f = lane < k ? forced[(size_t)t * k + lane] : -1 - lane;
      const unsigned same = __match_any_sync(0xffffffffu, f);
      const bool ok = __all_sync(0xffffffffu, lane >= k || (f >= 0 && f < E && __popc(same) == 1));
      if (ok) {
        for (int j = 0; j < k; ++j) {
          const int ej = __shfl_sync(0xffffffffu, f, j);
          const float pj = prob_of(p, ej);
          if (lane == j) {
            my_id = ej;
            my_p = pj;
          }
        }
      } else if (lane == 0 && dev_err) {
        atomicOr(dev_err, FK_DEVERR_EXPERT_IDS);
      }
    }
    const float wsum = warp_sum(lane < k ? my_p : 0.f);
    if (lane < k) {
      ids[(size_t)t * k + lane] = my_id;
      wts[(size_t)t * k + lane] = norm_topk ? my_p / wsum : my_p;
      atomicAdd(&hist[my_id], 1);
    }
    if (lane == 0 && margin) margin[t] = k < E ? p_kth - p_next : INFINITY;
  }
}

__global__ void __launch_bounds__(kRouteThreads)
    moe_route_kernel(const float* __restrict__ z, int ld, int T, int E, int k, int norm_topk,
                     const int32_t* __restrict__ forced, int32_t* __restrict__ ids, float* __restrict__ wts,
                     float* __restrict__ margin, int32_t* __restrict__ counts, unsigned* dev_err) {
  pdl_wait();  // inside a decode step: the predecessor's outputs, then release the successor
  pdl_trigger();
  __shared__ int hist[kMoeMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  route_block(z, ld, T, E, k, norm_topk, forced, ids, wts, margin, dev_err, blockIdx.x * kRouteTokens, hist);
  if (counts) {
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) counts[(size_t)blockIdx.x * E + e] = hist[e];
  }
}

// Exclusive prefix over n <= 256 values in smem (in -> out, out[n] = total),
// by warp 0.
FK_DEVICE void warp0_exclusive_scan(const int* in, int* out, int n) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x >= 32) return;
  int carry = 0;
  for (int g0 = 0; g0 < n; g0 += 32) {
    const int g = g0 + lane;
    const int x = g < n ? in[g] : 0;
    int v = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    if (g < n) out[g] = carry + v - x;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) out[n] = carry;
}

__global__ void __launch_bounds__(kMoeMaxExperts)
    moe_scan_kernel(const int32_t* __restrict__ counts, int nblk, int E, int32_t* __restrict__ base,
                    int32_t* __restrict__ group_off, int32_t* __restrict__ active) {
  pdl_wait();  // inside a decode step: the predecessor's outputs, then release the successor
  pdl_trigger();
  __shared__ int tot[kMoeMaxExperts];
  __shared__ int off[kMoeMaxExperts + 1];
  __shared__ int has[kMoeMaxExperts];
  __shared__ int apos[kMoeMaxExperts + 1];
  const int e = threadIdx.x;
  int run = 0;
  if (e < E) {
#pragma unroll 4
    for (int b = 0; b < nblk; ++b) {
      const int c = counts[(size_t)b * E + e];
      base[(size_t)b * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();
  warp0_exclusive_scan(tot, off, E);
  __syncthreads();
  if (e < E) {
    const int o = off[e];
#pragma unroll 4
    for (int b = 0; b < nblk; ++b) base[(size_t)b * E + e] += o;
    group_off[e] = o;
    has[e] = tot[e] > 0;
  }
  if (e == 0) group_off[E] = off[E];
  if (active) {  // the experts with rows, in id order; active[kMoeMaxExperts] = their number
    __syncthreads();
    warp0_exclusive_scan(has, apos, E);
    __syncthreads();
    if (e < E && has[e]) active[apos[e]] = e;
    if (e == 0) active[kMoeMaxExperts] = apos[E];
  }
}

__global__ void __launch_bounds__(256)
    moe_place_kernel(const int32_t* __restrict__ ids, int T, int E, int k, const int32_t* __restrict__ base,
                     int32_t* __restrict__ pos, int32_t* __restrict__ src) {
  pdl_wait();  // inside a decode step: the predecessor's outputs, then release the successor
  pdl_trigger();
  __shared__ unsigned long long mask[kMoeMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) mask[e] = 0ull;
  __syncthreads();
  const int t0 = blockIdx.x * kRouteTokens;
  const int n = min(kRouteTokens, T - t0) * k;
  const int32_t* bid = ids + (size_t)t0 * k;
  for (int i = threadIdx.x; i < n; i += blockDim.x) atomicOr(&mask[bid[i]], 1ull << (i / k));
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int tl = i / k, e = bid[i];
    const int r = __popcll(mask[e] & ((1ull << tl) - 1ull));
    const int p = base[(size_t)blockIdx.x * E + e] + r;
    pos[(size_t)t0 * k + i] = p;
    src[p] = t0 + tl;
  }
}

// At most one routing block (T <= 64 tokens): routing, the expert offsets and
// the placement in one CTA (the three steps above without their launches).
__global__ void __launch_bounds__(kRouteThreads)
    moe_route_small_kernel(const float* __restrict__ z, int ld, int T, int E, int k, int norm_topk,
                           const int32_t* __restrict__ forced, int32_t* __restrict__ ids, float* __restrict__ wts,
                           float* __restrict__ margin, int32_t* __restrict__ group_off, int32_t* __restrict__ active,
                           int32_t* __restrict__ pos, int32_t* __restrict__ src, unsigned* dev_err,
                           const uint16_t* __restrict__ u, int H, uint16_t* __restrict__ xs) {
  pdl_wait();  // inside a decode step: the predecessor's outputs, then release the successor
  pdl_trigger();
  __shared__ int ssrc[kRouteTokens * kMoeMaxK];
  __shared__ int hist[kMoeMaxExperts];
  __shared__ int off[kMoeMaxExperts + 1];
  __shared__ int has[kMoeMaxExperts];
  __shared__ int apos[kMoeMaxExperts + 1];
  __shared__ unsigned long long mask[kMoeMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    hist[e] = 0;
    mask[e] = 0ull;
  }
  __syncthreads();
  route_block(z, ld, T, E, k, norm_topk, forced, ids, wts, margin, dev_err, 0, hist);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) has[e] = hist[e] > 0;
  warp0_exclusive_scan(hist, off, E);
  __syncthreads();
  warp0_exclusive_scan(has, apos, E);
  for (int e = threadIdx.x; e <= E; e += blockDim.x) group_off[e] = off[e];
  const int n = T * k;
  for (int i = threadIdx.x; i < n; i += blockDim.x) atomicOr(&mask[ids[i]], 1ull << (i / k));
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (has[e]) active[apos[e]] = e;
  if (threadIdx.x == 0) active[kMoeMaxExperts] = apos[E];
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int t = i / k, e = ids[i];
    const int p = off[e] + __popcll(mask[e] & ((1ull << t) - 1ull));
    pos[i] = p;
    src[p] = t;
    ssrc[p] = t;
  }
  if (xs) {  // the gather of the expert-sorted rows (few rows): xs[r] = u[src[r]], a warp per row
    __syncthreads();
    for (int r = threadIdx.x >> 5; r < n; r += blockDim.x >> 5) {
      const uint4* s4 = reinterpret_cast<const uint4*>(u + (size_t)ssrc[r] * H);
      uint4* d4 = reinterpret_cast<uint4*>(xs + (size_t)r * H);
      for (int c = threadIdx.x & 31; c < H / 8; c += 32) d4[c] = s4[c];
    }
  }
}

// xs[r] = u[src[r]]: one warp per 16-bit row of H elements (H % 64 == 0)
__global__ void __launch_bounds__(256)
    moe_gather_kernel(const uint16_t* __restrict__ u, int H, const int32_t* __restrict__ src, int rows,
                      uint16_t* __restrict__ xs) {
  pdl_wait();  // inside a decode step: the predecessor's outputs, then release the successor
  pdl_trigger();
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint4* s = reinterpret_cast<const uint4*>(u + (size_t)src[r] * H);
  uint4* d = reinterpret_cast<uint4*>(xs + (size_t)r * H);
  for (int c = threadIdx.x & 31; c < H / 8; c += 32) d[c] = s[c];
}

// out[t] = [res[t] +] sum_j w[t,j] ys[pos[t,j]] (j ascending, fp32). With
// NORM, also the RMSNorm of the row for the next consumer, u[t] =
// 16-bit(out * rsqrt(mean(out^2) + eps) * nw), with the row held in registers:
// thread i holds elements 4 (m blockDim + i) .. + 3 (m = 0, 1, ...) and the
// sums of squares are reduced in the order of the standalone row norm, so u
// equals what that kernel would make of out.
constexpr int kCombineMaxVec = 8;  // float4 per thread with NORM: H <= 8192
template <bool NORM>
__global__ void __launch_bounds__(256)
    moe_combine_kernel(const float* __restrict__ ys, int H, const int32_t* __restrict__ pos,
                       const float* __restrict__ w, int k, const float* __restrict__ res, float* __restrict__ out,
                       const __nv_bfloat16* __restrict__ nw, float eps, uint16_t* __restrict__ u, int u_f16) {
  pdl_wait();  // inside a decode step: the predecessor's outputs, then release the successor
  pdl_trigger();
  __shared__ int sp[kMoeMaxK];
  __shared__ float sw[kMoeMaxK];
  __shared__ float red[8];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    sp[threadIdx.x] = pos[(size_t)t * k + threadIdx.x];
    sw[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  float4 v[NORM ? kCombineMaxVec : 1];
  float ss = 0.f;
#pragma unroll
  for (int m = 0; m < (NORM ? kCombineMaxVec : 1 << 20); ++m) {
    const int c = (m * blockDim.x + threadIdx.x) * 4;
    if (c >= H) break;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float4 y = *reinterpret_cast<const float4*>(ys + (size_t)sp[j] * H + c);
      const float wj = sw[j];
      acc.x = fmaf(wj, y.x, acc.x);
      acc.y = fmaf(wj, y.y, acc.y);
      acc.z = fmaf(wj, y.z, acc.z);
      acc.w = fmaf(wj, y.w, acc.w);
    }
    if (res) {
      const float4 x = *reinterpret_cast<const float4*>(res + (size_t)t * H + c);
      acc.x = x.x + acc.x;
      acc.y = x.y + acc.y;
      acc.z = x.z + acc.z;
      acc.w = x.w + acc.w;
    }
    *reinterpret_cast<float4*>(out + (size_t)t * H + c) = acc;
    if constexpr (NORM) {
      v[m] = acc;
      ss += acc.x * acc.x + acc.y * acc.y + acc.z * acc.z + acc.w * acc.w;
    }
  }
  if constexpr (NORM) {
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
    const float r = rsqrtf(tot / H + eps);
    uint16_t* ur = u + (size_t)t * H;
#pragma unroll
    for (int m = 0; m < kCombineMaxVec; ++m) {
      const int c = (m * blockDim.x + threadIdx.x) * 4;
      if (c >= H) break;
      const uint2 wp = *reinterpret_cast<const uint2*>(nw + c);
      *reinterpret_cast<uint2*>(ur + c) =
          make_uint2(pack_16x2(v[m].x * r * bf16_lo(wp.x), v[m].y * r * bf16_hi(wp.x), u_f16),
                     pack_16x2(v[m].z * r * bf16_lo(wp.y), v[m].w * r * bf16_hi(wp.y), u_f16));
    }
  }
}

// ---------------------------------------------------------------------------
// Grouped split-K expert GEMM for few tokens
// ---------------------------------------------------------------------------
constexpr int kExpThreads = 128;
constexpr int kExpStages = 4;
constexpr int kExpMaxSplits = 8;
constexpr int kExpWBytes = 128 * 64 * 2;  // one 128-row x 64-column weight tile

struct ExpArgs {
  const int32_t* group_off;  // [E + 1] first sorted row of each expert
  const int32_t* active;     // [E + 1]: active experts in id order, then their number
  int glu, act;              // glu: a tile = 64 gate + 64 up rows, output act(gate) * up (16-bit)
  int tiles;                 // weight tiles per expert
  int group_rows;            // rows of one expert's matrix in each map
  int n_feat;                // output features per expert (Ie for gate/up, H for down)
  int nk;                    // k-blocks of 64
  int ab_f16, out_f16;
  void* out;                 // 16-bit (glu) or fp32 [rows][ldo]
  int ldo;
  float* part;               // [splits][rows][tiles * 128] fp32 partial sums (splits > 1)
  int rows;                  // routed rows of the call (T * k)
  unsigned* counters;        // [E * tiles], zero between launches
  unsigned* dev_err;
};

template <int BT>
struct ECfg {
  static constexpr int X_BYTES = BT * 64 * 2;
  static constexpr int STAGE = kExpWBytes + X_BYTES;
  static constexpr int SMEM = kExpStages * STAGE + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = BT < 32 ? 32 : BT;
  static_assert(kExpStages * STAGE >= 128 * BT * 4, "the result tile reuses the stage ring");
};

// Apply the epilogue to a [128 lanes][BT] fp32 tile in shared memory (lane
// = weight row of the tile): rows r0 .. r0 + cnt of the output.
FK_DEVICE void exp_store(const ExpArgs& a, const float* sD, int BT, int r0, int cnt, int tile) {
  const int per = a.glu ? 64 : 128;
  for (int i = threadIdx.x; i < per * cnt; i += kExpThreads) {
    const int f = i % per, t = i / per;
    const int feat = tile * per + f;
    if (feat >= a.n_feat) continue;
    const float v = sD[f * BT + t];
    if (a.glu) {
      const float u = sD[(64 + f) * BT + t];
      const float g = a.act ? 0.5f * v * (1.0f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)))
                            : v / (1.0f + expf(-v));
      store_16(static_cast<uint16_t*>(a.out) + (size_t)(r0 + t) * a.ldo + feat, g * u, a.out_f16);
    } else {
      static_cast<float*>(a.out)[(size_t)(r0 + t) * a.ldo + feat] = v;
    }
  }
}

template <int BT>
__global__ void __launch_bounds__(kExpThreads)
    moe_expert_gemv_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW0,
                           const __grid_constant__ CUtensorMap tmW1, const ExpArgs a) {
  using C = ECfg<BT>;
  pdl_wait();  // the routing and the inputs come from the preceding kernels
  pdl_trigger();
  const int slot = blockIdx.x / a.tiles, tile = blockIdx.x % a.tiles;
  if (slot >= a.active[kMoeMaxExperts]) return;  // fewer active experts than the grid's bound (whole CTA)
  const int g = a.active[slot];
  const int r0 = a.group_off[g], cnt = min(a.group_off[g + 1] - r0, BT);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kExpStages * C::STAGE);
  uint64_t* empty = full + kExpStages;
  uint64_t* done = empty + kExpStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last = abort_flag + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.y;
  const int kb0 = (int)((long)split * a.nk / gridDim.y), kb1 = (int)((long)(split + 1) * a.nk / gridDim.y);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kExpStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---- producer: the tile's two 64-row weight boxes and the expert's rows
    const int wrow = g * a.group_rows + tile * (a.glu ? 64 : 128);
    const bool second = a.glu || tile * 128 + 64 < a.group_rows;  // a plain tile's lower half exists
    const uint32_t bytes = kExpWBytes / (second ? 1 : 2) + C::X_BYTES;
    int issued[kExpStages] = {0, 0, 0, 0};
    for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
      const int stage = it % kExpStages;
      if (it >= kExpStages && !mbar_wait(&empty[stage], ((it / kExpStages) - 1) & 1, abort_flag, a.dev_err)) break;
      uint8_t* sa = smem + stage * C::STAGE;
      mbar_arrive_expect_tx(&full[stage], bytes);
      tma_load_2d(&tmW0, &full[stage], sa, kb * 64, wrow);
      if (second) tma_load_2d(a.glu ? &tmW1 : &tmW0, &full[stage], sa + kExpWBytes / 2, kb * 64, a.glu ? wrow : wrow + 64);
      tma_load_2d(&tmX, &full[stage], sa + kExpWBytes, kb * 64, r0);
      ++issued[stage];
    }
    if (*abort_flag) {  // let issued copies land before the CTA unwinds
      for (int s = 0; s < kExpStages; ++s) {
        if (!issued[s]) continue;
        const uint32_t fa = smem_u32(&full[s]);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(fa, (issued[s] - 1) & 1) && globaltimer_ns() - t0 < 100000000ull) {
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: D[128 weight rows][BT rows] += W · Xᵀ
    const uint32_t idesc = idesc_16b_f32(128, BT, a.ab_f16);
    for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
      const int stage = it % kExpStages;
      if (!mbar_wait(&full[stage], (it / kExpStages) & 1, abort_flag, a.dev_err)) break;
      tc_fence_after();
      uint8_t* sa = smem + stage * C::STAGE;
      const uint64_t ad = smem_desc_sw128(sa), bd = smem_desc_sw128(sa + kExpWBytes);
#pragma unroll
      for (int k = 0; k < 4; ++k) umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (it | k) != 0 ? 1u : 0u);
      umma_commit(&empty[stage]);
    }
    umma_commit(done);
  }
  __syncwarp();
  // ---- epilogue: the tile's fp32 result [128 lanes][BT] into shared memory (the ring is idle)
  const bool have = mbar_wait(done, 0, abort_flag, a.dev_err) && kb1 > kb0;
  tc_fence_after();
  float* sD = reinterpret_cast<float*>(smem);
  const int lrow = warp * 32 + lane;  // TMEM lane = weight row of the tile
#pragma unroll
  for (int c0 = 0; c0 < BT; c0 += 32) {
    float v[32];
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (c0 + j < BT) sD[lrow * BT + c0 + j] = have ? v[j] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (gridDim.y == 1) {  // one split: the epilogue straight away
    if (have) exp_store(a, sD, BT, r0, cnt, tile);
    return;
  }
  // ---- split K: this split's partial sums, then the last CTA of the tile adds them in split order
  const int nv = a.tiles * 128;
  float* mine = a.part + (size_t)split * a.rows * nv;
  for (int t = 0; t < cnt; ++t) mine[(size_t)(r0 + t) * nv + tile * 128 + lrow] = sD[lrow * BT + t];
  // the barrier orders every thread's partial stores before thread 0's
  // acquire-release arrival; in the last CTA it acquires the other splits'
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(&a.counters[g * a.tiles + tile])
                 : "memory");
    *last = prev == gridDim.y - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!*last) return;
  for (int t = 0; t < cnt; ++t) {
    float sum = 0.f;
    for (int s2 = 0; s2 < (int)gridDim.y; ++s2)
      sum += __ldcg(a.part + ((size_t)s2 * a.rows + r0 + t) * nv + tile * 128 + lrow);
    sD[lrow * BT + t] = sum;
  }
  __syncthreads();
  exp_store(a, sD, BT, r0, cnt, tile);
  if (threadIdx.x == 0) a.counters[g * a.tiles + tile] = 0;
}

#define FK_TRY_STATUS(expr)     \
  do {                          \
    fk_status _s = (expr);      \
    if (_s != FK_OK) return _s; \
  } while (0)
#define FK_TRY_LAUNCH(what)                                  \
  do {                                                       \
    cudaError_t _e = cudaGetLastError();                     \
    if (_e != cudaSuccess) return cuda_fail(_e, what);       \
  } while (0)

}  // namespace

// weight tiles per expert of the few-token expert GEMM: 64 gate + 64 up rows,
// or 128 rows of the down matrix
int moe_tiles(const MoeWeights& mw, bool glu) { return glu ? (mw.Ie + 63) / 64 : (mw.H + 127) / 128; }

size_t moe_scratch(const MoeWeights& mw, long T, MoeScratch* s, uint8_t* base) {
  const size_t E = mw.E, k = mw.k, H = mw.H, Ie = mw.Ie;
  const size_t nblk = (T + kRouteTokens - 1) / kRouteTokens;
  const size_t Tk = (size_t)T * k;
  size_t off = 0;
  auto take = [&](size_t bytes) -> uint8_t* {
    uint8_t* p = base ? base + off : nullptr;
    off += align_up(bytes);
    return p;
  };
  MoeScratch t;
  t.z = reinterpret_cast<float*>(take((size_t)T * E * 4));
  t.ids = reinterpret_cast<int32_t*>(take(Tk * 4));
  t.w = reinterpret_cast<float*>(take(Tk * 4));
  t.margin = reinterpret_cast<float*>(take((size_t)T * 4));
  t.counts = reinterpret_cast<int32_t*>(take(nblk * E * 4));
  t.base = reinterpret_cast<int32_t*>(take(nblk * E * 4));
  t.group_off = reinterpret_cast<int32_t*>(take((E + 1) * 4));
  t.active = reinterpret_cast<int32_t*>(take((kMoeMaxExperts + 1) * 4));
  // few-token expert GEMMs: arrival counters per (expert, weight tile), and
  // the split partial sums of up to kMoeFewMaxTokens tokens
  t.exp_counters_bytes = align_up(E * (size_t)std::max(moe_tiles(mw, true), moe_tiles(mw, false)) * 4);
  t.exp_counters = reinterpret_cast<unsigned*>(take(t.exp_counters_bytes));
  t.exp_part = reinterpret_cast<float*>(take((size_t)kExpMaxSplits * std::min<long>(T, kMoeFewMaxTokens) * k *
                                             std::max(moe_tiles(mw, true), moe_tiles(mw, false)) * 128 * 4));
  t.pos = reinterpret_cast<int32_t*>(take(Tk * 4));
  t.src = reinterpret_cast<int32_t*>(take(Tk * 4));
  t.xs = take(Tk * H * 2);
  t.hs = take(Tk * Ie * 2);
  t.ys = reinterpret_cast<float*>(take(Tk * H * 4));
  if (s) *s = t;
  return off;
}

namespace {

template <int BT>
fk_status launch_expert_bt(const CUtensorMap& tX, const GemmWeights& w, const ExpArgs& a, int grid_x, int splits,
                           cudaStream_t st) {
  using C = ECfg<BT>;
  static DeviceOnce once;
  const cudaError_t attr = once.run([] {
    return cudaFuncSetAttribute(moe_expert_gemv_kernel<BT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (attr != cudaSuccess) return cuda_fail(attr, "cudaFuncSetAttribute(moe_expert_gemv)");
  cudaError_t e = fk_launch(moe_expert_gemv_kernel<BT>, dim3(grid_x, splits), dim3(kExpThreads), C::SMEM, st, tX,
                            w.map[0], w.nseg > 1 ? w.map[1] : w.map[0], a);
  if (e != cudaSuccess) return cuda_fail(e, "moe_expert_gemv_kernel launch");
  return FK_OK;
}

// One expert GEMM of T <= kMoeFewMaxTokens tokens (T * k routed rows in X,
// sorted by expert): gate/up with the gated activation (16-bit out) or down
// (fp32 out).
fk_status moe_expert_gemv(const MoeWeights& mw, bool glu, const void* X, int T, const MoeScratch& s, void* out,
                          unsigned* dev_err, cudaStream_t st) {
  int sms = 0;
  fk_status stt = check_device(&sms);
  if (stt != FK_OK) return stt;
  const GemmWeights& w = glu ? mw.gate_up : mw.down;
  const int rows = T * mw.k;
  const int BT = T <= 16 ? 16 : (T <= 32 ? 32 : 64);  // an expert holds at most T of the rows
  CUtensorMap tX;
  stt = make_tmap_bf16(&tX, X, rows, w.K, w.K, BT);
  if (stt != FK_OK) return stt;
  ExpArgs a{};
  a.group_off = s.group_off;
  a.active = s.active;
  a.glu = glu ? 1 : 0;
  a.act = mw.act;
  a.tiles = moe_tiles(mw, glu);
  a.group_rows = w.group_rows;
  a.n_feat = glu ? mw.Ie : mw.H;
  a.nk = (w.K + 63) / 64;
  a.ab_f16 = w.f16;
  a.out_f16 = mw.act_f16;
  a.out = out;
  a.ldo = glu ? mw.Ie : mw.H;
  a.part = s.exp_part;
  a.rows = rows;
  a.counters = s.exp_counters;
  a.dev_err = dev_err;
  // at most min(E, rows) experts have rows; split K so that about one wave of
  // CTAs streams the active experts' tiles
  const int act_max = std::min(mw.E, rows);
  const int smem = BT == 16 ? ECfg<16>::SMEM : (BT == 32 ? ECfg<32>::SMEM : ECfg<64>::SMEM);
  const int per_sm = std::max(1, std::min(16, (228 << 10) / (smem + 1024)));
  const int splits = std::max(1, std::min({kExpMaxSplits, a.nk, per_sm * sms / (act_max * a.tiles)}));
  const int grid_x = act_max * a.tiles;
  if (BT == 16) return launch_expert_bt<16>(tX, w, a, grid_x, splits, st);
  if (BT == 32) return launch_expert_bt<32>(tX, w, a, grid_x, splits, st);
  return launch_expert_bt<64>(tX, w, a, grid_x, splits, st);
}

}  // namespace

fk_status moe_route_launch(const float* z, int T, int E, int ld, int k, int norm_topk, const int32_t* forced,
                           int32_t* ids, float* w, float* margin, int32_t* counts, unsigned* dev_err,
                           cudaStream_t st) {
  if (T == 0) return FK_OK;
  const int nblk = (T + kRouteTokens - 1) / kRouteTokens;
  moe_route_kernel<<<nblk, kRouteThreads, 0, st>>>(z, ld, T, E, k, norm_topk, forced, ids, w, margin, counts, dev_err);
  FK_TRY_LAUNCH("moe_route_kernel launch");
  return FK_OK;
}

fk_status moe_ffn_run(const MoeWeights& mw, const void* u, int T, const MoeScratch& s, const int32_t* forced,
                      int32_t* trace_ids, float* trace_margin, float* out, const float* res, unsigned* dev_err,
                      cudaStream_t st, bool few, void* gemv, size_t gemv_bytes, size_t gemv_counter,
                      const NormOut* next_norm) {
  if (T == 0) return FK_OK;
  const int E = mw.E, k = mw.k, H = mw.H;
  const int Tk = T * k;
  const int nblk = (T + kRouteTokens - 1) / kRouteTokens;
  {
    ProfScope ps("moe_router", st);
    GemmOut oz;
    oz.epi = EPI_F32;
    oz.out = s.z;
    oz.ldo = E;
    FK_TRY_STATUS(gemm_run(u, T, H, mw.router, oz, dev_err, st, gemv, gemv_bytes, gemv_counter));
  }
  // few routed rows: the routing CTA copies them into expert order itself
  const bool fused_gather = T <= kRouteTokens && Tk <= kFusedGatherRows;
  if (T <= kRouteTokens) {  // one routing block: routing, offsets and placement in one CTA
    ProfScope ps("moe_route", st);
    cudaError_t e = fk_launch(moe_route_small_kernel, dim3(1), dim3(kRouteThreads), 0, st, (const float*)s.z, E, T, E,
                              k, mw.norm_topk, forced, s.ids, s.w, s.margin, s.group_off, s.active, s.pos, s.src,
                              dev_err, static_cast<const uint16_t*>(u), H,
                              fused_gather ? static_cast<uint16_t*>(s.xs) : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "moe_route_small_kernel launch");
  } else {
    ProfScope ps("moe_route", st);
    FK_TRY_STATUS(moe_route_launch(s.z, T, E, E, k, mw.norm_topk, forced, s.ids, s.w, s.margin, s.counts, dev_err, st));
    moe_scan_kernel<<<1, kMoeMaxExperts, 0, st>>>(s.counts, nblk, E, s.base, s.group_off, s.active);
    FK_TRY_LAUNCH("moe_scan_kernel launch");
    moe_place_kernel<<<nblk, 256, 0, st>>>(s.ids, T, E, k, s.base, s.pos, s.src);
    FK_TRY_LAUNCH("moe_place_kernel launch");
  }
  if (!fused_gather) {
    ProfScope ps("moe_gather", st);
    cudaError_t e = fk_launch(moe_gather_kernel, dim3((Tk + 7) / 8), dim3(256), 0, st, static_cast<const uint16_t*>(u),
                              H, (const int32_t*)s.src, Tk, static_cast<uint16_t*>(s.xs));
    if (e != cudaSuccess) return cuda_fail(e, "moe_gather_kernel launch");
  }
  few = few && T <= kMoeFewMaxTokens;
  if (few) {
    ProfScope ps("moe_gate_up", st);
    FK_TRY_STATUS(moe_expert_gemv(mw, true, s.xs, T, s, s.hs, dev_err, st));
  } else {
    ProfScope ps("moe_gate_up", st);
    GemmOut og;
    og.epi = EPI_GLU_BF16;
    og.out = s.hs;
    og.ldo = mw.Ie;
    og.act = mw.act;
    og.out_f16 = mw.act_f16;
    FK_TRY_STATUS(gemm_run_grouped(s.xs, Tk, H, mw.gate_up, og, s.group_off, dev_err, st));
  }
  if (few) {
    ProfScope ps("moe_down", st);
    FK_TRY_STATUS(moe_expert_gemv(mw, false, s.hs, T, s, s.ys, dev_err, st));
  } else {
    ProfScope ps("moe_down", st);
    GemmOut od;
    od.epi = EPI_F32;
    od.out = s.ys;
    od.ldo = H;
    FK_TRY_STATUS(gemm_run_grouped(s.hs, Tk, mw.Ie, mw.down, od, s.group_off, dev_err, st));
  }
  {
    ProfScope ps("moe_combine", st);
    const bool norm = next_norm && H % 128 == 0 && H <= 256 * 4 * kCombineMaxVec;  // whole warps
    cudaError_t e =
        norm ? fk_launch(moe_combine_kernel<true>, dim3(T), dim3(std::min(256, H / 4)), 0, st, (const float*)s.ys, H,
                         (const int32_t*)s.pos, (const float*)s.w, k, res, out,
                         static_cast<const __nv_bfloat16*>(next_norm->w), next_norm->eps,
                         static_cast<uint16_t*>(next_norm->u), next_norm->f16)
             : fk_launch(moe_combine_kernel<false>, dim3(T), dim3(std::min(256, H / 4)), 0, st, (const float*)s.ys, H,
                         (const int32_t*)s.pos, (const float*)s.w, k, res, out, (const __nv_bfloat16*)nullptr, 0.f,
                         (uint16_t*)nullptr, 0);
    if (e != cudaSuccess) return cuda_fail(e, "moe_combine_kernel launch");
    if (next_norm && !norm)
      FK_CUDA_TRY(launch_rmsnorm(out, H, T, H, next_norm->w, next_norm->eps, next_norm->u, H, st, next_norm->f16));
  }
  if (trace_ids) FK_CUDA_TRY(cudaMemcpyAsync(trace_ids, s.ids, (size_t)Tk * 4, cudaMemcpyDeviceToDevice, st));
  if (trace_margin) FK_CUDA_TRY(cudaMemcpyAsync(trace_margin, s.margin, (size_t)T * 4, cudaMemcpyDeviceToDevice, st));
  return FK_OK;
}

}  // namespace fk

extern "C" fk_status fk_op_moe_route(const float* d_logits, int32_t T, int32_t E, int32_t ld, int32_t k,
                                     int32_t norm_topk, const int32_t* d_forced, int32_t* d_ids, float* d_weights,
                                     float* d_margin, void* stream) {
  using fk::fail;
  if (!d_logits || !d_ids || !d_weights || T < 0 || E < 1 || E > fk::kMoeMaxExperts || ld < E)
    return fail(FK_ERR_INVALID_ARG, "fk_op_moe_route: bad argument");
  if (k < 1 || k > std::min(E, fk::kMoeMaxK)) return fail(FK_ERR_INVALID_ARG, "fk_op_moe_route: need 1 <= k <= min(E, 16)");
  if (norm_topk != 0 && norm_topk != 1) return fail(FK_ERR_INVALID_ARG, "fk_op_moe_route: norm_topk must be 0 or 1");
  fk_status s = fk::check_device(nullptr);
  if (s != FK_OK) return s;
  unsigned* ctl = nullptr;
  s = fk::op_control_block(&ctl);
  if (s != FK_OK) return s;
  return fk::moe_route_launch(d_logits, T, E, ld, k, norm_topk, d_forced, d_ids, d_weights, d_margin, nullptr, ctl,
                              static_cast<cudaStream_t>(stream));
}
