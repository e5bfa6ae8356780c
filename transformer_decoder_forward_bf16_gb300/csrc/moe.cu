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
#include <algorithm>

#include "fk_common.cuh"
#include "fk_internal.h"

namespace fk {

namespace {

constexpr int kRouteTokens = 64;  // tokens per routing block (one 64-bit mask per expert)
constexpr int kRouteThreads = 256;
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

__global__ void __launch_bounds__(kRouteThreads)
    moe_route_kernel(const float* __restrict__ z, int ld, int T, int E, int k, int norm_topk,
                     const int32_t* __restrict__ forced, int32_t* __restrict__ ids, float* __restrict__ wts,
                     float* __restrict__ margin, int32_t* __restrict__ counts, unsigned* dev_err) {
  __shared__ int hist[kMoeMaxExperts];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int t_begin = blockIdx.x * kRouteTokens;
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
                    int32_t* __restrict__ group_off) {
  __shared__ int tot[kMoeMaxExperts];
  __shared__ int off[kMoeMaxExperts + 1];
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
  }
  if (e == 0) group_off[E] = off[E];
}

__global__ void __launch_bounds__(256)
    moe_place_kernel(const int32_t* __restrict__ ids, int T, int E, int k, const int32_t* __restrict__ base,
                     int32_t* __restrict__ pos, int32_t* __restrict__ src) {
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

// xs[r] = u[src[r]]: one warp per 16-bit row of H elements (H % 64 == 0)
__global__ void __launch_bounds__(256)
    moe_gather_kernel(const uint16_t* __restrict__ u, int H, const int32_t* __restrict__ src, int rows,
                      uint16_t* __restrict__ xs) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint4* s = reinterpret_cast<const uint4*>(u + (size_t)src[r] * H);
  uint4* d = reinterpret_cast<uint4*>(xs + (size_t)r * H);
  for (int c = threadIdx.x & 31; c < H / 8; c += 32) d[c] = s[c];
}

// out[t] = [res[t] +] sum_j w[t,j] ys[pos[t,j]] (j ascending, fp32)
__global__ void __launch_bounds__(256)
    moe_combine_kernel(const float* __restrict__ ys, int H, const int32_t* __restrict__ pos,
                       const float* __restrict__ w, int k, const float* __restrict__ res, float* __restrict__ out) {
  __shared__ int sp[kMoeMaxK];
  __shared__ float sw[kMoeMaxK];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    sp[threadIdx.x] = pos[(size_t)t * k + threadIdx.x];
    sw[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  for (int c = threadIdx.x * 4; c < H; c += blockDim.x * 4) {
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
  }
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
  t.pos = reinterpret_cast<int32_t*>(take(Tk * 4));
  t.src = reinterpret_cast<int32_t*>(take(Tk * 4));
  t.xs = take(Tk * H * 2);
  t.hs = take(Tk * Ie * 2);
  t.ys = reinterpret_cast<float*>(take(Tk * H * 4));
  if (s) *s = t;
  return off;
}

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
                      cudaStream_t st, void* gemv, size_t gemv_bytes, size_t gemv_counter) {
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
  {
    ProfScope ps("moe_route", st);
    FK_TRY_STATUS(moe_route_launch(s.z, T, E, E, k, mw.norm_topk, forced, s.ids, s.w, s.margin, s.counts, dev_err, st));
    moe_scan_kernel<<<1, kMoeMaxExperts, 0, st>>>(s.counts, nblk, E, s.base, s.group_off);
    FK_TRY_LAUNCH("moe_scan_kernel launch");
    moe_place_kernel<<<nblk, 256, 0, st>>>(s.ids, T, E, k, s.base, s.pos, s.src);
    FK_TRY_LAUNCH("moe_place_kernel launch");
  }
  {
    ProfScope ps("moe_gather", st);
    moe_gather_kernel<<<(Tk + 7) / 8, 256, 0, st>>>(static_cast<const uint16_t*>(u), H, s.src, Tk,
                                                    static_cast<uint16_t*>(s.xs));
    FK_TRY_LAUNCH("moe_gather_kernel launch");
  }
  {
    ProfScope ps("moe_gate_up", st);
    GemmOut og;
    og.epi = EPI_GLU_BF16;
    og.out = s.hs;
    og.ldo = mw.Ie;
    og.act = mw.act;
    og.out_f16 = mw.act_f16;
    FK_TRY_STATUS(gemm_run_grouped(s.xs, Tk, H, mw.gate_up, og, s.group_off, dev_err, st));
  }
  {
    ProfScope ps("moe_down", st);
    GemmOut od;
    od.epi = EPI_F32;
    od.out = s.ys;
    od.ldo = H;
    FK_TRY_STATUS(gemm_run_grouped(s.hs, Tk, mw.Ie, mw.down, od, s.group_off, dev_err, st));
  }
  {
    ProfScope ps("moe_combine", st);
    moe_combine_kernel<<<T, std::min(256, H / 4), 0, st>>>(s.ys, H, s.pos, s.w, k, res, out);
    FK_TRY_LAUNCH("moe_combine_kernel launch");
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
