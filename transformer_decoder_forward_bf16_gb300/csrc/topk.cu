// Log-softmax and top-k of fp32 logit rows ("pegainfer issue #878",
// Acceptance Criteria: the distributional comparison at the window edge reads
// log-probabilities at the top-64 ids of each position).
//
// One 1024-thread CTA per row (a 262144-word row is 1 MB and stays in L2
// across the passes):
//   1. row maximum and sum of exp(z - max), per thread online, then a block
//      reduction: lse = max + log(sum); optionally the whole row of z - lse;
//   2. the k-th largest value by radix selection on order-preserving 32-bit
//      keys of the floats (four 8-bit digits, most significant first; each
//      warp keeps its own 256-bin histogram, merged per digit);
//   3. the elements above that value, and the lowest-index ones equal to it
//      until k are taken (each thread scans one contiguous run of indices;
//      a block prefix count orders the equal ones by index);
//   4. the k candidates ranked by (value descending, index ascending) and
//      written as ids and log-probabilities z - lse.
#include <algorithm>

#include "fk_common.cuh"
#include "fk_internal.h"

namespace fk {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxK = 128;

// float -> unsigned key with the same order (negative values reversed)
FK_DEVICE uint32_t okey(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads, 1)
    logsoftmax_topk_kernel(const float* __restrict__ z, int V, int ld, int k, float* __restrict__ lse_out,
                           int32_t* __restrict__ top_ids, float* __restrict__ top_lp, float* __restrict__ lp_out) {
  __shared__ uint32_t hist[kWarps][256];
  __shared__ float red_m[kWarps], red_s[kWarps];
  __shared__ uint32_t sh_prefix, sh_want;
  __shared__ int scan[kThreads];
  __shared__ int cand_n;
  __shared__ int cand_i[kMaxK];
  __shared__ float cand_v[kMaxK];
  const int row = blockIdx.x;
  const float* zr = z + (size_t)row * ld;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- 1. max and sum of exponentials
  float m = -INFINITY, s = 0.f;
  for (int c = tid; c < V; c += kThreads) {
    const float v = zr[c];
    if (v > m) {
      s = s * expf(m - v) + 1.f;
      m = v;
    } else {
      s += expf(v - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float mm = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * expf(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * expf(m2 - mm));
    m = mm;
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_s[warp] = s;
  }
  __syncthreads();
  float M = -INFINITY;
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w]);
  float S = 0.f;
  for (int w = 0; w < kWarps; ++w)
    if (red_m[w] != -INFINITY) S += red_s[w] * expf(red_m[w] - M);
  const float lse = M + logf(S);
  if (tid == 0 && lse_out) lse_out[row] = lse;
  if (lp_out) {
    float* lr = lp_out + (size_t)row * V;
    for (int c = tid; c < V; c += kThreads) lr[c] = zr[c] - lse;
  }

  // ---- 2. radix selection of the k-th largest key
  if (tid == 0) {
    sh_prefix = 0;
    sh_want = (uint32_t)k;
  }
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < kWarps * 256; i += kThreads) (&hist[0][0])[i] = 0;
    __syncthreads();
    const uint32_t prefix = sh_prefix;
    const uint32_t hi_mask = shift == 24 ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int c = tid; c < V; c += kThreads) {
      const uint32_t key = okey(zr[c]);
      if ((key & hi_mask) == prefix) atomicAdd(&hist[warp][(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    // merge the warps' histograms: thread b < 256 owns bin b
    if (tid < 256) {
      uint32_t t = 0;
      for (int w = 0; w < kWarps; ++w) t += hist[w][tid];
      hist[0][tid] = t;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t want = sh_want, above = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (above + hist[0][d] >= want) break;
        above += hist[0][d];
      }
      sh_want = want - above;  // still to take at or below this digit
      sh_prefix = prefix | ((uint32_t)d << shift);
    }
    __syncthreads();
  }
  const uint32_t T = sh_prefix;  // key of the k-th largest value
  const uint32_t n_eq = sh_want;   // how many of the elements equal to it are taken

  // ---- 3. candidates: every element above T, the lowest-index n_eq equal to T
  const int run = (V + kThreads - 1) / kThreads;
  const int c0 = tid * run, c1 = min(V, c0 + run);
  int my_eq = 0;
  for (int c = c0; c < c1; ++c) my_eq += okey(zr[c]) == T;
  scan[tid] = my_eq;
  if (tid == 0) cand_n = 0;
  __syncthreads();
  for (int o = 1; o < kThreads; o <<= 1) {  // inclusive prefix sum over the threads
    const int add = tid >= o ? scan[tid - o] : 0;
    __syncthreads();
    scan[tid] += add;
    __syncthreads();
  }
  int rank = scan[tid] - my_eq;  // equal elements before this thread's run
  for (int c = c0; c < c1; ++c) {
    const float v = zr[c];
    const uint32_t key = okey(v);
    bool take = key > T;
    if (key == T) {
      take = (uint32_t)rank < n_eq;
      ++rank;
    }
    if (take) {
      const int slot = atomicAdd(&cand_n, 1);
      if (slot < kMaxK) {
        cand_i[slot] = c;
        cand_v[slot] = v;
      }
    }
  }
  __syncthreads();

  // ---- 4. rank the candidates: value descending, index ascending
  if (tid < k) {
    const float v = cand_v[tid];
    const int id = cand_i[tid];
    int r = 0;
    for (int j = 0; j < k; ++j) {
      const float vj = cand_v[j];
      r += (vj > v) || (vj == v && cand_i[j] < id);
    }
    top_ids[(size_t)row * k + r] = id;
    top_lp[(size_t)row * k + r] = v - lse;
  }
}

}  // namespace

}  // namespace fk

extern "C" fk_status fk_op_logsoftmax_topk(const float* d_logits, int32_t rows, int32_t vocab, int32_t ld, int32_t k,
                                           float* d_lse, int32_t* d_top_ids, float* d_top_logprobs,
                                           float* d_logprobs, void* stream) {
  using fk::fail;
  if (!d_logits || !d_top_ids || !d_top_logprobs || rows < 1 || vocab < 1 || ld < vocab)
    return fail(FK_ERR_INVALID_ARG, "fk_op_logsoftmax_topk: bad argument");
  if (k < 1 || k > fk::kMaxK || k > vocab)
    return fail(FK_ERR_INVALID_ARG, "fk_op_logsoftmax_topk: need 1 <= k <= min(128, vocab)");
  fk_status s = fk::check_device(nullptr);
  if (s != FK_OK) return s;
  fk::logsoftmax_topk_kernel<<<rows, fk::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      d_logits, vocab, ld, k, d_lse, d_top_ids, d_top_logprobs, d_logprobs);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fk::cuda_fail(e, "logsoftmax_topk_kernel launch");
  return FK_OK;
}
