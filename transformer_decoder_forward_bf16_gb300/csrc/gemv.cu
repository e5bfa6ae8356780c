// Skinny GEMM for few tokens (decode, short prompts): out = epilogue(X · Wᵀ)
// with X [M <= 64, K] and a weight operand of up to three stacked matrices.
//
// The contraction is the projection of "N7 · model/forward-parity", Thm 1 (and
// "N9 · metalgemm", Thm 1: Y = X·Wᵀ); at M <= 64 it is bound by streaming the
// weights from HBM, so the kernel is laid out for bandwidth:
//   * operands swapped: the weight tile (128 output features x 64 K) is the
//     M=128 side of tcgen05.mma and the tokens are the N side (16/32/64), so
//     TMEM lane = output feature and column = token;
//   * split-K over a 2-D grid (feature tiles x K splits) sized to one wave
//     with the same number of CTAs on every SM (three at <= 16 tokens), each
//     streaming its weight slab through a 4-deep TMA ring (~190 KB of loads
//     in flight per SM);
//   * fp32 partial sums per split, added in a fixed order (bitwise-
//     reproducible) by the last CTA of each feature tile (<= 8 tokens) or by
//     one reduction kernel, which applies the fused epilogue (bf16 store,
//     fp32 + softcap, fp32 residual add, or the gated FFN activation
//     act(gate) * up);
//   * operands under 8 MB with K <= 1024 take a single split and apply the epilogue straight
//     from TMEM;
//   * an RMSNorm of the input may be fused in front (one or two tokens): the
//     two otherwise idle warps read the fp32 rows, form the inverse RMS and
//     write each k-block of the normalised 16-bit tokens into the pipeline
//     stage themselves, in the layout the TMA copy of a stored input would
//     have (the norm kernel and its launch boundary drop out of the chain).
#include <algorithm>

#include "fk_common.cuh"
#include "fk_internal.h"

namespace fk {

namespace {

constexpr int kThreads = 128;
constexpr int kStages = 4;
constexpr int A_BYTES = 128 * 64 * 2;

struct SkinnyArgs {
  int M, K, n_rows, nseg;
  int seg_start[4];
  int nk;  // k-blocks of 64; split s covers [s*nk/S, (s+1)*nk/S), S = gridDim.y
  float* part;  // [splits][M][n_rows]
  unsigned* dev_err;
  // fused reduction: the last CTA to finish a feature group sums the splits
  unsigned* counters;  // one per group, zero between launches (the last CTA resets it)
  int fused, glu_tiles;  // glu_tiles: feature tiles of one half of a gate|up pair (0 = not GLU)
  int direct;            // one split: the epilogue is applied straight from TMEM
  int epi, act, n_out, ldo, ldr;
  int ab_f16, out_f16;  // operand type (f16 or bf16); type of 16-bit outputs
  void* out;
  const float* res;
  float softcap;
  // fused input RMSNorm (xn != NULL): tokens = 16-bit(xn[t] * rsqrt(mean(xn[t]^2) + eps) * nw);
  // nssq (optional): the upstream GEMM's per-group sums of squares of xn, [M][n_ssq]
  const float* xn;
  int ldxn;
  const __nv_bfloat16* nw;
  float neps;
  const float* nssq;
  int n_ssq;
  // fused reduction of an EPI_ADD_F32 output: per 128-feature group sums of
  // squares of each stored row, [M][gridDim.x] (for a fused norm downstream)
  float* ssq_out;
};

FK_DEVICE float act_silu(float g) { return g / (1.0f + expf(-g)); }
FK_DEVICE float act_gelu_tanh(float g) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * g * (1.0f + tanhf(k0 * (g + 0.044715f * g * g * g)));
}

// The epilogue for output feature f of token t: v = the sum over K (the gate
// for GLU), u = the up projection (GLU only).
FK_DEVICE void store_out(const SkinnyArgs& a, int t, int f, float v, float u) {
  if (a.epi == EPI_GLU_BF16) {
    store_16(static_cast<uint16_t*>(a.out) + (size_t)t * a.ldo + f, (a.act ? act_gelu_tanh(v) : act_silu(v)) * u,
             a.out_f16);
  } else if (a.epi == EPI_BF16) {
    store_16(static_cast<uint16_t*>(a.out) + (size_t)t * a.ldo + f, v, a.out_f16);
  } else if (a.epi == EPI_ADD_F32) {
    static_cast<float*>(a.out)[(size_t)t * a.ldo + f] = a.res[(size_t)t * a.ldr + f] + v;
  } else {
    static_cast<float*>(a.out)[(size_t)t * a.ldo + f] = a.softcap > 0.f ? a.softcap * tanhf(v / a.softcap) : v;
  }
}

// Sum the splits of one feature for every token (fixed split order) and store
// the epilogue's result. v: gate (or plain) feature f, u: up feature (GLU).
FK_DEVICE void reduce_store(const SkinnyArgs& a, int S, int f) {
  constexpr int U = 16;  // splits loaded per batch (all in flight before the in-order adds)
  const size_t sstride = (size_t)a.M * a.n_rows;
  for (int t = 0; t < a.M; ++t) {
    float v = 0.f, u = 0.f;
    const float* p = a.part + (size_t)t * a.n_rows + f;
    for (int s0 = 0; s0 < S; s0 += U) {
      float tv[U], tu[U];
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const bool in = s0 + j < S;
        tv[j] = in ? __ldcg(p + (size_t)(s0 + j) * sstride) : 0.f;
        tu[j] = in && a.glu_tiles ? __ldcg(p + (size_t)(s0 + j) * sstride + a.n_out) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        v += tv[j];
        u += tu[j];
      }
    }
    store_out(a, t, f, v, u);
  }
}

template <int BT>
struct SCfg {
  static constexpr int B_BYTES = BT * 64 * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int SMEM = kStages * STAGE + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = BT < 32 ? 32 : BT;
};

template <int BT>
__global__ void __launch_bounds__(kThreads) gemv_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                                                           const __grid_constant__ CUtensorMap tmW0,
                                                           const __grid_constant__ CUtensorMap tmW1,
                                                           const __grid_constant__ CUtensorMap tmW2,
                                                           const SkinnyArgs args) {
  using C = SCfg<BT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * C::STAGE);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  __shared__ int s_norm_ok;            // fused norm: the stage wait's outcome, for both warps
  __shared__ float s_ssq[4][kNormFuseMaxTokens];  // per-warp sums of squares of stored rows
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * 128;
  const int split = blockIdx.y;
  const int kb0 = (int)((long)split * args.nk / gridDim.y);
  const int kb1 = (int)((long)(split + 1) * args.nk / gridDim.y);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], args.xn ? 2 : 1);  // fused norm: the token tile's writers arrive too
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW0);
    if (args.nseg > 1) tma_prefetch_desc(&tmW1);
    if (args.nseg > 2) tma_prefetch_desc(&tmW2);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The dependent kernel is released only after this grid's wait, i.e. once
  // every kernel before this one has completed: a dependent may then read,
  // before its own wait, anything those kernels wrote (the decode attention
  // reads the KV cache's earlier positions while this projection runs).
  if (!(warp == 0 && lane == 0)) {
    pdl_wait();
    pdl_trigger();
  }
  if (warp == 0 && lane == 0) {
    // ---- producer: two 64-row weight boxes + one token box per stage. The
    // weights do not depend on the previous kernel, so the first stages are
    // requested before waiting for it; the token rows only after.
    const CUtensorMap* maps[3] = {&tmW0, &tmW1, &tmW2};
    int map[2], row[2];
    bool valid[2];
    uint32_t bytes = args.xn ? 0u : (uint32_t)C::B_BYTES;  // fused norm: no token-tile copy
    for (int i = 0; i < 2; ++i) {
      const int v = n0 + i * 64;
      int m = 0;
      if (args.nseg > 1 && v >= args.seg_start[1]) m = 1;
      if (args.nseg > 2 && v >= args.seg_start[2]) m = 2;
      map[i] = m;
      row[i] = v - args.seg_start[m];
      valid[i] = v < args.n_rows;
      if (valid[i]) bytes += 64 * 64 * 2;
    }
    const uint64_t evict_first = l2_policy_evict_first();
    int issued[kStages] = {0, 0, 0, 0};
    bool ok = true;
    const int npre = min(kStages, kb1 - kb0);
    // test control (word 2 of the control block): leave stage 0 unarmed, so
    // the MMA issuer's bounded wait on it runs out
    const bool stall = args.dev_err && *reinterpret_cast<volatile unsigned*>(args.dev_err + 2) != 0;
    for (int it = 0; it < npre; ++it) {  // fresh ring: every stage is free
      if (stall && it == 0) continue;
      uint8_t* sa = smem + it * C::STAGE;
      mbar_arrive_expect_tx(&full[it], bytes);
      for (int i = 0; i < 2; ++i)
        if (valid[i])
          tma_load_2d_hint(maps[map[i]], &full[it], sa + i * 64 * 128, (kb0 + it) * 64, row[i], evict_first);
    }
    pdl_wait();
    pdl_trigger();
    for (int it = 0; it < npre; ++it) {
      if (stall && it == 0) continue;
      if (!args.xn) tma_load_2d(&tmX, &full[it], smem + it * C::STAGE + A_BYTES, (kb0 + it) * 64, 0);
      ++issued[it];
    }
    for (int kb = kb0 + npre, it = npre; kb < kb1; ++kb, ++it) {
      const int stage = it % kStages;
      const uint32_t phase = (it / kStages) & 1;
      if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.dev_err)) {
        ok = false;
        break;
      }
      uint8_t* sa = smem + stage * C::STAGE;
      mbar_arrive_expect_tx(&full[stage], bytes);
      for (int i = 0; i < 2; ++i)
        if (valid[i])
          tma_load_2d_hint(maps[map[i]], &full[stage], sa + i * 64 * 128, kb * 64, row[i], evict_first);
      if (!args.xn) tma_load_2d(&tmX, &full[stage], sa + A_BYTES, kb * 64, 0);
      ++issued[stage];
    }
    if (!ok) {
      for (int s = 0; s < kStages; ++s) {
        if (issued[s] == 0) continue;
        const uint32_t a = smem_u32(&full[s]);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(a, (issued[s] - 1) & 1) && globaltimer_ns() - t0 < 100000000ull) {
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer
    const uint32_t idesc = idesc_16b_f32(128, BT, args.ab_f16);
    for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
      const int stage = it % kStages;
      const uint32_t phase = (it / kStages) & 1;
      if (!mbar_wait(&full[stage], phase, abort_flag, args.dev_err)) break;
      tc_fence_after();
      uint8_t* sa = smem + stage * C::STAGE;
      const uint64_t ad = smem_desc_sw128(sa);
      const uint64_t bd = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
      for (int k = 0; k < 4; ++k) umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (it | k) != 0 ? 1u : 0u);
      umma_commit(&empty[stage]);
    }
    umma_commit(done);
  } else if (args.xn && warp >= 2) {
    // ---- fused input RMSNorm: warp 2 writes token 0's row of every stage's
    // token tile, warp 3 token 1's (at most kNormFuseMaxTokens tokens)
    const int nt = threadIdx.x - 64;  // 0..63
    const int M = args.M, K = args.K;
    const int t = warp - 2, pc = lane * 2;  // this thread's token row and column pair of a k-block
    const bool act = t < M;
    // rows M..BT-1 of the token tiles stay zero
    for (int i = nt; i < kStages * (C::B_BYTES / 16); i += 64) {
      const int stage = i / (C::B_BYTES / 16), chunk = i % (C::B_BYTES / 16);
      if (chunk >= M * 8) *reinterpret_cast<uint4*>(smem + stage * C::STAGE + A_BYTES + chunk * 16) = make_uint4(0, 0, 0, 0);
    }
    const float* xr = args.xn + (size_t)(act ? t : 0) * args.ldxn;
    // the first stages' inputs are requested with the row statistics (one round trip)
    float2 xv[kStages];
    uint32_t wv[kStages];
#pragma unroll
    for (int j = 0; j < kStages; ++j) {
      const int col = (kb0 + j) * 64 + pc;
      const bool in = act && kb0 + j < kb1 && col < K;
      xv[j] = in ? __ldcg(reinterpret_cast<const float2*>(xr + col)) : make_float2(0.f, 0.f);
      wv[j] = in ? *reinterpret_cast<const uint32_t*>(args.nw + col) : 0u;
    }
    float q = 0.f;
    if (args.nssq) {  // the upstream reduction's group sums, in group order
      if (act)
        for (int g = lane; g < args.n_ssq; g += 32) q += __ldcg(args.nssq + (size_t)t * args.n_ssq + g);
    } else if (act) {  // the whole row
#pragma unroll 8
      for (int c = lane * 4; c < K; c += 128) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(xr + c));
        q += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
    }
    const float inv = rsqrtf(warp_sum(q) / K + args.neps);
    auto write = [&](int stage, float2 x, uint32_t wp) {
      if (!act) return;
      uint8_t* xs = smem + stage * C::STAGE + A_BYTES;
      // 128-byte swizzle: 16-byte chunk j of row t sits at chunk position j ^ (t % 8)
      *reinterpret_cast<uint32_t*>(xs + t * 128 + ((((pc * 2) >> 4) ^ (t & 7)) << 4) + ((pc * 2) & 15)) =
          pack_16x2(x.x * inv * bf16_lo(wp), x.y * inv * bf16_hi(wp), args.ab_f16);
    };
    auto publish = [&](int stage) {  // the tile's writes, then one arrival for both warps
      fence_proxy_async_smem();
      asm volatile("bar.sync 1, 64;" ::: "memory");
      if (nt == 0) mbar_arrive(&full[stage]);
    };
#pragma unroll
    for (int j = 0; j < kStages; ++j) {  // fresh ring: every stage is free
      if (kb0 + j >= kb1) break;
      write(j, xv[j], wv[j]);
      publish(j);
    }
    for (int kb = kb0 + kStages, it = kStages; kb < kb1; ++kb, ++it) {
      const int stage = it % kStages;
      // the stage's previous k-block has been consumed (one waiter, then both warps)
      if (nt == 0) s_norm_ok = mbar_wait(&empty[stage], ((it / kStages) - 1) & 1, abort_flag, args.dev_err);
      asm volatile("bar.sync 1, 64;" ::: "memory");
      if (!s_norm_ok) break;
      const int col = kb * 64 + pc;
      const bool in = act && col < K;
      write(stage, in ? __ldcg(reinterpret_cast<const float2*>(xr + col)) : make_float2(0.f, 0.f),
            in ? *reinterpret_cast<const uint32_t*>(args.nw + col) : 0u);
      publish(stage);
    }
  }
  __syncwarp();
  // ---- epilogue: every warp drains its 32 TMEM lanes (= 32 output features)
  const bool have = mbar_wait(done, 0, abort_flag, args.dev_err);
  tc_fence_after();
  const int feat = n0 + warp * 32 + lane;
  if (args.direct) {  // one split: the epilogue straight from TMEM
#pragma unroll
    for (int c0 = 0; c0 < (BT < 32 ? 32 : BT); c0 += 32) {
      float v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
      if (have && feat < args.n_rows) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j < args.M) store_out(args, c0 + j, feat, v[j], 0.f);
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
    return;
  }
  float* part = args.part + (size_t)split * args.M * args.n_rows;
#pragma unroll
  for (int c0 = 0; c0 < (BT < 32 ? 32 : BT); c0 += 32) {
    float v[32];
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
    if (have && feat < args.n_rows && kb1 > kb0) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < args.M) part[(size_t)(c0 + j) * args.n_rows + feat] = v[j];
    } else if (have && feat < args.n_rows) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < args.M) part[(size_t)(c0 + j) * args.n_rows + feat] = 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (!args.fused) return;
  // ---- fused split-K reduction: the last CTA of this feature group finishes it.
  // A CTA whose pipeline gave up (the error word is set; its partials are
  // not valid) still takes part in the arrival, so the counter returns to
  // zero for the next launch.
  volatile int* last = abort_flag + 1;
  const int group = args.glu_tiles ? (int)blockIdx.x % args.glu_tiles : (int)blockIdx.x;
  const unsigned expect = gridDim.y * (args.glu_tiles ? 2u : 1u);
  // The CTA barrier orders every thread's partial stores before thread 0's
  // arrival; thread 0's acquire-release atomic publishes them at GPU scope
  // and, in the last CTA, acquires every other CTA's partials (the barrier
  // after it extends that to all threads of the CTA).
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(&args.counters[group]) : "memory");
    *last = prev == expect - 1 ? 1 : 0;
  }
  __syncthreads();
  if (!*last) return;
  const int f = group * 128 + threadIdx.x;
  if (f < args.n_out) reduce_store(args, gridDim.y, f);
  if (threadIdx.x == 0) args.counters[group] = 0;
  if (args.ssq_out) {  // this group's sum of squares of every stored row (fixed order)
    for (int t = 0; t < args.M; ++t) {
      const float y = f < args.n_out ? static_cast<const float*>(args.out)[(size_t)t * args.ldo + f] : 0.f;
      const float q = warp_sum(y * y);
      if (lane == 0) s_ssq[warp][t] = q;
    }
    __syncthreads();
    if (threadIdx.x < args.M)
      args.ssq_out[(size_t)threadIdx.x * gridDim.x + group] =
          ((s_ssq[0][threadIdx.x] + s_ssq[1][threadIdx.x]) + s_ssq[2][threadIdx.x]) + s_ssq[3][threadIdx.x];
  }
}

// Sum the splits in order and apply the epilogue; one thread per (token, 4 features).
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int S, int M, int n_rows, int n_out, int epi,
                                     int act, void* out, int ldo, const float* res, int ldr, float softcap,
                                     int out_f16) {
  pdl_trigger();
  pdl_wait();
  const int per_row = (n_out + 3) / 4;
  const long total = (long)M * per_row;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int t = (int)(i / per_row);
    const int f = (int)(i % per_row) * 4;
    const int nf = min(4, n_out - f);
    float v[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < S; ++s) {
      const float* p = part + ((size_t)s * M + t) * n_rows;
      for (int j = 0; j < nf; ++j) v[j] += p[f + j];
      if (epi == EPI_GLU_BF16)
        for (int j = 0; j < nf; ++j) u[j] += p[n_out + f + j];
    }
    if (epi == EPI_GLU_BF16) {
      uint16_t* o = static_cast<uint16_t*>(out) + (size_t)t * ldo + f;
      for (int j = 0; j < nf; ++j) store_16(o + j, (act ? act_gelu_tanh(v[j]) : act_silu(v[j])) * u[j], out_f16);
    } else if (epi == EPI_BF16) {
      uint16_t* o = static_cast<uint16_t*>(out) + (size_t)t * ldo + f;
      for (int j = 0; j < nf; ++j) store_16(o + j, v[j], out_f16);
    } else if (epi == EPI_ADD_F32) {
      float* o = static_cast<float*>(out) + (size_t)t * ldo + f;
      const float* r = res + (size_t)t * ldr + f;
      for (int j = 0; j < nf; ++j) o[j] = r[j] + v[j];
    } else {
      float* o = static_cast<float*>(out) + (size_t)t * ldo + f;
      if (softcap > 0.f) {
        const float inv = 1.0f / softcap;
        for (int j = 0; j < nf; ++j) o[j] = softcap * tanhf(v[j] * inv);
      } else {
        for (int j = 0; j < nf; ++j) o[j] = v[j];
      }
    }
  }
}

template <int BT>
cudaError_t set_smem_attr() {
  static DeviceOnce once;
  return once.run([] {
    cudaError_t attr =
        cudaFuncSetAttribute(gemv_tc_kernel<BT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SCfg<BT>::SMEM);
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(gemv_tc_kernel<BT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared);
    return attr;
  });
}

template <int BT>
fk_status launch_bt(const CUtensorMap& tX, const GemmWeights& w, const SkinnyArgs& a, int n_tiles, int splits,
                    cudaStream_t st) {
  using C = SCfg<BT>;
  cudaError_t attr = set_smem_attr<BT>();
  if (attr != cudaSuccess) return cuda_fail(attr, "cudaFuncSetAttribute(gemv)");
  cudaError_t e = fk_launch(gemv_tc_kernel<BT>, dim3(n_tiles, splits), kThreads, C::SMEM, st, tX, w.map[0],
                            w.nseg > 1 ? w.map[1] : w.map[0], w.nseg > 2 ? w.map[2] : w.map[0], a);
  if (e != cudaSuccess) return cuda_fail(e, "gemv_tc_kernel launch");
  return FK_OK;
}

}  // namespace

// CTAs of the skinny kernel that fit on one SM at once: shared memory bound
// (the kernels ask for the largest shared-memory carveout, so this is the
// SM's whole shared memory over each CTA's dynamic + reserved bytes).
static int resident_per_sm(int M) {
  const int i = M <= 16 ? 0 : (M <= 32 ? 1 : 2);
  int dev = 0, smem_sm = 0, reserved = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  const int smem = i == 0 ? SCfg<16>::SMEM : (i == 1 ? SCfg<32>::SMEM : SCfg<64>::SMEM);
  return std::max(1, std::min(2048 / kThreads, smem_sm / (smem + reserved)));
}

// Small operands (under kDirectBytes of weights and kDirectMaxKBlocks k-blocks,
// not a gate/up pair) take a single split: the CTAs write the epilogue straight from TMEM, with no
// partial sums, arrival counters or ordered reduction on the critical path,
// which for so few bytes cost more than the split's extra bandwidth gains.
constexpr size_t kDirectBytes = 8u << 20;
constexpr int kDirectMaxKBlocks = 16;

// Split K so that the whole grid is one wave of resident CTAs, every SM
// holding the same number: each CTA starts at once and streams an equal
// share of the weights (splits differ by at most one k-block).
SkinnyPlan skinny_plan(int M, int K, int n_rows, int sm_count, bool allow_direct) {
  SkinnyPlan p;
  const int nk = (K + 63) / 64;
  const int n_tiles = (n_rows + 127) / 128;
  const int wave = resident_per_sm(M) * sm_count;
  // a single split streams 128 rows x K per CTA: only for short K (a router
  // of 128 experts x 2048 would leave one CTA streaming 512 KB)
  p.direct = allow_direct && (size_t)n_rows * K * 2 < kDirectBytes && nk <= kDirectMaxKBlocks;
  p.splits = p.direct ? 1 : std::max(1, std::min(nk, wave / n_tiles));
  p.kb_per_split = (nk + p.splits - 1) / p.splits;  // the longest split
  p.n_tiles = n_tiles;
  p.nk = nk;
  p.counter_bytes = ((size_t)n_tiles * sizeof(unsigned) + 255) / 256 * 256;
  p.part_bytes = p.counter_bytes + (p.direct ? 0 : (size_t)p.splits * M * n_rows * sizeof(float));
  return p;
}


bool skinny_fused_tail(const GemmWeights& w, int M, int sm_count, int epi) {
  if (epi != EPI_ADD_F32 || w.glu || M < 1 || M > kNormFuseMaxTokens) return false;
  return !skinny_plan(M, w.K, w.seg_start[w.nseg], sm_count, true).direct;
}

size_t skinny_counter_bytes(const GemmWeights& w, int M, int sm_count) {
  if (M <= 0 || M > kSkinnyMaxTokens) return 0;
  return skinny_plan(M, w.K, w.seg_start[w.nseg], sm_count, !w.glu).counter_bytes;
}

size_t skinny_partial_bytes(const GemmWeights& w, int M, int sm_count) {
  if (M <= 0 || M > kSkinnyMaxTokens) return 0;
  // splits depend on M only through the tile width (16/32/64 tokens): the
  // largest product of splits and tokens is at the top of a width class
  size_t b = 0;
  for (int m : {std::min(M, 16), std::min(M, 32), M}) {
    const SkinnyPlan p = skinny_plan(m, w.K, w.seg_start[w.nseg], sm_count, !w.glu);
    b = std::max(b, p.part_bytes - p.counter_bytes);
  }
  return b;
}

fk_status gemm_run_skinny(const void* A, int M, int lda, const GemmWeights& w, const GemmOut& o, void* scratch,
                          size_t scratch_bytes, unsigned* dev_err, cudaStream_t st, bool counters_zeroed,
                          size_t counter_region, const NormIn* norm) {
  int sms = 0;
  fk_status s = check_device(&sms);
  if (s != FK_OK) return s;
  if (norm && (M > kNormFuseMaxTokens || !norm->x || !norm->w || norm->ldx < w.K || norm->ldx % 4 || w.K % 4))
    return fail(FK_ERR_INVALID_ARG, "skinny GEMM: fused norm needs <= kNormFuseMaxTokens rows and fp32 rows of K");
  if (o.ssq && !skinny_fused_tail(w, M, sms, o.epi))
    return fail(FK_ERR_INVALID_ARG, "skinny GEMM: row sums of squares need the fused reduction of a residual output");
  const int n_rows = w.seg_start[w.nseg];
  const SkinnyPlan p = skinny_plan(M, w.K, n_rows, sms, !w.glu);
  const size_t creg = counter_region ? counter_region : p.counter_bytes;
  if (creg < p.counter_bytes || creg % 256) return fail(FK_ERR_INVALID_ARG, "skinny GEMM: counter region too small");
  if (!scratch || scratch_bytes < creg + (p.part_bytes - p.counter_bytes))
    return fail(FK_ERR_WORKSPACE, "skinny GEMM scratch too small");
  const int BT = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
  CUtensorMap tX;
  s = make_tmap_bf16(&tX, A, M, w.K, lda, BT);
  if (s != FK_OK) return s;
  const int n_out = w.glu ? w.n_out : n_rows;
  SkinnyArgs a{};
  a.M = M;
  a.K = w.K;
  a.n_rows = n_rows;
  a.nseg = w.nseg;
  for (int i = 0; i < 4; ++i) a.seg_start[i] = w.seg_start[i];
  a.nk = p.nk;
  a.counters = static_cast<unsigned*>(scratch);
  a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + creg);
  a.dev_err = dev_err;
  a.ab_f16 = w.f16;
  a.out_f16 = o.out_f16;
  // a gate|up pair fuses only when each half is a whole number of 128-row tiles
  // (the last CTA sums M x splits values per feature: worth it only for few tokens)
  a.direct = p.direct;
  a.fused = !p.direct && M <= 8 && !(w.glu && n_out % 128);
  a.glu_tiles = w.glu ? n_out / 128 : 0;
  a.epi = o.epi;
  a.act = o.act;
  a.n_out = n_out;
  a.out = o.out;
  a.ldo = o.ldo;
  a.res = o.res;
  a.ldr = o.ldr;
  a.softcap = o.softcap;
  if (norm) {
    a.xn = norm->x;
    a.ldxn = norm->ldx;
    a.nw = static_cast<const __nv_bfloat16*>(norm->w);
    a.neps = norm->eps;
    a.nssq = norm->ssq;
    a.n_ssq = norm->n_ssq;
  }
  a.ssq_out = o.ssq;
  if (a.fused && !counters_zeroed) FK_CUDA_TRY(cudaMemsetAsync(a.counters, 0, p.counter_bytes, st));
  if (BT == 16)
    s = launch_bt<16>(tX, w, a, p.n_tiles, p.splits, st);
  else if (BT == 32)
    s = launch_bt<32>(tX, w, a, p.n_tiles, p.splits, st);
  else
    s = launch_bt<64>(tX, w, a, p.n_tiles, p.splits, st);
  if (s != FK_OK || a.fused || a.direct) return s;
  const long work = (long)M * ((n_out + 3) / 4);
  const int blocks = (int)std::min<long>((work + 255) / 256, 8L * sms);
  cudaError_t e = fk_launch(splitk_reduce_kernel, blocks, 256, 0, st, (const float*)a.part, p.splits, M, n_rows, n_out,
                            o.epi, o.act, o.out, o.ldo, o.res, o.ldr, o.softcap, o.out_f16);
  if (e != cudaSuccess) return cuda_fail(e, "splitk_reduce_kernel launch");
  return FK_OK;
}

}  // namespace fk

extern "C" size_t fk_gemm_bf16_splitk_scratch_bytes(int32_t P, int32_t K, int32_t N) {
  if (P < 1 || P > fk::kSkinnyMaxTokens || K < 8 || N < 8) return 0;
  int sms = 0;
  if (fk::check_device(&sms) != FK_OK) return 0;
  return fk::skinny_plan(P, K, N, sms, true).part_bytes;
}

namespace fk {
// The op-level few-row GEMM over a scratch buffer of scratch_bytes at
// d_scratch (validation, then the split-K kernel with its counters cleared).
fk_status gemm_splitk_op(const void* d_x, const void* d_w, int P, int K, int N, void* d_y, int y_fp32,
                         void* d_scratch, size_t scratch_bytes, cudaStream_t st) {
  if (!d_x || !d_w || !d_y || P < 1 || P > kSkinnyMaxTokens || K <= 0 || N <= 0)
    return fail(FK_ERR_INVALID_ARG, "fk_gemm_bf16_splitk: bad argument (1 <= P <= 64)");
  if (K % 8 || N % 8) return fail(FK_ERR_INVALID_ARG, "fk_gemm_bf16_splitk: K and N must be multiples of 8");
  if ((reinterpret_cast<uintptr_t>(d_x) | reinterpret_cast<uintptr_t>(d_w) | reinterpret_cast<uintptr_t>(d_y) |
       reinterpret_cast<uintptr_t>(d_scratch)) & 15)
    return fail(FK_ERR_INVALID_ARG, "fk_gemm_bf16_splitk: buffers must be 16-byte aligned");
  GemmWeights w;
  const void* mats[1] = {d_w};
  int rows[1] = {N};
  fk_status s = gemm_weights_init(&w, mats, rows, 1, K, 0);
  if (s != FK_OK) return s;
  unsigned* ctl = nullptr;
  s = op_control_block(&ctl);
  if (s != FK_OK) return s;
  GemmOut o;
  o.epi = y_fp32 ? EPI_F32 : EPI_BF16;
  o.out = d_y;
  o.ldo = N;
  return gemm_run_skinny(d_x, P, K, w, o, d_scratch, scratch_bytes, ctl, st, false);
}
}  // namespace fk

extern "C" fk_status fk_gemm_bf16_splitk(const void* d_x, const void* d_w, int32_t P, int32_t K, int32_t N, void* d_y,
                                         int32_t y_fp32, void* d_scratch, size_t scratch_bytes, void* stream) {
  return fk::gemm_splitk_op(d_x, d_w, P, K, N, d_y, y_fp32, d_scratch, scratch_bytes,
                            static_cast<cudaStream_t>(stream));
}
