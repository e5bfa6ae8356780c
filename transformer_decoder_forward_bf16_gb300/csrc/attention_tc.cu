// Causal GQA flash attention for prefill on the 5th-generation tensor cores
// ("N7 · model/forward-parity", Thm 1: causal multi-head/GQA attention;
// Thm 2 and "pegainfer #878": sliding-window local layers).
//
// One CTA per (128 queries, head, sequence); key blocks of 64 positions; two
// CTAs per SM (shared memory and TMEM both sized for it) so each scheduler
// runs two softmax warps.
//   warp 0     TMA producer: the Q tile once, then K and Vᵀ tiles through a
//              2-stage ring (all 128-byte swizzled, K-major).
//   warp 1     TMEM allocator and single-thread MMA issuer:
//                S_j = Q·K_jᵀ   (M=128 queries, N=64 keys) into one of two
//                               TMEM S buffers, issued one block ahead;
//                O  += P_j·V_j  (M=128, N=head_dim) into the TMEM O buffer.
//   warps 2-5  softmax, one query row per thread (TMEM lane = row): read S_j,
//              mask (causal, window, sequence end), running max in the exp2
//              domain, P = exp2(S - m) rounded to bf16 into shared memory for
//              the PV MMA. The running max is raised lazily: O and the row sum
//              are rescaled (tcgen05.ld/st on O) only when the max grows by
//              more than 2^8, so most blocks skip the rescale; P <= 2^8 keeps
//              bf16 well inside range. At the end O / l is stored as bf16.
// Every mbarrier wait is bounded (FK_DEVERR_PIPE_TIMEOUT on expiry). Every
// tcgen05.ld/st is executed by whole warps (they are warp-collective), so
// per-row decisions that touch TMEM are taken warp-wide.
#include <algorithm>
#include <mutex>

#include "fk_common.cuh"
#include "fk_internal.h"
#include "fk_ops.h"

namespace fk {

namespace {

constexpr int kThreads = 192;
constexpr int BQ = 128, BKV = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyRescale = 8.0f;  // log2 units

template <int HD>
struct FaCfg {
  static constexpr int Q_BYTES = BQ * HD * 2;   // HD/64 column blocks of [128 rows][128 B]
  static constexpr int K_BYTES = BKV * HD * 2;  // HD/64 column blocks of [128 keys][128 B]
  static constexpr int V_BYTES = HD * BKV * 2;  // BKV/64 column blocks of [HD rows][128 B]
  static constexpr int P_BYTES = BQ * BKV * 2;  // BKV/64 column blocks of [128 rows][128 B]
  static constexpr int STAGES = 2;
  // tiles then 128 bytes of barriers; no alignment slack (two CTAs must fit
  // in an SM): the dynamic window starts 1024-byte aligned, checked on entry
  static constexpr int SMEM = Q_BYTES + STAGES * (K_BYTES + V_BYTES) + P_BYTES + 128;
  // S0 [0,BKV), S1 [BKV,2 BKV), O [2 BKV, 2 BKV + HD): 256 columns, two CTAs per SM
  static constexpr uint32_t TMEM_COLS = 2 * BKV + HD <= 256 ? 256 : 512;
  static constexpr uint32_t O_COL = 2 * BKV;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BQ, BKV);
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(BQ, HD);
};

FK_DEVICE void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
// 2^x with the hardware approximation (ex2.approx, relative error ~2^-22,
// far below the bf16 rounding P receives next).
FK_DEVICE float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
FK_DEVICE void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
FK_DEVICE void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int HD>
__global__ void __launch_bounds__(kThreads, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, int S, int pos0, int Hq, int Hkv, int cap, int window,
                   float scale_log2, __nv_bfloat16* __restrict__ out, unsigned* dev_err) {
  using C = FaCfg<HD>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && dev_err) atomicOr(dev_err, FK_DEVERR_PIPE_TIMEOUT);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::Q_BYTES;                      // [STAGES][K_BYTES]
  uint8_t* sV = sK + C::STAGES * C::K_BYTES;          // [STAGES][V_BYTES]
  uint8_t* sP = sV + C::STAGES * C::V_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + C::P_BYTES);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;
  uint64_t* pv_done = bars + 8;
  uint64_t* mma_done = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hb = blockIdx.x;  // (head, sequence), fastest: the first wave covers every head
  const int h = hb % Hq, b = hb / Hq;
  const int nqb = (S + BQ - 1) / BQ;
  const int qb = nqb - 1 - (int)blockIdx.y;  // longest (latest) query blocks first
  const int g = h / (Hq / Hkv);
  const int kv_len = pos0 + S;
  const int q_lo = qb * BQ;
  const int q_hi = min(S, q_lo + BQ) - 1;
  const int qp_lo = pos0 + q_lo, qp_hi = pos0 + q_hi;
  const int k_lo = window > 0 ? max(0, qp_lo - window + 1) : 0;
  const int kb_lo = k_lo / BKV, kb_hi = qp_hi / BKV;
  const int nkb = kb_hi - kb_lo + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&s_full[i], 1);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
      for (int blk = 0; blk < HD / 64; ++blk)
        tma_load_2d(&tmQ, q_full, sQ + blk * BQ * 128, h * HD + blk * 64, b * S + q_lo);
      const int krow = (b * Hkv + g) * cap;
      const int vrow = (b * Hkv + g) * HD;
      int issued[2] = {0, 0};
      for (int j = 0; j < nkb; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&kv_empty[st], ((j >> 1) & 1) ^ 1, abort_flag, dev_err)) break;
        mbar_arrive_expect_tx(&kv_full[st], C::K_BYTES + C::V_BYTES);
        const int kb = kb_lo + j;
#pragma unroll
        for (int blk = 0; blk < HD / 64; ++blk)
          tma_load_2d(&tmK, &kv_full[st], sK + st * C::K_BYTES + blk * BKV * 128, blk * 64, krow + kb * BKV);
#pragma unroll
        for (int blk = 0; blk < BKV / 64; ++blk)
          tma_load_2d(&tmV, &kv_full[st], sV + st * C::V_BYTES + blk * HD * 128, kb * BKV + blk * 64, vrow);
        ++issued[st];
      }
      if (*abort_flag) {  // let issued copies land before the CTA unwinds
        for (int st = 0; st < 2; ++st) {
          if (!issued[st]) continue;
          const uint32_t a = smem_u32(&kv_full[st]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a, (issued[st] - 1) & 1) && globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      bool ok = mbar_wait(q_full, 0, abort_flag, dev_err);
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&kv_full[st], (j >> 1) & 1, abort_flag, dev_err)) return false;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(j & 1) * BKV;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint64_t ad = smem_desc_sw128(sQ + (k >> 2) * BQ * 128) + 2 * (k & 3);
          const uint64_t bd = smem_desc_sw128(sK + st * C::K_BYTES + (k >> 2) * BKV * 128) + 2 * (k & 3);
          umma_bf16(d, ad, bd, C::IDESC_S, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nkb && ok; ++j) {
        if (j + 1 < nkb && !issue_s(j + 1)) break;
        if (!mbar_wait(p_full, j & 1, abort_flag, dev_err)) break;
        tc_fence_after();
        const int st = j & 1;
#pragma unroll
        for (int k = 0; k < BKV / 16; ++k) {
          const uint64_t ad = smem_desc_sw128(sP + (k >> 2) * BQ * 128) + 2 * (k & 3);
          const uint64_t bd = smem_desc_sw128(sV + st * C::V_BYTES + (k >> 2) * HD * 128) + 2 * (k & 3);
          umma_bf16(tmem + C::O_COL, ad, bd, C::IDESC_O, (j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(pv_done);
        umma_commit(&kv_empty[st]);
      }
      umma_commit(mma_done);
      const uint32_t a = smem_u32(mma_done);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else {
    // ---------------- softmax (warps 2-5) ----------------
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // query row of this thread = TMEM lane
    const int qp = qp_lo + r;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkb && ok; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, dev_err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_addr = lane_base + (uint32_t)(j & 1) * BKV;
      const int key0 = (kb_lo + j) * BKV;
      const bool edge = (key0 + BKV - 1 > qp_lo) || (key0 + BKV > kv_len) || (window > 0 && qp_hi - key0 >= window);
      float v[32];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) {
        tmem_ld32(s_addr + c * 32, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x = v[e] * scale_log2;
          if (edge) {
            const int key = key0 + c * 32 + e;
            if (!(key <= qp && key < kv_len && (window == 0 || qp - key < window))) x = -INFINITY;
          }
          mx = fmaxf(mx, x);
        }
      }
      const float m_new = fmaxf(m, mx);
      float m_use = m;
      bool rescale = false;
      if (m == -INFINITY) {
        m_use = m_new;  // nothing accumulated yet in this row (O and l are 0)
      } else if (m_new > m + kLazyRescale) {
        m_use = m_new;
        rescale = true;
      }
      // P_j goes into the single P buffer and O may be rescaled: PV_{j-1} must be done
      if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1, abort_flag, dev_err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // tcgen05.ld/st are warp-collective: the whole warp rescales when any of
      // its rows needs it, each lane with its own factor (1 for the others)
      if (__any_sync(0xffffffffu, rescale)) {
        const float corr = rescale ? exp2f(m - m_use) : 1.f;
        l *= corr;
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          tmem_ld32(lane_base + C::O_COL + c * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] *= corr;
          tmem_st32(lane_base + C::O_COL + c * 32, v);
        }
        tmem_st_wait();
      }
      m = m_use;
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) {
        tmem_ld32(s_addr + c * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p0, p1;
          {
            float x = v[e] * scale_log2;
            const int key = key0 + c * 32 + e;
            const bool okk = !edge || (key <= qp && key < kv_len && (window == 0 || qp - key < window));
            p0 = (okk && m_use != -INFINITY) ? fast_exp2(x - m_use) : 0.f;
          }
          {
            float x = v[e + 1] * scale_log2;
            const int key = key0 + c * 32 + e + 1;
            const bool okk = !edge || (key <= qp && key < kv_len && (window == 0 || qp - key < window));
            p1 = (okk && m_use != -INFINITY) ? fast_exp2(x - m_use) : 0.f;
          }
          l += p0 + p1;
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
        // 4 chunks of 8 keys; key chunk index ci = c*4 + i -> column block ci/8, chunk ci%8
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ci = c * 4 + i;
          uint8_t* dst = sP + (ci >> 3) * BQ * 128 + r * 128 + (((ci & 7) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // epilogue: O / l -> bf16
    const bool have = ok && mbar_wait(pv_done, (nkb - 1) & 1, abort_flag, dev_err);
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int qi = q_lo + r;
    __nv_bfloat16* orow = out + ((size_t)b * S + qi) * ((size_t)Hq * HD) + (size_t)h * HD;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      float v[32];
      tmem_ld32(lane_base + C::O_COL + c * 32, v);
      if (have && qi < S) {
#pragma unroll
        for (int e = 0; e < 32; e += 8)
          *reinterpret_cast<uint4*>(orow + c * 32 + e) =
              make_uint4(pack_bf16x2(v[e] * inv, v[e + 1] * inv), pack_bf16x2(v[e + 2] * inv, v[e + 3] * inv),
                         pack_bf16x2(v[e + 4] * inv, v[e + 5] * inv), pack_bf16x2(v[e + 6] * inv, v[e + 7] * inv));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int HD>
fk_status launch_tc(const void* q, int ldq, const void* kc, const void* vc, int cap, int B, int S, int pos0, int Hq,
                    int Hkv, int window, float scale, void* o, unsigned* dev_err, cudaStream_t st) {
  using C = FaCfg<HD>;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(attn_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (attr != cudaSuccess) return cuda_fail(attr, "cudaFuncSetAttribute(attn_tc)");
  CUtensorMap tQ, tK, tV;
  fk_status s = make_tmap_bf16(&tQ, q, (int64_t)B * S, ldq, ldq, BQ);
  if (s == FK_OK) s = make_tmap_bf16(&tK, kc, (int64_t)B * Hkv * cap, HD, HD, BKV);
  if (s == FK_OK) s = make_tmap_bf16(&tV, vc, (int64_t)B * Hkv * HD, cap, cap, HD);
  if (s != FK_OK) return s;
  const int nqb = (S + BQ - 1) / BQ;
  attn_tc_kernel<HD><<<dim3(Hq * B, nqb), kThreads, C::SMEM, st>>>(tQ, tK, tV, S, pos0, Hq, Hkv, cap, window,
                                                                   scale * kLog2e, static_cast<__nv_bfloat16*>(o),
                                                                   dev_err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_tc_kernel launch");
  return FK_OK;
}

}  // namespace

bool attention_prefill_tc_supported(int hd, int ldq, int cap) {
  return (hd == 64 || hd == 128) && ldq % 8 == 0 && cap % 64 == 0;
}

fk_status attention_prefill_tc(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B, int S,
                               int pos0, int Hq, int Hkv, int hd, int window, float scale, void* o,
                               unsigned* dev_err, cudaStream_t st) {
  if (B == 0 || S == 0) return FK_OK;
  if (hd == 64)
    return launch_tc<64>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, dev_err, st);
  if (hd == 128)
    return launch_tc<128>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, dev_err, st);
  return fail(FK_ERR_INVALID_ARG, "tensor-core attention: head_dim 64 or 128");
}

}  // namespace fk

extern "C" fk_status fk_attention_prefill(const void* d_q, const void* d_kcache, const void* d_vcache, int32_t batch,
                                          int32_t seq, int32_t pos0, int32_t n_q_heads, int32_t n_kv_heads,
                                          int32_t head_dim, int32_t cap, int32_t window, void* d_out, void* stream) {
  using namespace fk;
  if (!d_q || !d_kcache || !d_vcache || !d_out || batch < 1 || seq < 1 || pos0 < 0 || window < 0)
    return fail(FK_ERR_INVALID_ARG, "attention prefill: bad argument");
  if (n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads)
    return fail(FK_ERR_INVALID_ARG, "attention prefill: n_q_heads must be a multiple of n_kv_heads");
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(FK_ERR_INVALID_ARG, "attention prefill: head_dim 64/128/256");
  if (pos0 + seq > cap || cap % 64) return fail(FK_ERR_INVALID_ARG, "attention prefill: need pos0 + seq <= cap, cap % 64 == 0");
  if ((reinterpret_cast<uintptr_t>(d_q) | reinterpret_cast<uintptr_t>(d_kcache) |
       reinterpret_cast<uintptr_t>(d_vcache) | reinterpret_cast<uintptr_t>(d_out)) & 15)
    return fail(FK_ERR_INVALID_ARG, "attention prefill: buffers must be 16-byte aligned");
  fk_status s = check_device(nullptr);
  if (s != FK_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int ldq = n_q_heads * head_dim;
  const float scale = 1.0f / sqrtf((float)head_dim);
  if (attention_prefill_tc_supported(head_dim, ldq, cap))
    return attention_prefill_tc(d_q, ldq, d_kcache, d_vcache, cap, batch, seq, pos0, n_q_heads, n_kv_heads, head_dim,
                                window, scale, d_out, nullptr, st);
  cudaError_t e = launch_attention_prefill(d_q, ldq, d_kcache, d_vcache, cap, batch, seq, pos0, n_q_heads, n_kv_heads,
                                           head_dim, window, scale, d_out, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention prefill launch");
  return FK_OK;
}
