// Causal GQA flash attention for prefill on the 5th-generation tensor cores
// ("N7 · model/forward-parity", Thm 1: causal multi-head/GQA attention;
// Thm 2 and "pegainfer #878": sliding-window local layers).
//
// One CTA per (128 queries, head, sequence); key blocks of 64 positions; two
// CTAs per SM at head_dim 128 (96 KB of shared memory and 256 TMEM columns
// each), one at head_dim 256 (197 KB, 512 columns: O alone takes 256).
//   warp 0     TMA producers: lane 0 streams K tiles, lane 1 Vᵀ tiles, each
//              through its own 2-deep ring (128-byte swizzled, K-major), so
//              the K tile of block j+2 never waits behind the V tile of j.
//   warp 1     TMEM allocator and single-thread MMA issuer:
//                S_j = Q·K_jᵀ   (M=128 queries, N=64 keys) into TMEM buffer j%2,
//                               two blocks ahead of the softmax;
//                O  += P_j·V_j  with P_j read from TMEM (it overwrites S_j)
//                               and Vᵀ_j from shared memory; O in TMEM.
//   warps 2-5  softmax, one query row per thread (TMEM lane = row): one TMEM
//              read of S_j, mask (causal, window, sequence end), running max
//              in the exp2 domain, P = exp2(S - m) packed to 16 bits and stored
//              back into the same TMEM columns for the PV MMA. The running
//              max is raised lazily (only when it grows by more than 2^8), and
//              only then does a warp wait for the previous PV and rescale its
//              rows of O (tcgen05.ld/st); P <= 2^8 keeps bf16 and f16 in range.
// q, K, Vᵀ and P are bf16, or all IEEE f16 (io_f16); the output bf16 or f16.
// Every mbarrier wait is bounded (FK_DEVERR_PIPE_TIMEOUT on expiry). Every
// tcgen05.ld/st is executed by whole warps (they are warp-collective), so
// per-row decisions that touch TMEM are taken warp-wide.
#include <algorithm>

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
  static constexpr int K_BYTES = BKV * HD * 2;  // HD/64 column blocks of [64 keys][128 B]
  static constexpr int V_BYTES = HD * BKV * 2;  // one column block of [HD rows][128 B]
  static constexpr int STAGES = 2;
  // tiles then 256 bytes for 16 barriers and two words; no alignment slack:
  // the dynamic window starts 1024-byte aligned (checked on entry)
  static constexpr int SMEM = Q_BYTES + STAGES * (K_BYTES + V_BYTES) + 256;
  // S/P buffers [0, BKV) and [BKV, 2 BKV); O [2 BKV, 2 BKV + HD)
  static constexpr uint32_t TMEM_COLS = 2 * BKV + HD <= 256 ? 256 : 512;
  static constexpr uint32_t O_COL = 2 * BKV;
};

FK_DEVICE void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
FK_DEVICE void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] · B[smem]ᵀ (A operand read from TMEM: M lanes, K/2
// columns of packed bf16 pairs, lower k in the low half).
FK_DEVICE void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2^x with the hardware approximation (ex2.approx, relative error ~2^-22,
// far below the bf16 rounding P receives next).
FK_DEVICE float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int HD, bool F16>
__global__ void __launch_bounds__(kThreads, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, int S, int pos0, int Hq, int Hkv, int cap, int window,
                   float scale_log2, uint16_t* __restrict__ out, unsigned* dev_err, int out_f16) {
  constexpr int io_f16 = F16 ? 1 : 0;  // q, K, Vᵀ and P are IEEE f16 (else bf16)
  using C = FaCfg<HD>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && dev_err) atomicOr(dev_err, FK_DEVERR_PIPE_TIMEOUT);
    return;
  }
  uint8_t* sQ = smem_raw;
  uint8_t* sK = sQ + C::Q_BYTES;              // [STAGES][K_BYTES]
  uint8_t* sV = sK + C::STAGES * C::K_BYTES;  // [STAGES][V_BYTES]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + C::STAGES * C::V_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* k_empty = bars + 3;   // [2]
  uint64_t* v_full = bars + 5;    // [2]
  uint64_t* v_empty = bars + 7;   // [2]
  uint64_t* s_full = bars + 9;    // [2]
  uint64_t* p_full = bars + 11;   // [2]
  uint64_t* pv_done = bars + 13;  // [2]: PV_j commits to pv_done[j%2]
  uint64_t* mma_done = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
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
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
    }
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
    if (lane < 2) {
      // ---------------- TMA producers: lane 0 K (and Q), lane 1 Vᵀ ----------------
      const bool is_k = lane == 0;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      if (is_k) {
        mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
        for (int blk = 0; blk < HD / 64; ++blk)
          tma_load_2d(&tmQ, q_full, sQ + blk * BQ * 128, h * HD + blk * 64, b * S + q_lo);
      }
      const int krow = (b * Hkv + g) * cap;
      const int vrow = (b * Hkv + g) * HD;
      int issued[2] = {0, 0};
      for (int j = 0; j < nkb; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&empty[st], ((j >> 1) & 1) ^ 1, abort_flag, dev_err)) break;
        const int kb = kb_lo + j;
        if (is_k) {
          mbar_arrive_expect_tx(&full[st], C::K_BYTES);
#pragma unroll
          for (int blk = 0; blk < HD / 64; ++blk)
            tma_load_2d(&tmK, &full[st], sK + st * C::K_BYTES + blk * BKV * 128, blk * 64, krow + (kb * BKV) % cap);
        } else {
          mbar_arrive_expect_tx(&full[st], C::V_BYTES);
          tma_load_2d(&tmV, &full[st], sV + st * C::V_BYTES, (kb * BKV) % cap, vrow);
        }
        ++issued[st];
      }
      if (*abort_flag) {  // let issued copies land before the CTA unwinds
        for (int st = 0; st < 2; ++st) {
          if (!issued[st]) continue;
          const uint32_t a = smem_u32(&full[st]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a, (issued[st] - 1) & 1) && globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc_s = idesc_16b_f32(BQ, BKV, io_f16);  // S = Q K^T
      const uint32_t idesc_o = idesc_16b_f32(BQ, HD, io_f16);   // O += P V
      bool ok = mbar_wait(q_full, 0, abort_flag, dev_err);
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&k_full[st], (j >> 1) & 1, abort_flag, dev_err)) return false;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)st * BKV;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint64_t ad = smem_desc_sw128(sQ + (k >> 2) * BQ * 128) + 2 * (k & 3);
          const uint64_t bd = smem_desc_sw128(sK + st * C::K_BYTES + (k >> 2) * BKV * 128) + 2 * (k & 3);
          umma_bf16(d, ad, bd, idesc_s, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[st]);
        umma_commit(&k_empty[st]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && nkb > 1) ok = issue_s(1);
      for (int j = 0; j < nkb && ok; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&p_full[st], (j >> 1) & 1, abort_flag, dev_err)) break;
        if (!mbar_wait(&v_full[st], (j >> 1) & 1, abort_flag, dev_err)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < BKV / 16; ++k) {
          const uint64_t bd = smem_desc_sw128(sV + st * C::V_BYTES) + 2 * k;
          umma_bf16_ts(tmem + C::O_COL, tmem + (uint32_t)st * BKV + 8 * k, bd, idesc_o, (j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&pv_done[st]);
        umma_commit(&v_empty[st]);
        // S_{j+2} reuses this TMEM buffer: issued after PV_j, the tensor core
        // reads P_j before it writes S_{j+2}
        if (j + 2 < nkb && !issue_s(j + 2)) break;
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
    for (int j = 0; j < nkb; ++j) {
      const int st = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[st], (j >> 1) & 1, abort_flag, dev_err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t s_addr = lane_base + (uint32_t)st * BKV;
      const int key0 = (kb_lo + j) * BKV;
      const bool edge = (key0 + BKV - 1 > qp_lo) || (key0 + BKV > kv_len) || (window > 0 && qp_hi - key0 >= window);
      float x[BKV];
      tmem_ld32(s_addr, x);
      tmem_ld32(s_addr + 32, x + 32);
      float mx0 = -INFINITY, mx1 = -INFINITY;
      // masked and unmasked blocks take separate loops (edge is warp-uniform)
      if (edge) {
#pragma unroll
        for (int e = 0; e < BKV; e += 2) {
          float a0 = x[e] * scale_log2, a1 = x[e + 1] * scale_log2;
          const int k0 = key0 + e, k1 = k0 + 1;
          if (!(k0 <= qp && k0 < kv_len && (window == 0 || qp - k0 < window))) a0 = -INFINITY;
          if (!(k1 <= qp && k1 < kv_len && (window == 0 || qp - k1 < window))) a1 = -INFINITY;
          x[e] = a0;
          x[e + 1] = a1;
          mx0 = fmaxf(mx0, a0);
          mx1 = fmaxf(mx1, a1);
        }
      } else {
#pragma unroll
        for (int e = 0; e < BKV; e += 2) {
          x[e] *= scale_log2;
          x[e + 1] *= scale_log2;
          mx0 = fmaxf(mx0, x[e]);
          mx1 = fmaxf(mx1, x[e + 1]);
        }
      }
      const float m_new = fmaxf(m, fmaxf(mx0, mx1));
      float m_use = m;
      bool rescale = false;
      if (m == -INFINITY) {
        m_use = m_new;  // nothing accumulated in this row yet (O and l are 0)
      } else if (m_new > m + kLazyRescale) {
        m_use = m_new;
        rescale = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O may only change after the last issued PV (PV_{j-1}) is done
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, dev_err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float corr = rescale ? fast_exp2(m - m_use) : 1.f;
        l *= corr;
        float o[32];
#pragma unroll
        for (int c = 0; c < HD / 32; ++c) {
          tmem_ld32(lane_base + C::O_COL + c * 32, o);
          uint32_t ob[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) ob[e] = __float_as_uint(o[e] * corr);
          tmem_st32(lane_base + C::O_COL + c * 32, ob);
        }
        tmem_st_wait();
      }
      m = m_use;
      uint32_t pk[BKV / 2];
      const bool live = m_use != -INFINITY;
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int e = 0; e < BKV; e += 2) {
        const float p0 = live ? fast_exp2(x[e] - m_use) : 0.f;
        const float p1 = live ? fast_exp2(x[e + 1] - m_use) : 0.f;
        l0 += p0;
        l1 += p1;
        pk[e >> 1] = pack_16x2(p0, p1, io_f16);
      }
      l += l0 + l1;
      tmem_st32(s_addr, pk);  // P_j over S_j: 32 columns of bf16 pairs
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[st]);
    }
    // epilogue: O / l -> bf16
    const int jl = nkb - 1;
    const bool have =
        __all_sync(0xffffffffu, ok && mbar_wait(&pv_done[jl & 1], (jl >> 1) & 1, abort_flag, dev_err));
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int qi = q_lo + r;
    uint16_t* orow = out + ((size_t)b * S + qi) * ((size_t)Hq * HD) + (size_t)h * HD;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      float v[32];
      tmem_ld32(lane_base + C::O_COL + c * 32, v);
      if (have && qi < S) {
#pragma unroll
        for (int e = 0; e < 32; e += 8)
          *reinterpret_cast<uint4*>(orow + c * 32 + e) =
              make_uint4(pack_16x2(v[e] * inv, v[e + 1] * inv, out_f16), pack_16x2(v[e + 2] * inv, v[e + 3] * inv, out_f16),
                         pack_16x2(v[e + 4] * inv, v[e + 5] * inv, out_f16),
                         pack_16x2(v[e + 6] * inv, v[e + 7] * inv, out_f16));
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
                    int Hkv, int window, float scale, void* o, unsigned* dev_err, cudaStream_t st, int io_f16,
                    int out_f16) {
  using C = FaCfg<HD>;
  static DeviceOnce once;
  const cudaError_t attr = once.run([] {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_tc_kernel<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    return e;
  });
  if (attr != cudaSuccess) return cuda_fail(attr, "cudaFuncSetAttribute(attn_tc)");
  CUtensorMap tQ, tK, tV;
  fk_status s = make_tmap_bf16(&tQ, q, (int64_t)B * S, ldq, ldq, BQ);
  if (s == FK_OK) s = make_tmap_bf16(&tK, kc, (int64_t)B * Hkv * cap, HD, HD, BKV);
  if (s == FK_OK) s = make_tmap_bf16(&tV, vc, (int64_t)B * Hkv * HD, cap, cap, HD);
  if (s != FK_OK) return s;
  const int nqb = (S + BQ - 1) / BQ;
  auto kernel = io_f16 ? attn_tc_kernel<HD, true> : attn_tc_kernel<HD, false>;
  kernel<<<dim3(Hq * B, nqb), kThreads, C::SMEM, st>>>(tQ, tK, tV, S, pos0, Hq, Hkv, cap, window, scale * kLog2e,
                                                       static_cast<uint16_t*>(o), dev_err, out_f16);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_tc_kernel launch");
  return FK_OK;
}

}  // namespace

fk_status attention_prefill_tc(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B, int S,
                               int pos0, int Hq, int Hkv, int hd, int window, float scale, void* o,
                               unsigned* dev_err, cudaStream_t st, int io_f16, int out_f16) {
  if (B == 0 || S == 0) return FK_OK;
  if (ldq % 8 || cap % 64) return fail(FK_ERR_INVALID_ARG, "tensor-core attention: ldq % 8 and cap % 64 must be 0");
  if (hd == 64 || hd == 128)
    return attention_prefill_pp(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, hd, window, scale, o, dev_err, st,
                                io_f16, out_f16);
  if (hd == 64)
    return launch_tc<64>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, dev_err, st, io_f16,
                           out_f16);
  if (hd == 128)
    return launch_tc<128>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, dev_err, st, io_f16,
                           out_f16);
  if (hd == 256)
    return launch_tc<256>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, dev_err, st, io_f16,
                           out_f16);
  return fail(FK_ERR_INVALID_ARG, "tensor-core attention: head_dim 64, 128 or 256");
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
  // position p lives in slot p mod cap: every key a query reads must still be
  // there, so either nothing wrapped or the window plus the chunk fits
  if (cap < 64 || cap % 64 || (pos0 + seq > cap && (window == 0 || window + seq - 1 > cap)))
    return fail(FK_ERR_INVALID_ARG,
                "attention prefill: need cap % 64 == 0 and pos0 + seq <= cap (or window + seq - 1 <= cap)");
  if ((reinterpret_cast<uintptr_t>(d_q) | reinterpret_cast<uintptr_t>(d_kcache) |
       reinterpret_cast<uintptr_t>(d_vcache) | reinterpret_cast<uintptr_t>(d_out)) & 15)
    return fail(FK_ERR_INVALID_ARG, "attention prefill: buffers must be 16-byte aligned");
  fk_status s = check_device(nullptr);
  if (s != FK_OK) return s;
  unsigned* ctl = nullptr;
  s = op_control_block(&ctl);
  if (s != FK_OK) return s;
  const int ldq = n_q_heads * head_dim;
  return attention_prefill_tc(d_q, ldq, d_kcache, d_vcache, cap, batch, seq, pos0, n_q_heads, n_kv_heads, head_dim,
                              window, 1.0f / sqrtf((float)head_dim), d_out, ctl, static_cast<cudaStream_t>(stream));
}
