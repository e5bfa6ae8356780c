// Causal GQA attention over the bf16 KV cache ("N7 · model/forward-parity",
// Thm 1: causal multi-head/GQA attention; Thm 2 and "pegainfer #878":
// sliding-window local layers).
//
// Prefill: flash-style, one CTA per (64 queries, head, sequence), 4 warps x 16
// query rows, 64-key blocks double-buffered in shared memory with cp.async,
// QKᵀ and PV on tensor cores (mma.sync m16n8k16 bf16, fp32 accumulate), online
// softmax in fp32 (exp2 domain), P rounded to bf16 for the PV product.
// Only the key blocks inside the causal (and window) range are visited.
//
// Decode: split-KV. Each CTA takes one (sequence, kv head, key chunk), scores
// all query heads of its group against the chunk with 16-byte loads, and
// writes an unnormalised partial (max, sum, output); a combine kernel merges
// the partials in split order, so the result does not depend on scheduling.
#include <algorithm>
#include <mutex>

#include "fk_common.cuh"
#include "fk_ops.h"

namespace fk {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

FK_DEVICE void cp_async16(void* smem_dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
FK_DEVICE void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
FK_DEVICE void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

FK_DEVICE void ldsm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
FK_DEVICE void ldsm_x4_t(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
FK_DEVICE void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// element (r, c) of a [rows][COLS] bf16 tile, 16-byte chunks XOR-swizzled by row
template <int COLS>
FK_DEVICE int swz(int r, int c) {
  return r * COLS + ((((c >> 3) ^ (r & 7))) << 3) + (c & 7);
}

constexpr int BQ = 64, BKV = 64;

template <int HD>
__global__ void __launch_bounds__(128) attn_prefill_kernel(const __nv_bfloat16* __restrict__ q, int ldq,
                                                           const __nv_bfloat16* __restrict__ kc,
                                                           const __nv_bfloat16* __restrict__ vc, int cap, int S,
                                                           int pos0, int Hq, int Hkv, int window, float scale_log2,
                                                           __nv_bfloat16* __restrict__ o) {
  extern __shared__ uint4 smem_u4[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem_u4);
  __nv_bfloat16* sK = sQ + BQ * HD;
  __nv_bfloat16* sV = sK + 2 * BKV * HD;
  const int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (Hq / Hkv);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kv_len = pos0 + S;
  const int q_lo = qb * BQ;
  const int q_hi = min(S, q_lo + BQ) - 1;
  const int qp_lo = pos0 + q_lo, qp_hi = pos0 + q_hi;
  const int k_lo = window > 0 ? max(0, qp_lo - window + 1) : 0;
  const int kb_lo = k_lo / BKV, kb_hi = qp_hi / BKV;
  const size_t head_off = ((size_t)b * Hkv + g) * cap * HD;
  const __nv_bfloat16* kbase = kc + head_off;
  const __nv_bfloat16* vbase = vc + head_off;  // V^T: [HD][cap]
  constexpr int CPR = HD / 8;  // 16-byte chunks per K row
  constexpr int CPV = BKV / 8;  // 16-byte chunks per V^T row of a tile

  for (int i = tid; i < BQ * CPR; i += 128) {
    const int r = i / CPR, cc = i % CPR;
    const int qi = q_lo + r;
    const __nv_bfloat16* src = q + (size_t)(b * S + min(qi, S - 1)) * ldq + (size_t)h * HD + cc * 8;
    cp_async16(sQ + swz<HD>(r, cc * 8), src, qi < S ? 16 : 0);
  }
  auto load_kv = [&](int kb, int buf) {
    __nv_bfloat16* dk = sK + buf * BKV * HD;
    __nv_bfloat16* dv = sV + buf * BKV * HD;
    for (int i = tid; i < BKV * CPR; i += 128) {
      const int r = i / CPR, cc = i % CPR;
      const int kp = kb * BKV + r;
      const int ok = kp < kv_len ? 16 : 0;
      cp_async16(dk + swz<HD>(r, cc * 8), kbase + (size_t)min(kp, kv_len - 1) * HD + cc * 8, ok);
    }
    // V^T rows: keys [kb*BKV, kb*BKV + BKV) are inside the cache (cap is a
    // multiple of 64); keys past kv_len hold finite values and get p = 0
    for (int i = tid; i < HD * CPV; i += 128) {
      const int d = i / CPV, cc = i % CPV;
      cp_async16(dv + swz<BKV>(d, cc * 8), vbase + (size_t)d * cap + kb * BKV + cc * 8, 16);
    }
  };
  load_kv(kb_lo, 0);
  cp_async_commit();

  float oacc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int qr0 = qp_lo + warp * 16 + (lane >> 2);  // positions of this thread's two rows
  const int qr1 = qr0 + 8;
  const int mat = lane >> 3, mr = lane & 7;

  for (int kb = kb_lo; kb <= kb_hi; ++kb) {
    const int buf = (kb - kb_lo) & 1;
    if (kb < kb_hi) {
      load_kv(kb + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const __nv_bfloat16* tK = sK + buf * BKV * HD;
    const __nv_bfloat16* tV = sV + buf * BKV * HD;

    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < HD; k0 += 16) {
      uint32_t a[4];
      ldsm_x4(a, sQ + swz<HD>(warp * 16 + mr + (mat & 1) * 8, k0 + (mat >> 1) * 8));
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bb[4];
        ldsm_x4(bb, tK + swz<HD>(np * 16 + mr + (mat >> 1) * 8, k0 + (mat & 1) * 8));
        mma_bf16_16816(s[2 * np], a, bb[0], bb[1]);
        mma_bf16_16816(s[2 * np + 1], a, bb[2], bb[3]);
      }
    }
    // mask (causal, window, cache end) and move to the exp2 domain
    const int key0 = kb * BKV + 2 * (lane & 3);
    const bool edge = (kb * BKV + BKV - 1 > qp_lo + warp * 16) || (kb * BKV + BKV > kv_len) ||
                      (window > 0 && qp_hi - kb * BKV >= window);
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = s[nt][e] * scale_log2;
        if (edge) {
          const int key = key0 + nt * 8 + (e & 1);
          const int qp = e < 2 ? qr0 : qr1;
          const bool ok = key <= qp && key < kv_len && (window == 0 || qp - key < window);
          v = ok ? v : -INFINITY;
        }
        s[nt][e] = v;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0;
    const float base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float corr0 = exp2f(m0 - base0), corr1 = exp2f(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - base0);
      s[nt][1] = exp2f(s[nt][1] - base0);
      s[nt][2] = exp2f(s[nt][2] - base1);
      s[nt][3] = exp2f(s[nt][3] - base1);
      rs0 += s[nt][0] + s[nt][1];
      rs1 += s[nt][2] + s[nt][3];
    }
    l0 = l0 * corr0 + rs0;
    l1 = l1 * corr1 + rs1;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      oacc[i][0] *= corr0;
      oacc[i][1] *= corr0;
      oacc[i][2] *= corr1;
      oacc[i][3] *= corr1;
    }
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t a[4];
      a[0] = pack_bf16x2(s[2 * ks][0], s[2 * ks][1]);
      a[1] = pack_bf16x2(s[2 * ks][2], s[2 * ks][3]);
      a[2] = pack_bf16x2(s[2 * ks + 1][0], s[2 * ks + 1][1]);
      a[3] = pack_bf16x2(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
      for (int dp = 0; dp < HD / 16; ++dp) {
        uint32_t bb[4];
        ldsm_x4(bb, tV + swz<BKV>(dp * 16 + mr + (mat >> 1) * 8, ks * 16 + (mat & 1) * 8));
        mma_bf16_16816(oacc[2 * dp], a, bb[0], bb[1]);
        mma_bf16_16816(oacc[2 * dp + 1], a, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int qi0 = q_lo + warp * 16 + (lane >> 2), qi1 = qi0 + 8;
  const size_t ldo = (size_t)Hq * HD;
#pragma unroll
  for (int dt = 0; dt < HD / 8; ++dt) {
    const int col = h * HD + dt * 8 + 2 * (lane & 3);
    if (qi0 < S)
      *reinterpret_cast<uint32_t*>(o + (size_t)(b * S + qi0) * ldo + col) =
          pack_bf16x2(oacc[dt][0] * inv0, oacc[dt][1] * inv0);
    if (qi1 < S)
      *reinterpret_cast<uint32_t*>(o + (size_t)(b * S + qi1) * ldo + col) =
          pack_bf16x2(oacc[dt][2] * inv1, oacc[dt][3] * inv1);
  }
}

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------
// One CTA per (key chunk, kv head, sequence). The query heads of the GQA group
// (<= 8) form the 16 MMA rows (rows >= group are zero); each of the 4 warps
// takes 16 keys of every 64-key tile, keeps its own online-softmax state, and
// the warps are merged in shared memory at the end. K/V tiles stream through
// an NST-deep cp.async ring, so each CTA keeps NST-1 tiles in flight.
constexpr int kDecThreads = 128;
constexpr int kMaxGroup = 8;
constexpr int kDecTile = 64;

template <int HD>
struct DecCfg {
  static constexpr int NST = HD == 256 ? 3 : (HD == 128 ? 3 : 4);
  static constexpr int TILE_ELEMS = kDecTile * HD;
  static constexpr int SMEM = (16 * HD + NST * 2 * TILE_ELEMS) * 2;
};

template <int HD>
__global__ void __launch_bounds__(kDecThreads) attn_decode_kernel(
    const __nv_bfloat16* __restrict__ q, int ldq, const __nv_bfloat16* __restrict__ kc,
    const __nv_bfloat16* __restrict__ vc, int cap, int ctx_host, const int* d_ctx, int Hq, int Hkv, int window,
    float scale_log2, int chunk, int n_splits, float* __restrict__ part_o, float* __restrict__ part_ml) {
  pdl_trigger();
  pdl_wait();
  using C = DecCfg<HD>;
  extern __shared__ uint4 smem_u4[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem_u4);
  __nv_bfloat16* sKV = sQ + 16 * HD;  // [NST][K tile, V tile]
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int group = Hq / Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ctx = d_ctx ? *d_ctx + 1 : ctx_host;  // *d_ctx: tokens before the new one
  const int qpos = ctx - 1;
  int lo = split * chunk;
  const int hi = min(ctx, lo + chunk);
  if (window > 0) lo = max(lo, qpos - window + 1);
  // tiles start on a 64-key boundary (16-byte aligned V^T rows); keys outside
  // [lo, hi) inside a tile are masked
  const int t0 = lo & ~(kDecTile - 1);
  const int ntiles = hi > lo ? (hi - t0 + kDecTile - 1) / kDecTile : 0;
  const size_t head_off = ((size_t)b * Hkv + g) * cap * HD;
  const __nv_bfloat16* kbase = kc + head_off;
  const __nv_bfloat16* vbase = vc + head_off;  // V^T: [HD][cap]
  constexpr int CPR = HD / 8;
  constexpr int CPV = kDecTile / 8;

  for (int i = tid; i < 16 * CPR; i += kDecThreads) {
    const int r = i / CPR, cc = i % CPR;
    const __nv_bfloat16* src = q + (size_t)b * ldq + (size_t)(g * group + min(r, group - 1)) * HD + cc * 8;
    cp_async16(sQ + swz<HD>(r, cc * 8), src, r < group ? 16 : 0);
  }
  auto load_tile = [&](int t, int buf) {
    __nv_bfloat16* dk = sKV + (size_t)buf * 2 * C::TILE_ELEMS;
    __nv_bfloat16* dv = dk + C::TILE_ELEMS;
    for (int i = tid; i < kDecTile * CPR; i += kDecThreads) {
      const int r = i / CPR, cc = i % CPR;
      const int kp = t0 + t * kDecTile + r;
      const int ok = (kp >= lo && kp < hi) ? 16 : 0;
      cp_async16(dk + swz<HD>(r, cc * 8), kbase + (size_t)min(max(kp, lo), hi - 1) * HD + cc * 8, ok);
    }
    for (int i = tid; i < HD * CPV; i += kDecThreads) {
      const int d = i / CPV, cc = i % CPV;
      cp_async16(dv + swz<kDecTile>(d, cc * 8), vbase + (size_t)d * cap + t0 + t * kDecTile + cc * 8, 16);
    }
  };
  cp_async_commit();  // Q
#pragma unroll
  for (int t = 0; t < C::NST - 1; ++t) {
    if (t < ntiles) load_tile(t, t);
    cp_async_commit();
  }

  float oacc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int mat = lane >> 3, mr = lane & 7;

  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<C::NST - 2>();
    __syncthreads();
    {
      const int tn = t + C::NST - 1;
      if (tn < ntiles) load_tile(tn, tn % C::NST);
      cp_async_commit();
    }
    const __nv_bfloat16* tK = sKV + (size_t)(t % C::NST) * 2 * C::TILE_ELEMS;
    const __nv_bfloat16* tV = tK + C::TILE_ELEMS;
    const int kr = warp * 16;  // this warp's 16 keys of the tile
    float s[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < HD; k0 += 16) {
      uint32_t a[4], bb[4];
      ldsm_x4(a, sQ + swz<HD>(mr + (mat & 1) * 8, k0 + (mat >> 1) * 8));
      ldsm_x4(bb, tK + swz<HD>(kr + mr + (mat >> 1) * 8, k0 + (mat & 1) * 8));
      mma_bf16_16816(s[0], a, bb[0], bb[1]);
      mma_bf16_16816(s[1], a, bb[2], bb[3]);
    }
    const int key0 = t0 + t * kDecTile + kr + 2 * (lane & 3);
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key0 + nt * 8 + (e & 1);
        const bool ok = key >= lo && key < hi;
        s[nt][e] = ok ? s[nt][e] * scale_log2 : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0;
    const float base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float corr0 = exp2f(m0 - base0), corr1 = exp2f(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] = exp2f(s[nt][0] - base0);
      s[nt][1] = exp2f(s[nt][1] - base0);
      s[nt][2] = exp2f(s[nt][2] - base1);
      s[nt][3] = exp2f(s[nt][3] - base1);
      rs0 += s[nt][0] + s[nt][1];
      rs1 += s[nt][2] + s[nt][3];
    }
    l0 = l0 * corr0 + rs0;
    l1 = l1 * corr1 + rs1;
    uint32_t a[4];
    a[0] = pack_bf16x2(s[0][0], s[0][1]);
    a[1] = pack_bf16x2(s[0][2], s[0][3]);
    a[2] = pack_bf16x2(s[1][0], s[1][1]);
    a[3] = pack_bf16x2(s[1][2], s[1][3]);
#pragma unroll
    for (int dp = 0; dp < HD / 16; ++dp) {
      oacc[2 * dp][0] *= corr0;
      oacc[2 * dp][1] *= corr0;
      oacc[2 * dp][2] *= corr1;
      oacc[2 * dp][3] *= corr1;
      oacc[2 * dp + 1][0] *= corr0;
      oacc[2 * dp + 1][1] *= corr0;
      oacc[2 * dp + 1][2] *= corr1;
      oacc[2 * dp + 1][3] *= corr1;
      uint32_t bb[4];
      ldsm_x4(bb, tV + swz<kDecTile>(dp * 16 + mr + (mat >> 1) * 8, kr + (mat & 1) * 8));
      mma_bf16_16816(oacc[2 * dp], a, bb[0], bb[1]);
      mma_bf16_16816(oacc[2 * dp + 1], a, bb[2], bb[3]);
    }
  }
  cp_async_wait<0>();
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  __syncthreads();  // the K/V ring is free: reuse it for the cross-warp merge
  float* sO = reinterpret_cast<float*>(sKV);  // [4 warps][16 rows][HD]
  float* sM = sO + 4 * 16 * HD;               // [4][16]
  float* sL = sM + 64;
  const int r0 = lane >> 2, r1 = r0 + 8;
#pragma unroll
  for (int dt = 0; dt < HD / 8; ++dt) {
    const int col = dt * 8 + 2 * (lane & 3);
    sO[(warp * 16 + r0) * HD + col] = oacc[dt][0];
    sO[(warp * 16 + r0) * HD + col + 1] = oacc[dt][1];
    sO[(warp * 16 + r1) * HD + col] = oacc[dt][2];
    sO[(warp * 16 + r1) * HD + col + 1] = oacc[dt][3];
  }
  if ((lane & 3) == 0) {
    sM[warp * 16 + r0] = m0;
    sM[warp * 16 + r1] = m1;
    sL[warp * 16 + r0] = l0;
    sL[warp * 16 + r1] = l1;
  }
  __syncthreads();
  for (int i = tid; i < group * HD; i += kDecThreads) {
    const int r = i / HD, d = i % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, sM[w * 16 + r]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = sM[w * 16 + r];
        if (mw != -INFINITY) {
          const float f = exp2f(mw - M);
          L += sL[w * 16 + r] * f;
          acc += sO[(w * 16 + r) * HD + d] * f;
        }
      }
    }
    const int h = g * group + r;
    const size_t base = ((size_t)b * Hq + h) * n_splits + split;
    part_o[base * HD + d] = acc;
    if (d == 0) {
      part_ml[base * 2] = M;
      part_ml[base * 2 + 1] = L;
    }
  }
}

template <int HD>
__global__ void attn_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml, int Hq,
                                    int n_splits, __nv_bfloat16* __restrict__ o) {
  pdl_trigger();
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y;
  const size_t base = ((size_t)b * Hq + h) * n_splits;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, part_ml[(base + s) * 2]);
  float L = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    const float m = part_ml[(base + s) * 2];
    if (m != -INFINITY) L += part_ml[(base + s) * 2 + 1] * exp2f(m - M);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  for (int d = threadIdx.x; d < HD; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < n_splits; ++s) {
      const float m = part_ml[(base + s) * 2];
      if (m != -INFINITY) acc += part_o[(base + s) * HD + d] * exp2f(m - M);
    }
    o[((size_t)b * Hq + h) * HD + d] = __float2bfloat16_rn(acc * inv);
  }
}

template <int HD>
cudaError_t prefill_hd(const void* q, int ldq, const void* kc, const void* vc, int cap, int B, int S, int pos0, int Hq,
                       int Hkv, int window, float scale, void* o, cudaStream_t st) {
  constexpr int smem = (BQ + 4 * BKV) * HD * 2;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(attn_prefill_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (err != cudaSuccess) return err;
  dim3 grid((S + BQ - 1) / BQ, Hq, B);
  attn_prefill_kernel<HD><<<grid, 128, smem, st>>>(
      static_cast<const __nv_bfloat16*>(q), ldq, static_cast<const __nv_bfloat16*>(kc),
      static_cast<const __nv_bfloat16*>(vc), cap, S, pos0, Hq, Hkv, window, scale * kLog2e,
      static_cast<__nv_bfloat16*>(o));
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_prefill(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B,
                                     int S, int pos0, int Hq, int Hkv, int hd, int window, float scale, void* o,
                                     cudaStream_t st) {
  if (B == 0 || S == 0) return cudaSuccess;
  switch (hd) {
    case 64: return prefill_hd<64>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, st);
    case 128: return prefill_hd<128>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, st);
    case 256: return prefill_hd<256>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, st);
  }
  return cudaErrorInvalidValue;
}

size_t decode_attention_scratch_bytes(int B, int Hq, int hd, int max_splits) {
  return (size_t)B * Hq * max_splits * (hd + 2) * sizeof(float) + 256;
}

int decode_attention_splits(int B, int Hkv, int max_ctx, int sm_count, int* chunk) {
  const long target = 4L * sm_count;
  long c = ((long)max_ctx * B * Hkv + target - 1) / target;
  c = (c + kDecTile - 1) / kDecTile * kDecTile;
  c = std::max((long)kDecTile, c);
  *chunk = (int)c;
  return (int)((max_ctx + c - 1) / c);
}

template <int HD>
cudaError_t decode_hd(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B, int ctx,
                      const int* d_ctx, int Hq, int Hkv, int window, float sl, int chunk, int n_splits, float* part_o,
                      float* part_ml, void* o, cudaStream_t st) {
  using C = DecCfg<HD>;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(attn_decode_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (err != cudaSuccess) return err;
  dim3 grid(n_splits, Hkv, B);
  cudaError_t e = fk_launch(attn_decode_kernel<HD>, grid, kDecThreads, C::SMEM, st, static_cast<const __nv_bfloat16*>(q),
                            ldq, static_cast<const __nv_bfloat16*>(kcache), static_cast<const __nv_bfloat16*>(vcache),
                            cap, ctx, d_ctx, Hq, Hkv, window, sl, chunk, n_splits, part_o, part_ml);
  if (e != cudaSuccess) return e;
  return fk_launch(attn_combine_kernel<HD>, dim3(Hq, B), HD < 128 ? HD : 128, 0, st, (const float*)part_o,
                   (const float*)part_ml, Hq, n_splits, static_cast<__nv_bfloat16*>(o));
}

cudaError_t launch_attention_decode(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B,
                                    int ctx, const int* d_ctx, int Hq, int Hkv, int hd, int window, float scale,
                                    int chunk, int n_splits, void* scratch, void* o, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  if (Hq / Hkv > kMaxGroup || chunk % kDecTile) return cudaErrorInvalidValue;
  float* part_o = static_cast<float*>(scratch);
  float* part_ml = part_o + (size_t)B * Hq * n_splits * hd;
  const float sl = scale * kLog2e;
  switch (hd) {
    case 64: return decode_hd<64>(q, ldq, kcache, vcache, cap, B, ctx, d_ctx, Hq, Hkv, window, sl, chunk, n_splits, part_o, part_ml, o, st);
    case 128: return decode_hd<128>(q, ldq, kcache, vcache, cap, B, ctx, d_ctx, Hq, Hkv, window, sl, chunk, n_splits, part_o, part_ml, o, st);
    case 256: return decode_hd<256>(q, ldq, kcache, vcache, cap, B, ctx, d_ctx, Hq, Hkv, window, sl, chunk, n_splits, part_o, part_ml, o, st);
  }
  return cudaErrorInvalidValue;
}
}  // namespace fk

// ---------------------------------------------------------------------------
// op-level entry point: one decode-attention step over a caller's KV cache
// ---------------------------------------------------------------------------
#include "fk_internal.h"

namespace {
fk_status check_decode_args(const void* q, const void* kc, const void* vc, int B, int Hq, int Hkv, int hd, int cap,
                            int ctx, int window, const void* out) {
  using fk::fail;
  if (!q || !kc || !vc || !out) return fail(FK_ERR_INVALID_ARG, "attention decode: null pointer");
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Hq / Hkv > 8)
    return fail(FK_ERR_INVALID_ARG, "attention decode: need batch >= 1 and 1..8 query heads per kv head");
  if (hd != 64 && hd != 128 && hd != 256) return fail(FK_ERR_INVALID_ARG, "attention decode: head_dim 64/128/256");
  if (ctx < 1 || ctx > cap || window < 0 || cap % 64)
    return fail(FK_ERR_INVALID_ARG, "attention decode: need 1 <= ctx <= cap, cap a multiple of 64");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kc) | reinterpret_cast<uintptr_t>(vc)) & 15)
    return fail(FK_ERR_INVALID_ARG, "attention decode: q and caches must be 16-byte aligned");
  return FK_OK;
}
}  // namespace

namespace fk {
// shared by the scratch-taking and the allocation-free entry points
fk_status attention_decode_plan(int B, int Hq, int Hkv, int hd, int ctx, int* chunk, int* splits, size_t* bytes) {
  int sms = 0;
  fk_status s = check_device(&sms);
  if (s != FK_OK) return s;
  *splits = decode_attention_splits(B, Hkv, ctx, sms, chunk);
  *bytes = decode_attention_scratch_bytes(B, Hq, hd, *splits);
  return FK_OK;
}
fk_status attention_decode_run(const void* q, const void* kc, const void* vc, int B, int Hq, int Hkv, int hd, int cap,
                               int ctx, int window, int chunk, int splits, void* scratch, void* out,
                               cudaStream_t st) {
  cudaError_t e = launch_attention_decode(q, Hq * hd, kc, vc, cap, B, ctx, nullptr, Hq, Hkv, hd, window,
                                          1.0f / sqrtf((float)hd), chunk, splits, scratch, out, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention decode launch");
  return FK_OK;
}
}  // namespace fk

extern "C" size_t fk_attention_decode_scratch_bytes(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads,
                                                    int32_t head_dim, int32_t ctx) {
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || ctx < 1) return 0;
  int chunk = 0, splits = 0;
  size_t bytes = 0;
  if (fk::attention_decode_plan(batch, n_q_heads, n_kv_heads, head_dim, ctx, &chunk, &splits, &bytes) != FK_OK)
    return 0;
  return bytes;
}

extern "C" fk_status fk_attention_decode(const void* d_q, const void* d_kcache, const void* d_vcache, int32_t batch,
                                         int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t cap,
                                         int32_t ctx, int32_t window, void* d_scratch, size_t scratch_bytes,
                                         void* d_out, void* stream) {
  fk_status s = check_decode_args(d_q, d_kcache, d_vcache, batch, n_q_heads, n_kv_heads, head_dim, cap, ctx, window,
                                  d_out);
  if (s != FK_OK) return s;
  int chunk = 0, splits = 0;
  size_t need = 0;
  s = fk::attention_decode_plan(batch, n_q_heads, n_kv_heads, head_dim, ctx, &chunk, &splits, &need);
  if (s != FK_OK) return s;
  if (!d_scratch || scratch_bytes < need) return fk::fail(FK_ERR_WORKSPACE, "attention decode: scratch too small");
  if (reinterpret_cast<uintptr_t>(d_scratch) & 15) return fk::fail(FK_ERR_INVALID_ARG, "scratch must be 16-byte aligned");
  return fk::attention_decode_run(d_q, d_kcache, d_vcache, batch, n_q_heads, n_kv_heads, head_dim, cap, ctx, window,
                                  chunk, splits, d_scratch, d_out, static_cast<cudaStream_t>(stream));
}
