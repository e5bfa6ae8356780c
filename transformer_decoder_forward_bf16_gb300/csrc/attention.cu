// Causal GQA attention over the bf16 KV cache ("N7 · model/forward-parity",
// Thm 1: causal multi-head/GQA attention; Thm 2 and "pegainfer #878":
// sliding-window local layers).
//
// Prefill (used where the tcgen05 kernel of attention_tc.cu does not apply:
// row strides or caches without the 16-byte / 64-position alignment its TMA
// tiles need): flash-style, one CTA per (64 queries, head, sequence), 4 warps
// x 16 query rows, 64-key blocks double-buffered in shared memory with
// cp.async, QKᵀ and PV on mma.sync m16n8k16 (bf16, fp32 accumulate), online
// softmax in fp32 (exp2 domain), P rounded to bf16 for the PV product. Only
// the key blocks inside the causal (and window) range are visited.
//
// Decode: split-KV over a thread-block cluster. The CTAs of one cluster share
// one (sequence, kv head) and split its key range into equal runs of 64-key
// tiles streamed by TMA; each scores all query heads of the GQA group against
// its tiles and keeps an unnormalised partial (max, sum, output) in its
// shared memory. After a cluster barrier the CTAs merge the partials through
// distributed shared memory, each CTA finishing a slice of the outputs and
// adding the partials in rank order, so the result does not depend on
// scheduling and no partial result leaves the chip.
#include <algorithm>
#include <mutex>

#include "fk_common.cuh"
#include "fk_internal.h"
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
// One CTA per (key split, kv head, sequence); the splits of a (sequence, kv
// head) form one cluster of `gridDim.x` CTAs. Warp 4 streams the CTA's 64-key
// K and V^T tiles into an NST-deep shared-memory ring with TMA (mbarrier
// completion; with fused RoPE it starts before the previous kernel has
// finished, since it reads only earlier cache positions). Warps 0-3 consume
// the ring: the query heads of the GQA group (<= 8) form the 16 MMA rows
// (rows >= group are zero), each warp takes 16 keys of every tile, keeps its
// own online-softmax state and releases the slot when done, so loads and
// math overlap with no CTA-wide barrier per tile. The four warps are merged
// in shared memory at the end.
constexpr int kDecConsumers = 128;
constexpr int kDecThreads = kDecConsumers + 32;
constexpr int kMaxGroup = 8;
constexpr int kDecTile = 64;
constexpr int kMaxCluster = 16;

template <int HD>
struct DecCfg {
  static constexpr int NST = HD == 64 ? 4 : (HD == 128 ? 3 : 2);
  static constexpr int TILE_ELEMS = kDecTile * HD;          // K tile = V^T tile elements
  static constexpr int STAGE_BYTES = 2 * TILE_ELEMS * 2;    // K + V^T
  static constexpr int Q_BYTES = 16 * HD * 2;
  static constexpr int RING_OFF = (Q_BYTES + 1023) / 1024 * 1024;
  static constexpr int BAR_OFF = RING_OFF + NST * STAGE_BYTES;
  static constexpr int SMEM = BAR_OFF + 128 + 1024;  // + barriers/flags, + base alignment slack
};

FK_DEVICE void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kDecConsumers) : "memory"); }
FK_DEVICE void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// element (r, c) of a K tile [64 keys][HD] stored as HD/64 TMA boxes of
// [64][64] with the 128-byte swizzle
template <int HD>
FK_DEVICE int kswz(int r, int c) {
  return (c >> 6) * (kDecTile * 64) + r * 64 + ((((c >> 3) & 7) ^ (r & 7)) << 3) + (c & 7);
}

// Arguments of the decode kernel. With fused RoPE (a session's decode step),
// q points at the token's qkv row [q heads | k heads | v heads] (ldq = the row
// stride): the kernel applies [QK-norm and] RoPE at position ctx-1, writes
// the new key and value into the caches and attends over them; otherwise q
// holds the query heads with RoPE applied and the caches are complete.
struct DecArgs {
  const __nv_bfloat16* q;
  int ldq;
  int cap, ctx_host;
  const int* d_ctx;  // non-null: ctx = *d_ctx + 1
  int Hq, Hkv, window;
  float scale_log2;
  __nv_bfloat16* o;
  unsigned* dev_err;  // optional device error word (pipeline timeouts)
  // fused RoPE
  const float2* rope;  // [positions][HD/2] (cos, sin) of frequency j
  int qk_norm;
  const __nv_bfloat16* q_norm;
  const __nv_bfloat16* k_norm;
  float eps;
  __nv_bfloat16* kc_w;  // the caches, written at position ctx-1
  __nv_bfloat16* vc_w;
};

// [QK-norm and] RoPE of one head held by a warp: lane owns elements
// e0..e0+C-1 of each half (pairs (j, j+HD/2)); cs: this lane's (cos, sin).
template <int HD>
FK_DEVICE void rope_head(const __nv_bfloat16* src, const DecArgs& a, const __nv_bfloat16* nw, const float2* cs,
                         int lane, float* olo, float* ohi) {
  constexpr int C = HD / 64, HALF = HD / 2;
  const int e0 = lane * C;
  float lo[C], hi[C];
#pragma unroll
  for (int i = 0; i < C; ++i) {
    lo[i] = __bfloat162float(src[e0 + i]);
    hi[i] = __bfloat162float(src[HALF + e0 + i]);
  }
  if (a.qk_norm) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < C; ++i) ss += lo[i] * lo[i] + hi[i] * hi[i];
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / HD + a.eps);
#pragma unroll
    for (int i = 0; i < C; ++i) {
      lo[i] = lo[i] * r * __bfloat162float(nw[e0 + i]);
      hi[i] = hi[i] * r * __bfloat162float(nw[HALF + e0 + i]);
    }
  }
#pragma unroll
  for (int i = 0; i < C; ++i) {
    olo[i] = lo[i] * cs[i].x - hi[i] * cs[i].y;
    ohi[i] = hi[i] * cs[i].x + lo[i] * cs[i].y;
  }
}

template <int HD, bool ROPE>
__global__ void __launch_bounds__(kDecThreads) attn_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV,
                                                                  const DecArgs a) {
  using C = DecCfg<HD>;
  constexpr int NC = HD / 64, HALF = HD / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  uint8_t* ring = smem + C::RING_OFF;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::NST);
  __shared__ __align__(16) __nv_bfloat16 sNew[2][HD];  // fused RoPE: the new key and value
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int n_splits = gridDim.x;  // = the cluster size: blockIdx.x is the rank
  const int Hq = a.Hq, Hkv = a.Hkv, cap = a.cap, window = a.window;
  const int group = Hq / Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecConsumers / 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_trigger();
  // Without fused RoPE everything below depends on the previous kernel. With
  // it, the cache positions before the new token and the length were written
  // by kernels that completed before the previous kernel (the QKV projection)
  // passed its own wait, which precedes its trigger: the K/V tiles are
  // requested first, and only the new token's q/k/v wait for the projection.
  if (!ROPE) pdl_wait();
  const int ctx = a.d_ctx ? *a.d_ctx + 1 : a.ctx_host;  // *d_ctx: tokens before the new one
  const int qpos = ctx - 1;
  // visible keys [lo, hi); tiles start on a 64-key boundary and the splits
  // take equal runs of tiles; keys outside [lo, hi) inside a tile are masked
  const int lo = window > 0 ? max(0, qpos - window + 1) : 0;
  const int hi = ctx;
  const int tfirst = lo / kDecTile, n_all = (hi + kDecTile - 1) / kDecTile - tfirst;
  const int ta = tfirst + (int)((long)split * n_all / n_splits);
  const int ntiles = tfirst + (int)((long)(split + 1) * n_all / n_splits) - ta;
  const int t0 = ta * kDecTile;
  const int t_new = ROPE ? qpos / kDecTile - ta : -1;  // this CTA's tile holding the new token, if any
  const int head_row = (b * Hkv + g);                  // (sequence, kv head) index

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float oacc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

  if (warp == kDecConsumers / 32) {
    // ---- producer: K tile = HD/64 boxes [64 keys][64], V^T tile = one box [HD][64 keys]
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int issued[C::NST];
#pragma unroll
      for (int s = 0; s < C::NST; ++s) issued[s] = 0;
      for (int t = 0; t < ntiles; ++t) {
        const int stage = t % C::NST;
        if (t >= C::NST && !mbar_wait(&empty[stage], ((t / C::NST) - 1) & 1, abort_flag, a.dev_err)) break;
        uint8_t* sk = ring + stage * C::STAGE_BYTES;
        uint8_t* sv = sk + C::TILE_ELEMS * 2;
        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
        const int pos = t0 + t * kDecTile;
#pragma unroll
        for (int c = 0; c < NC; ++c)
          tma_load_2d(&tmK, &full[stage], sk + c * kDecTile * 64 * 2, c * 64, head_row * cap + pos);
        tma_load_2d(&tmV, &full[stage], sv, pos, head_row * HD);
        ++issued[stage];
      }
      // leave only when every requested tile has landed
      for (int s = 0; s < C::NST; ++s) {
        if (!issued[s]) continue;
        const uint32_t fa = smem_u32(&full[s]);
        const uint64_t w0 = globaltimer_ns();
        while (!mbar_try_wait(fa, (issued[s] - 1) & 1) && globaltimer_ns() - w0 < kWaitLimitNs) {
        }
      }
    }
    __syncwarp();
  } else {
    // ---- consumers
    if (ROPE) {
      constexpr int CC = NC;
      float2 cs[CC];  // this lane's (cos, sin) at the new position: no dependence on the projection
#pragma unroll
      for (int i = 0; i < CC; ++i) cs[i] = a.rope[(size_t)qpos * HALF + lane * CC + i];
      pdl_wait();
      const __nv_bfloat16* row = a.q + (size_t)b * a.ldq;
      for (int r = warp; r < 16; r += kDecConsumers / 32) {
        float olo[NC], ohi[NC];
        if (r < group) {
          rope_head<HD>(row + (size_t)(g * group + r) * HD, a, a.q_norm, cs, lane, olo, ohi);
        } else {
#pragma unroll
          for (int i = 0; i < NC; ++i) olo[i] = ohi[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          sQ[swz<HD>(r, lane * NC + i)] = __float2bfloat16_rn(olo[i]);
          sQ[swz<HD>(r, HALF + lane * NC + i)] = __float2bfloat16_rn(ohi[i]);
        }
      }
      if (warp == 0) {
        float olo[NC], ohi[NC];
        rope_head<HD>(row + (size_t)(Hq + g) * HD, a, a.k_norm, cs, lane, olo, ohi);
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          sNew[0][lane * NC + i] = __float2bfloat16_rn(olo[i]);
          sNew[0][HALF + lane * NC + i] = __float2bfloat16_rn(ohi[i]);
        }
      } else if (warp == 1) {
        const __nv_bfloat16* vs = row + (size_t)(Hq + Hkv + g) * HD;
        for (int d = lane; d < HD; d += 32) sNew[1][d] = vs[d];
      }
      consumers_sync();
      if (t_new >= 0 && t_new < ntiles) {  // the one CTA whose tiles hold the new token stores it
        __nv_bfloat16* kw = a.kc_w + ((size_t)head_row * cap + qpos) * HD;
        __nv_bfloat16* vw = a.vc_w + (size_t)head_row * HD * cap + qpos;
        for (int d = tid; d < HD; d += kDecConsumers) {
          kw[d] = sNew[0][d];
          vw[(size_t)d * cap] = sNew[1][d];
        }
      }
    } else {
      constexpr int CPR = HD / 8;
      for (int i = tid; i < 16 * CPR; i += kDecConsumers) {
        const int r = i / CPR, cc = i % CPR;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < group) v = *reinterpret_cast<const uint4*>(a.q + (size_t)b * a.ldq + (size_t)(g * group + r) * HD + cc * 8);
        *reinterpret_cast<uint4*>(sQ + swz<HD>(r, cc * 8)) = v;
      }
      consumers_sync();
    }
    const float scale_log2 = a.scale_log2;
    const int mat = lane >> 3, mr = lane & 7;
    const int kr = warp * 16;  // this warp's 16 keys of every tile
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % C::NST;
      if (!mbar_wait(&full[stage], (t / C::NST) & 1, abort_flag, a.dev_err)) break;
      __nv_bfloat16* tK = reinterpret_cast<__nv_bfloat16*>(ring + stage * C::STAGE_BYTES);
      __nv_bfloat16* tV = tK + C::TILE_ELEMS;
      const bool patch = ROPE && t == t_new && (qpos - (t0 + t * kDecTile)) / 16 == warp;
      if (patch) {  // the cached copy of the new token is stale: this warp's key row
        const int r = qpos - (t0 + t * kDecTile);
        for (int d = lane; d < HD; d += 32) {
          tK[kswz<HD>(r, d)] = sNew[0][d];
          tV[swz<kDecTile>(d, r)] = sNew[1][d];
        }
        __syncwarp();
      }
      float s[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
      for (int k0 = 0; k0 < HD; k0 += 16) {
        uint32_t qa[4], bb[4];
        ldsm_x4(qa, sQ + swz<HD>(mr + (mat & 1) * 8, k0 + (mat >> 1) * 8));
        ldsm_x4(bb, tK + kswz<HD>(kr + mr + (mat >> 1) * 8, k0 + (mat & 1) * 8));
        mma_bf16_16816(s[0], qa, bb[0], bb[1]);
        mma_bf16_16816(s[1], qa, bb[2], bb[3]);
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
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[0][0], s[0][1]);
      pa[1] = pack_bf16x2(s[0][2], s[0][3]);
      pa[2] = pack_bf16x2(s[1][0], s[1][1]);
      pa[3] = pack_bf16x2(s[1][2], s[1][3]);
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
        mma_bf16_16816(oacc[2 * dp], pa, bb[0], bb[1]);
        mma_bf16_16816(oacc[2 * dp + 1], pa, bb[2], bb[3]);
      }
      if (patch) fence_proxy_async_smem();  // generic writes before the slot is refilled by TMA
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }
  __syncthreads();  // the ring is drained (the producer waited for its last tiles): reuse it
  float* sO = reinterpret_cast<float*>(ring);  // [4 warps][16 rows][HD]
  float* sM = sO + 4 * 16 * HD;                // [4][16]
  float* sL = sM + 64;
  float* sP = sL + 64;  // this CTA's partial per query head: [group][HD] (unnormalised), sPM, sPL
  float* sPM = sP + kMaxGroup * HD;
  float* sPL = sPM + kMaxGroup;
  if (warp < kDecConsumers / 32) {
    const int r0 = lane >> 2, r1 = r0 + 8;
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt) {
      const int col = dt * 8 + 2 * (lane & 3);
      if (r0 < group) {
        sO[(warp * 16 + r0) * HD + col] = oacc[dt][0];
        sO[(warp * 16 + r0) * HD + col + 1] = oacc[dt][1];
      }
      if (r1 < group) {
        sO[(warp * 16 + r1) * HD + col] = oacc[dt][2];
        sO[(warp * 16 + r1) * HD + col + 1] = oacc[dt][3];
      }
    }
    if ((lane & 3) == 0) {
      sM[warp * 16 + r0] = m0;
      sM[warp * 16 + r1] = m1;
      sL[warp * 16 + r0] = l0;
      sL[warp * 16 + r1] = l1;
    }
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
    sP[r * HD + d] = acc;
    if (d == 0) {
      sPM[r] = M;
      sPL[r] = L;
    }
  }
  cluster_sync();  // every split's partial is in its shared memory
  // CTA `split` finishes outputs [split*per, (split+1)*per) of the group's
  // group*HD values, reading the n_splits partials in rank order
  const int total = group * HD;
  const int per = (total + n_splits - 1) / n_splits;
  const int i_end = min(total, (split + 1) * per);
  for (int i = split * per + tid; i < i_end; i += kDecThreads) {
    const int r = i / HD;
    float m[kMaxCluster], v[kMaxCluster], l[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      m[c] = -INFINITY;
      v[c] = l[c] = 0.f;
      if (c < n_splits) {
        m[c] = dsmem_ld(dsmem_addr(sPM + r, c));
        l[c] = dsmem_ld(dsmem_addr(sPL + r, c));
        v[c] = dsmem_ld(dsmem_addr(sP + i, c));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) M = fmaxf(M, m[c]);
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (m[c] != -INFINITY) {
        const float f = exp2f(m[c] - M);
        L += l[c] * f;
        acc += v[c] * f;
      }
    }
    a.o[((size_t)b * Hq + g * group + r) * HD + (i - r * HD)] = __float2bfloat16_rn(L > 0.f ? acc / L : 0.f);
  }
  cluster_sync();  // no CTA leaves while another may still read its partial
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

// Largest cluster of decode CTAs the GPU co-schedules for this head_dim
// (a cluster of 16 is beyond the portable size and is allowed explicitly).
template <int HD, bool ROPE>
cudaError_t decode_attrs() {
  using C = DecCfg<HD>;
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<HD, ROPE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<HD, ROPE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <int HD>
int decode_max_cluster(cudaError_t* err) {
  using C = DecCfg<HD>;
  static std::once_flag once;
  static cudaError_t e0 = cudaSuccess;
  static int n = 1;
  std::call_once(once, [] {
    e0 = decode_attrs<HD, false>();
    if (e0 == cudaSuccess) e0 = decode_attrs<HD, true>();
    if (e0 != cudaSuccess) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kMaxCluster, 1, 1);
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    int c = 0, c2 = 0;
    if (cudaOccupancyMaxPotentialClusterSize(&c, attn_decode_kernel<HD, false>, &cfg) != cudaSuccess ||
        cudaOccupancyMaxPotentialClusterSize(&c2, attn_decode_kernel<HD, true>, &cfg) != cudaSuccess || c < 1 ||
        c2 < 1) {
      cudaGetLastError();
      c = c2 = 8;  // the portable size
    }
    n = std::min(std::min(c, c2), kMaxCluster);
  });
  *err = e0;
  return n;
}

template <int HD>
int decode_resident_per_sm() {
  int dev = 0, smem_sm = 0, reserved = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  return std::max(1, smem_sm / (DecCfg<HD>::SMEM + 2 * HD * 2 + reserved));
}

// Splits per (sequence, kv head): the largest power of two that keeps the
// grid within one wave of resident CTAs (the CTAs of a split then stream
// their keys side by side), at most the co-schedulable cluster size and the
// number of 64-key tiles.
int decode_attention_splits(int B, int Hkv, int hd, int max_ctx, int sm_count) {
  cudaError_t e = cudaSuccess;
  int maxc = 1, res = 1;
  switch (hd) {
    case 64: maxc = decode_max_cluster<64>(&e); res = decode_resident_per_sm<64>(); break;
    case 128: maxc = decode_max_cluster<128>(&e); res = decode_resident_per_sm<128>(); break;
    case 256: maxc = decode_max_cluster<256>(&e); res = decode_resident_per_sm<256>(); break;
    default: return 1;
  }
  if (e != cudaSuccess) return 1;
  const long want = std::max(1L, (long)res * sm_count / ((long)B * Hkv));
  const long lim = std::min<long>({(long)maxc, want, (max_ctx + kDecTile - 1L) / kDecTile});
  int cs = 1;
  while (cs * 2 <= lim) cs *= 2;
  return cs;
}

template <int HD>
cudaError_t decode_hd(const void* kcache, const void* vcache, const DecArgs& a, bool rope, int B, int n_splits,
                      cudaStream_t st) {
  using C = DecCfg<HD>;
  cudaError_t err = cudaSuccess;
  const int maxc = decode_max_cluster<HD>(&err);
  if (err != cudaSuccess) return err;
  if (n_splits < 1 || n_splits > maxc) return cudaErrorInvalidValue;
  CUtensorMap tK, tV;
  if (make_tmap_bf16(&tK, kcache, (int64_t)B * a.Hkv * a.cap, HD, HD, kDecTile) != FK_OK ||
      make_tmap_bf16(&tV, vcache, (int64_t)B * a.Hkv * HD, a.cap, a.cap, HD) != FK_OK)
    return cudaErrorInvalidValue;
  const dim3 grid(n_splits, a.Hkv, B);
  if (rope)
    return fk_launch_cluster(attn_decode_kernel<HD, true>, grid, kDecThreads, C::SMEM, st, n_splits, tK, tV, a);
  return fk_launch_cluster(attn_decode_kernel<HD, false>, grid, kDecThreads, C::SMEM, st, n_splits, tK, tV, a);
}

cudaError_t decode_dispatch(const void* kcache, const void* vcache, const DecArgs& a, bool rope, int hd, int B,
                            int n_splits, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  if (a.Hq / a.Hkv > kMaxGroup || a.cap % kDecTile) return cudaErrorInvalidValue;
  switch (hd) {
    case 64: return decode_hd<64>(kcache, vcache, a, rope, B, n_splits, st);
    case 128: return decode_hd<128>(kcache, vcache, a, rope, B, n_splits, st);
    case 256: return decode_hd<256>(kcache, vcache, a, rope, B, n_splits, st);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention_decode(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B,
                                    int ctx, const int* d_ctx, int Hq, int Hkv, int hd, int window, float scale,
                                    int n_splits, void* o, cudaStream_t st) {
  DecArgs a = {};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.ldq = ldq;
  a.cap = cap;
  a.ctx_host = ctx;
  a.d_ctx = d_ctx;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.window = window;
  a.scale_log2 = scale * kLog2e;
  a.o = static_cast<__nv_bfloat16*>(o);
  return decode_dispatch(kcache, vcache, a, false, hd, B, n_splits, st);
}

cudaError_t launch_attention_decode_rope(const void* qkv, int ldqkv, void* kcache, void* vcache, int cap, int B,
                                         const int* d_ctx, int Hq, int Hkv, int hd, int window, float scale,
                                         const float2* rope, int qk_norm, const void* q_norm, const void* k_norm,
                                         float eps, int n_splits, void* o, unsigned* dev_err, cudaStream_t st) {
  if (!d_ctx) return cudaErrorInvalidValue;
  DecArgs a = {};
  a.q = static_cast<const __nv_bfloat16*>(qkv);
  a.ldq = ldqkv;
  a.kc_w = static_cast<__nv_bfloat16*>(kcache);
  a.vc_w = static_cast<__nv_bfloat16*>(vcache);
  a.cap = cap;
  a.d_ctx = d_ctx;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.window = window;
  a.scale_log2 = scale * kLog2e;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.dev_err = dev_err;
  a.rope = rope;
  a.qk_norm = qk_norm;
  a.q_norm = static_cast<const __nv_bfloat16*>(q_norm);
  a.k_norm = static_cast<const __nv_bfloat16*>(k_norm);
  a.eps = eps;
  return decode_dispatch(kcache, vcache, a, true, hd, B, n_splits, st);
}
}  // namespace fk

// ---------------------------------------------------------------------------
// op-level entry point: one decode-attention step over a caller's KV cache
// ---------------------------------------------------------------------------

namespace {
// The scratch of fk_attention_decode is kept in the interface (a later kernel
// may use it) but the cluster kernel writes nothing there.
constexpr size_t kDecodeScratchBytes = 256;

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
// shared by the scratch-taking and the allocation-free entry points: the
// kernel keeps its split partials on chip, so neither needs device memory
fk_status attention_decode_plan(int B, int Hkv, int hd, int ctx, int* splits) {
  int sms = 0;
  fk_status s = check_device(&sms);
  if (s != FK_OK) return s;
  *splits = decode_attention_splits(B, Hkv, hd, ctx, sms);
  return FK_OK;
}
fk_status attention_decode_run(const void* q, const void* kc, const void* vc, int B, int Hq, int Hkv, int hd, int cap,
                               int ctx, int window, int splits, void* out, cudaStream_t st) {
  cudaError_t e = launch_attention_decode(q, Hq * hd, kc, vc, cap, B, ctx, nullptr, Hq, Hkv, hd, window,
                                          1.0f / sqrtf((float)hd), splits, out, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention decode launch");
  return FK_OK;
}
}  // namespace fk

extern "C" size_t fk_attention_decode_scratch_bytes(int32_t batch, int32_t n_q_heads, int32_t n_kv_heads,
                                                    int32_t head_dim, int32_t ctx) {
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || ctx < 1) return 0;
  return kDecodeScratchBytes;
}

extern "C" fk_status fk_attention_decode(const void* d_q, const void* d_kcache, const void* d_vcache, int32_t batch,
                                         int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t cap,
                                         int32_t ctx, int32_t window, void* d_scratch, size_t scratch_bytes,
                                         void* d_out, void* stream) {
  fk_status s = check_decode_args(d_q, d_kcache, d_vcache, batch, n_q_heads, n_kv_heads, head_dim, cap, ctx, window,
                                  d_out);
  if (s != FK_OK) return s;
  if (!d_scratch || scratch_bytes < kDecodeScratchBytes)
    return fk::fail(FK_ERR_WORKSPACE, "attention decode: scratch too small");
  int splits = 1;
  s = fk::attention_decode_plan(batch, n_kv_heads, head_dim, ctx, &splits);
  if (s != FK_OK) return s;
  return fk::attention_decode_run(d_q, d_kcache, d_vcache, batch, n_q_heads, n_kv_heads, head_dim, cap, ctx, window,
                                  splits, d_out, static_cast<cudaStream_t>(stream));
}
