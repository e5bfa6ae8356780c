// Causal GQA attention over the bf16 KV cache ("N7 · model/forward-parity",
// Thm 1: causal multi-head/GQA attention; Thm 2 and "pegainfer #878":
// sliding-window local layers).
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

#include "fk_common.cuh"
#include "fk_internal.h"
#include "fk_ops.h"

namespace fk {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

FK_DEVICE void ldsm_x4(uint32_t* r, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
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
FK_DEVICE void mma_f16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// both operands bf16, or both IEEE f16
FK_DEVICE void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1, int f16) {
  if (f16)
    mma_f16_16816(d, a, b0, b1);
  else
    mma_bf16_16816(d, a, b0, b1);
}

// element (r, c) of a [rows][COLS] bf16 tile, 16-byte chunks XOR-swizzled by row
template <int COLS>
FK_DEVICE int swz(int r, int c) {
  return r * COLS + ((((c >> 3) ^ (r & 7))) << 3) + (c & 7);
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
  const uint16_t* q;  // 16-bit: bf16 or IEEE f16 (io_f16)
  int ldq;
  int cap, ctx_host;
  const int* d_ctx;  // non-null: ctx = *d_ctx + 1
  int Hq, Hkv, window;
  float scale_log2;
  uint16_t* o;  // bf16 or f16 (out_f16)
  unsigned* dev_err;  // optional device error word (pipeline timeouts)
  // fused RoPE
  const float2* rope;  // [positions][HD/2] (cos, sin) of frequency j
  int qk_norm;
  const __nv_bfloat16* q_norm;
  const __nv_bfloat16* k_norm;
  float eps;
  uint16_t* kc_w;  // the caches, written at position ctx-1
  uint16_t* vc_w;
  int io_f16;   // q, k, v, the caches and the probabilities are IEEE f16 (else bf16): picks the kernel
  int out_f16;  // the output is stored as f16 (else bf16)
};

// [QK-norm and] RoPE of one head held by a warp: lane owns elements
// e0..e0+C-1 of each half (pairs (j, j+HD/2)); cs: this lane's (cos, sin).
template <int HD, bool F16>
FK_DEVICE void rope_head(const uint16_t* src, const DecArgs& a, const __nv_bfloat16* nw, const float2* cs,
                         int lane, float* olo, float* ohi) {
  constexpr int C = HD / 64, HALF = HD / 2;
  const int e0 = lane * C;
  float lo[C], hi[C];
#pragma unroll
  for (int i = 0; i < C; ++i) {
    lo[i] = load_16(src + e0 + i, F16);
    hi[i] = load_16(src + HALF + e0 + i, F16);
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

template <int HD, bool ROPE, bool F16>
__global__ void __launch_bounds__(kDecThreads) attn_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV,
                                                                  const DecArgs a) {
  constexpr int io_f16 = F16 ? 1 : 0;  // q, k, v, the caches and P are IEEE f16 (else bf16)
  using C = DecCfg<HD>;
  constexpr int NC = HD / 64, HALF = HD / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint16_t* sQ = reinterpret_cast<uint16_t*>(smem);
  uint8_t* ring = smem + C::RING_OFF;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::NST);
  __shared__ __align__(16) uint16_t sNew[2][HD];  // fused RoPE: the new key and value
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
          tma_load_2d(&tmK, &full[stage], sk + c * kDecTile * 64 * 2, c * 64, head_row * cap + pos % cap);
        tma_load_2d(&tmV, &full[stage], sv, pos % cap, head_row * HD);
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
      const uint16_t* row = a.q + (size_t)b * a.ldq;
      for (int r = warp; r < 16; r += kDecConsumers / 32) {
        float olo[NC], ohi[NC];
        if (r < group) {
          rope_head<HD, F16>(row + (size_t)(g * group + r) * HD, a, a.q_norm, cs, lane, olo, ohi);
        } else {
#pragma unroll
          for (int i = 0; i < NC; ++i) olo[i] = ohi[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          sQ[swz<HD>(r, lane * NC + i)] = bits_16(olo[i], io_f16);
          sQ[swz<HD>(r, HALF + lane * NC + i)] = bits_16(ohi[i], io_f16);
        }
      }
      if (warp == 0) {
        float olo[NC], ohi[NC];
        rope_head<HD, F16>(row + (size_t)(Hq + g) * HD, a, a.k_norm, cs, lane, olo, ohi);
#pragma unroll
        for (int i = 0; i < NC; ++i) {
          sNew[0][lane * NC + i] = bits_16(olo[i], io_f16);
          sNew[0][HALF + lane * NC + i] = bits_16(ohi[i], io_f16);
        }
      } else if (warp == 1) {
        const uint16_t* vs = row + (size_t)(Hq + Hkv + g) * HD;
        for (int d = lane; d < HD; d += 32) sNew[1][d] = vs[d];
      }
      consumers_sync();
      if (t_new >= 0 && t_new < ntiles) {  // the one CTA whose tiles hold the new token stores it
        uint16_t* kw = a.kc_w + ((size_t)head_row * cap + qpos % cap) * HD;
        uint16_t* vw = a.vc_w + (size_t)head_row * HD * cap + qpos % cap;
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
      uint16_t* tK = reinterpret_cast<uint16_t*>(ring + stage * C::STAGE_BYTES);
      uint16_t* tV = tK + C::TILE_ELEMS;
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
        mma_16816(s[0], qa, bb[0], bb[1], io_f16);
        mma_16816(s[1], qa, bb[2], bb[3], io_f16);
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
      pa[0] = pack_16x2(s[0][0], s[0][1], io_f16);
      pa[1] = pack_16x2(s[0][2], s[0][3], io_f16);
      pa[2] = pack_16x2(s[1][0], s[1][1], io_f16);
      pa[3] = pack_16x2(s[1][2], s[1][3], io_f16);
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
        mma_16816(oacc[2 * dp], pa, bb[0], bb[1], io_f16);
        mma_16816(oacc[2 * dp + 1], pa, bb[2], bb[3], io_f16);
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
    store_16(a.o + ((size_t)b * Hq + g * group + r) * HD + (i - r * HD), L > 0.f ? acc / L : 0.f, a.out_f16);
  }
  cluster_sync();  // no CTA leaves while another may still read its partial
}

}  // namespace

// Largest cluster of decode CTAs the GPU co-schedules for this head_dim
// (a cluster of 16 is beyond the portable size and is allowed explicitly).
template <int HD, bool ROPE, bool F16>
cudaError_t decode_attrs() {
  using C = DecCfg<HD>;
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<HD, ROPE, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_decode_kernel<HD, ROPE, F16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

template <int HD>
int decode_max_cluster(cudaError_t* err) {
  using C = DecCfg<HD>;
  static DeviceOnce once;
  static int n[kMaxDevices];
  int dev = 0;
  cudaGetDevice(&dev);
  *err = once.run([dev] {
    cudaError_t e0 = decode_attrs<HD, false, false>();
    if (e0 == cudaSuccess) e0 = decode_attrs<HD, true, false>();
    if (e0 == cudaSuccess) e0 = decode_attrs<HD, false, true>();
    if (e0 == cudaSuccess) e0 = decode_attrs<HD, true, true>();
    if (e0 != cudaSuccess) return e0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kMaxCluster, 1, 1);
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    int c = 0, c2 = 0;
    if (cudaOccupancyMaxPotentialClusterSize(&c, attn_decode_kernel<HD, false, false>, &cfg) != cudaSuccess ||
        cudaOccupancyMaxPotentialClusterSize(&c2, attn_decode_kernel<HD, true, false>, &cfg) != cudaSuccess || c < 1 ||
        c2 < 1) {
      cudaGetLastError();
      c = c2 = 8;  // the portable size
    }
    n[dev] = std::min(std::min(c, c2), kMaxCluster);
    return cudaSuccess;
  });
  return *err == cudaSuccess ? n[dev] : 1;
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
  auto kernel = rope ? (a.io_f16 ? attn_decode_kernel<HD, true, true> : attn_decode_kernel<HD, true, false>)
                     : (a.io_f16 ? attn_decode_kernel<HD, false, true> : attn_decode_kernel<HD, false, false>);
  return fk_launch_cluster(kernel, grid, kDecThreads, C::SMEM, st, n_splits, tK, tV, a);
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
                                    int n_splits, void* o, unsigned* dev_err, cudaStream_t st, int io_f16,
                                    int out_f16) {
  DecArgs a = {};
  a.dev_err = dev_err;
  a.q = static_cast<const uint16_t*>(q);
  a.ldq = ldq;
  a.cap = cap;
  a.ctx_host = ctx;
  a.d_ctx = d_ctx;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.window = window;
  a.scale_log2 = scale * kLog2e;
  a.o = static_cast<uint16_t*>(o);
  a.io_f16 = io_f16;
  a.out_f16 = out_f16;
  return decode_dispatch(kcache, vcache, a, false, hd, B, n_splits, st);
}

cudaError_t launch_attention_decode_rope(const void* qkv, int ldqkv, void* kcache, void* vcache, int cap, int B,
                                         const int* d_ctx, int Hq, int Hkv, int hd, int window, float scale,
                                         const float2* rope, int qk_norm, const void* q_norm, const void* k_norm,
                                         float eps, int n_splits, void* o, unsigned* dev_err, cudaStream_t st,
                                         int io_f16, int out_f16) {
  if (!d_ctx) return cudaErrorInvalidValue;
  DecArgs a = {};
  a.q = static_cast<const uint16_t*>(qkv);
  a.ldq = ldqkv;
  a.kc_w = static_cast<uint16_t*>(kcache);
  a.vc_w = static_cast<uint16_t*>(vcache);
  a.io_f16 = io_f16;
  a.out_f16 = out_f16;
  a.cap = cap;
  a.d_ctx = d_ctx;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.window = window;
  a.scale_log2 = scale * kLog2e;
  a.o = static_cast<uint16_t*>(o);
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
extern "C" fk_status fk_attention_decode(const void* d_q, const void* d_kcache, const void* d_vcache, int32_t batch,
                                         int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, int32_t cap,
                                         int32_t ctx, int32_t window, void* d_out, void* stream) {
  using fk::fail;
  if (!d_q || !d_kcache || !d_vcache || !d_out) return fail(FK_ERR_INVALID_ARG, "attention decode: null pointer");
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads || n_q_heads / n_kv_heads > 8)
    return fail(FK_ERR_INVALID_ARG, "attention decode: need batch >= 1 and 1..8 query heads per kv head");
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(FK_ERR_INVALID_ARG, "attention decode: head_dim 64/128/256");
  if (ctx < 1 || window < 0 || cap < 64 || cap % 64 || (ctx > cap && (window == 0 || window > cap)))
    return fail(FK_ERR_INVALID_ARG, "attention decode: need cap % 64 == 0 and 1 <= ctx <= cap (or window <= cap)");
  if ((reinterpret_cast<uintptr_t>(d_q) | reinterpret_cast<uintptr_t>(d_kcache) |
       reinterpret_cast<uintptr_t>(d_vcache) | reinterpret_cast<uintptr_t>(d_out)) & 15)
    return fail(FK_ERR_INVALID_ARG, "attention decode: buffers must be 16-byte aligned");
  int sms = 0;
  fk_status s = fk::check_device(&sms);
  if (s != FK_OK) return s;
  unsigned* ctl = nullptr;
  s = fk::op_control_block(&ctl);
  if (s != FK_OK) return s;
  const int splits = fk::decode_attention_splits(batch, n_kv_heads, head_dim, ctx, sms);
  cudaError_t e = fk::launch_attention_decode(d_q, n_q_heads * head_dim, d_kcache, d_vcache, cap, batch, ctx, nullptr,
                                              n_q_heads, n_kv_heads, head_dim, window, 1.0f / sqrtf((float)head_dim),
                                              splits, d_out, ctl, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fk::cuda_fail(e, "attention decode launch");
  return FK_OK;
}
