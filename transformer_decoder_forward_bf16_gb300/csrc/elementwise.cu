// Bandwidth-bound kernels of the forward pass: embedding gather (+scale) with
// the first RMSNorm fused, RMSNorm, the sandwich post-norm + residual +
// next-norm fusion, QK-norm + RoPE + K-cache write, the V-cache transpose of
// a prefill chunk, and the per-row argmax with its top-2 margin.
//
// Row kernels read with 16-byte vector loads and reduce with warp shuffles
// (one warp per row, or one block per row with the row held in registers);
// the V transpose stages its tile in shared memory so that both sides move
// 128-byte runs.
#include <algorithm>

#include "fk_common.cuh"
#include "fk_ops.h"

namespace fk {

namespace {

// 8 bf16 values from a 16-byte load, widened to fp32
FK_DEVICE void load8_bf16(const __nv_bfloat16* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(u.x);
  v[1] = bf16_hi(u.x);
  v[2] = bf16_lo(u.y);
  v[3] = bf16_hi(u.y);
  v[4] = bf16_lo(u.z);
  v[5] = bf16_hi(u.z);
  v[6] = bf16_lo(u.w);
  v[7] = bf16_hi(u.w);
}
// 8 values to 16 bytes of bf16 (f16 == 0) or IEEE f16
FK_DEVICE void store8_16(void* p, const float* v, int f16) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_16x2(v[0], v[1], f16), pack_16x2(v[2], v[3], f16),
                                            pack_16x2(v[4], v[5], f16), pack_16x2(v[6], v[7], f16));
}

// ---------------------------------------------------------------------------
// embedding: x[t] = E[id_t] * scale (fp32), u[t] = RMSNorm(x[t]) * w (bf16)
// ("N7 · model/forward-parity", Thm 1: embedding lookup; "pegainfer #878":
// scaled embedding; the first pre-attention RMSNorm is fused in).
// ---------------------------------------------------------------------------
__global__ void embed_norm_kernel(const int32_t* __restrict__ ids, const __nv_bfloat16* __restrict__ E, int T, int H,
                                  int V, float scale, const __nv_bfloat16* __restrict__ w, float eps,
                                  float* __restrict__ x, uint16_t* __restrict__ u, unsigned* dev_err, int u_f16) {
  pdl_trigger();
  pdl_wait();
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int id = ids[t];
  if (id < 0 || id >= V) {
    if (lane == 0 && dev_err) atomicOr(dev_err, FK_DEVERR_TOKEN_RANGE);
    id = id < 0 ? 0 : V - 1;
  }
  const __nv_bfloat16* e = E + (size_t)id * H;
  float* xr = x + (size_t)t * H;
  float ss = 0.f;
  for (int c = lane * 8; c < H; c += 256) {
    float v[8];
    load8_bf16(e + c, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] *= scale;
      ss += v[j] * v[j];
    }
    *reinterpret_cast<float4*>(xr + c) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(xr + c + 4) = make_float4(v[4], v[5], v[6], v[7]);
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / H + eps);
  uint16_t* ur = u + (size_t)t * H;
  for (int c = lane * 8; c < H; c += 256) {
    float v[8], wv[8];
    load8_bf16(e + c, v);
    load8_bf16(w + c, wv);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = v[j] * scale * r * wv[j];
    store8_16(ur + c, v, u_f16);
  }
}

// ---------------------------------------------------------------------------
// u[t] = RMSNorm(x[t]) * w  ("N7", Thm 1: RMSNorm), fp32 in, bf16 out
// ---------------------------------------------------------------------------
__global__ void rmsnorm_kernel(const float* __restrict__ x, int ldx, int T, int H, const __nv_bfloat16* __restrict__ w,
                               float eps, uint16_t* __restrict__ u, int ldu, int u_f16) {
  pdl_trigger();
  pdl_wait();
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* xr = x + (size_t)t * ldx;
  float ss = 0.f;
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(xr + c);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / H + eps);
  uint16_t* ur = u + (size_t)t * ldu;
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(xr + c);
    const uint2 wp = *reinterpret_cast<const uint2*>(w + c);
    *reinterpret_cast<uint2*>(ur + c) =
        make_uint2(pack_16x2(v.x * r * bf16_lo(wp.x), v.y * r * bf16_hi(wp.x), u_f16),
                   pack_16x2(v.z * r * bf16_lo(wp.y), v.w * r * bf16_hi(wp.y), u_f16));
  }
}

// The same normalisation for few rows: one 256-thread block per row, the row
// held in registers (16-byte loads, one read of x), block-wide reduction.
constexpr int kRowsThreads = 256;
constexpr int kRowsMaxVec = 8;  // float4 per thread: H <= 8192
__global__ void __launch_bounds__(kRowsThreads) rmsnorm_rows_kernel(const float* __restrict__ x, int ldx, int H,
                                                                    const __nv_bfloat16* __restrict__ w, float eps,
                                                                    uint16_t* __restrict__ u, int ldu, int u_f16) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[kRowsThreads / 32];
  const int t = blockIdx.x;
  const float* xr = x + (size_t)t * ldx;
  float4 v[kRowsMaxVec];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kRowsMaxVec; ++i) {
    const int c = (i * kRowsThreads + threadIdx.x) * 4;
    v[i] = c < H ? *reinterpret_cast<const float4*>(xr + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kRowsThreads / 32; ++i) tot += red[i];
  const float r = rsqrtf(tot / H + eps);
  uint16_t* ur = u + (size_t)t * ldu;
#pragma unroll
  for (int i = 0; i < kRowsMaxVec; ++i) {
    const int c = (i * kRowsThreads + threadIdx.x) * 4;
    if (c < H) {
      const uint2 wp = *reinterpret_cast<const uint2*>(w + c);
      *reinterpret_cast<uint2*>(ur + c) =
          make_uint2(pack_16x2(v[i].x * r * bf16_lo(wp.x), v[i].y * r * bf16_hi(wp.x), u_f16),
                     pack_16x2(v[i].z * r * bf16_lo(wp.y), v[i].w * r * bf16_hi(wp.y), u_f16));
    }
  }
}

// fp32-output variant for the final-norm hidden slot
__global__ void rmsnorm_f32_kernel(const float* __restrict__ x, int T, int H, const __nv_bfloat16* __restrict__ w,
                                   float eps, float* __restrict__ y) {
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* xr = x + (size_t)t * H;
  float ss = 0.f;
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(xr + c);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / H + eps);
  float* yr = y + (size_t)t * H;
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(xr + c);
    const uint2 wp = *reinterpret_cast<const uint2*>(w + c);
    *reinterpret_cast<float4*>(yr + c) =
        make_float4(v.x * r * bf16_lo(wp.x), v.y * r * bf16_hi(wp.x), v.z * r * bf16_lo(wp.y), v.w * r * bf16_hi(wp.y));
  }
}

// ---------------------------------------------------------------------------
// Sandwich norm: x_out = x_in + RMSNorm(a) * w_post, then
// u = RMSNorm(x_out) * w_next ("N7", Thm 2: gemma3 sandwich norm).
// x_out may alias x_in.
// ---------------------------------------------------------------------------
__global__ void post_norm_residual_kernel(const float* __restrict__ a, const float* x_in, float* x_out, int T, int H,
                                          const __nv_bfloat16* __restrict__ w_post,
                                          const __nv_bfloat16* __restrict__ w_next, float eps,
                                          uint16_t* __restrict__ u, int u_f16) {
  pdl_trigger();
  pdl_wait();
  const int warps = blockDim.x >> 5;
  const int t = blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* ar = a + (size_t)t * H;
  const float* xi = x_in + (size_t)t * H;
  float* xo = x_out + (size_t)t * H;
  float ss = 0.f;
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(ar + c);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / H + eps);
  float ss2 = 0.f;
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(ar + c);
    const float4 xv = *reinterpret_cast<const float4*>(xi + c);
    const uint2 wp = *reinterpret_cast<const uint2*>(w_post + c);
    float4 o;
    o.x = xv.x + v.x * r * bf16_lo(wp.x);
    o.y = xv.y + v.y * r * bf16_hi(wp.x);
    o.z = xv.z + v.z * r * bf16_lo(wp.y);
    o.w = xv.w + v.w * r * bf16_hi(wp.y);
    ss2 += o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w;
    *reinterpret_cast<float4*>(xo + c) = o;
  }
  ss2 = warp_sum(ss2);
  const float r2 = rsqrtf(ss2 / H + eps);
  __syncwarp();
  uint16_t* ur = u + (size_t)t * H;
  for (int c = lane * 4; c < H; c += 128) {
    const float4 v = *reinterpret_cast<const float4*>(xo + c);
    const uint2 wp = *reinterpret_cast<const uint2*>(w_next + c);
    *reinterpret_cast<uint2*>(ur + c) =
        make_uint2(pack_16x2(v.x * r2 * bf16_lo(wp.x), v.y * r2 * bf16_hi(wp.x), u_f16),
                   pack_16x2(v.z * r2 * bf16_lo(wp.y), v.w * r2 * bf16_hi(wp.y), u_f16));
  }
}

// ---------------------------------------------------------------------------
// QK-norm + RoPE + KV-cache write ("N7", Thm 1: RoPE on q and k; Thm 2: qwen3
// / gemma3 QK-norm). Head element j pairs with j + hd/2. Each lane owns 8
// consecutive elements of each half of a head (16-byte loads and stores), so
// a head takes hd/16 lanes and a warp covers 512/hd heads of one token (4 at
// hd = 128): enough bytes in flight per warp to stream at the memory's rate.
//   q: rotated in place inside the qkv rows;
//   k: rotated and written to kcache[b][g][pos][:]
// (v goes to the transposed value cache through v_cache_kernel below).
// rope: float2 (cos, sin) table [positions][hd/2].
// ---------------------------------------------------------------------------
template <int C>
__global__ void rope_qkv_kernel(uint16_t* qkv, int ldqkv, int T, int S, int pos0, int Hq,
                                int Hkv, const float2* __restrict__ rope, int qk_norm,
                                const __nv_bfloat16* __restrict__ q_norm, const __nv_bfloat16* __restrict__ k_norm,
                                float eps, uint16_t* kcache, int cap, int f16) {
  pdl_trigger();
  pdl_wait();
  constexpr int HD = C * 64;
  constexpr int HALF = HD / 2;
  constexpr int LPH = HALF / 8;    // lanes per head
  constexpr int HPW = 32 / LPH;    // heads per warp
  const int warps = blockDim.x >> 5;
  const long gw = (long)blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int nh = Hq + Hkv;  // q and k heads; v is moved by v_cache_kernel
  const int groups = (nh + HPW - 1) / HPW;
  if (gw >= (long)T * groups) return;  // warp-uniform
  const int t = (int)(gw / groups);
  const int h = (int)(gw % groups) * HPW + lane / LPH;
  const bool live = h < nh;
  const int b = t / S, s = t % S;
  const int pos = pos0 + s;
  const int e0 = (lane % LPH) * 8;  // within each half
  uint16_t* row = qkv + (size_t)t * ldqkv + (size_t)h * HD;
  float lo[8], hi[8];
  if (live) {
    const uint4 a = *reinterpret_cast<const uint4*>(row + e0);
    const uint4 c = *reinterpret_cast<const uint4*>(row + HALF + e0);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo[2 * i] = lo_16(aw[i], f16);
      lo[2 * i + 1] = hi_16(aw[i], f16);
      hi[2 * i] = lo_16(cw[i], f16);
      hi[2 * i + 1] = hi_16(cw[i], f16);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) lo[i] = hi[i] = 0.f;
  }
  const bool is_q = h < Hq;
  if (qk_norm) {  // every lane takes part in the shuffles
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += lo[i] * lo[i] + hi[i] * hi[i];
#pragma unroll
    for (int o = LPH / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / HD + eps);
    const __nv_bfloat16* nw = is_q ? q_norm : k_norm;
    if (live) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        lo[i] = lo[i] * r * __bfloat162float(nw[e0 + i]);
        hi[i] = hi[i] * r * __bfloat162float(nw[HALF + e0 + i]);
      }
    }
  }
  if (!live) return;
  const float4* cs = reinterpret_cast<const float4*>(rope + (size_t)pos * HALF + e0);
  uint32_t olo[4], ohi[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 c = cs[i];  // (cos, sin) of elements 2i and 2i + 1
    olo[i] = pack_16x2(lo[2 * i] * c.x - hi[2 * i] * c.y, lo[2 * i + 1] * c.z - hi[2 * i + 1] * c.w, f16);
    ohi[i] = pack_16x2(hi[2 * i] * c.x + lo[2 * i] * c.y, hi[2 * i + 1] * c.z + lo[2 * i + 1] * c.w, f16);
  }
  uint16_t* dst;
  if (is_q) {
    dst = row;
  } else {
    const int g = h - Hq;
    dst = kcache + (((size_t)b * Hkv + g) * cap + pos % cap) * HD;  // position p lives in slot p mod cap
  }
  *reinterpret_cast<uint4*>(dst + e0) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
  *reinterpret_cast<uint4*>(dst + HALF + e0) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
}

// V rows of a prefill chunk into the transposed cache vcache[b][g][d][pos]:
// one CTA per (64 positions, kv head, sequence) stages the [64][HD] tile in
// shared memory and writes each cache row d as one run of 64 positions, so
// both the reads and the writes are full 128-byte segments.
constexpr int kVTile = 64;
template <int HD>
__global__ void __launch_bounds__(256) v_cache_kernel(const __nv_bfloat16* __restrict__ qkv, int ldqkv, int S, int pos0,
                                                      int Hq, int Hkv, __nv_bfloat16* __restrict__ vcache, int cap) {
  pdl_trigger();
  pdl_wait();
  constexpr int LD = HD + 2;  // padded row: the transposed reads of 8 positions hit distinct banks
  __shared__ __align__(16) __nv_bfloat16 tile[kVTile * LD];
  const int s0 = blockIdx.x * kVTile, g = blockIdx.y, b = blockIdx.z;
  const int n = min(kVTile, S - s0);
  constexpr int CPR = HD / 8;  // 16-byte chunks per row
  for (int i = threadIdx.x; i < n * CPR; i += blockDim.x) {
    const int r = i / CPR, c = i % CPR;
    const uint4 v = *reinterpret_cast<const uint4*>(qkv + (size_t)(b * S + s0 + r) * ldqkv + (size_t)(Hq + Hkv + g) * HD +
                                                    c * 8);
    uint32_t* t32 = reinterpret_cast<uint32_t*>(tile + r * LD + c * 8);  // 4-byte aligned (LD even)
    t32[0] = v.x;
    t32[1] = v.y;
    t32[2] = v.z;
    t32[3] = v.w;
  }
  __syncthreads();
  // position P lives in slot P mod cap (cap a multiple of 64: a ring for
  // sliding-window layers, larger than every position otherwise)
  __nv_bfloat16* dst = vcache + ((size_t)b * Hkv + g) * HD * cap;
  const int P0 = pos0 + s0;
  if ((P0 & 7) == 0) {  // 16-byte aligned runs: 8 positions per store, never across the wrap
    constexpr int CPD = kVTile / 8;
    for (int i = threadIdx.x; i < HD * CPD; i += blockDim.x) {
      const int d = i / CPD, p = (i % CPD) * 8;
      if (p >= n) continue;
      __nv_bfloat16* row = dst + (size_t)d * cap;
      if (p + 8 <= n) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint16_t lo = reinterpret_cast<const uint16_t&>(tile[(p + 2 * j) * LD + d]);
          const uint16_t hi = reinterpret_cast<const uint16_t&>(tile[(p + 2 * j + 1) * LD + d]);
          w[j] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        *reinterpret_cast<uint4*>(row + (P0 + p) % cap) = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
        for (int j = p; j < n; ++j) row[(P0 + j) % cap] = tile[j * LD + d];
      }
    }
  } else {
    for (int i = threadIdx.x; i < HD * kVTile; i += blockDim.x) {
      const int d = i / kVTile, p = i % kVTile;
      if (p < n) dst[(size_t)d * cap + (P0 + p) % cap] = tile[p * LD + d];
    }
  }
}

// ---------------------------------------------------------------------------
// argmax per row over V fp32 values (lowest index wins ties) and the top-2
// margin: the row maximum minus the largest other value (0 on a tie), the
// quantity that decides whether rounding noise can flip the argmax ("N7 ·
// model/forward-parity", Thm 3: near-tie argmax flips).
// Each thread keeps (best value, its index, runner-up value); two such states
// merge into the better best, and the runner-up is the larger of the loser's
// best and the winner's runner-up. One block of 256 threads per row.
// ---------------------------------------------------------------------------
struct Top2 {
  float m;   // best value
  int i;     // its index (lowest on ties)
  float m2;  // largest value at any other index
};

FK_DEVICE bool wins(float m2, int i2, float m, int i) { return m2 > m || (m2 == m && i2 < i); }

FK_DEVICE void top2_push(Top2& t, float v, int c) {
  if (wins(v, c, t.m, t.i)) {
    t.m2 = fmaxf(t.m2, t.m);
    t.m = v;
    t.i = c;
  } else {
    t.m2 = fmaxf(t.m2, v);
  }
}

FK_DEVICE void top2_merge(Top2& t, const Top2& o) {
  if (wins(o.m, o.i, t.m, t.i)) {
    t.m2 = fmaxf(t.m, o.m2);
    t.m = o.m;
    t.i = o.i;
  } else {
    t.m2 = fmaxf(t.m2, o.m);
  }
}

FK_DEVICE Top2 top2_shfl(const Top2& t, int o) {
  Top2 r;
  r.m = __shfl_xor_sync(0xffffffffu, t.m, o);
  r.i = __shfl_xor_sync(0xffffffffu, t.i, o);
  r.m2 = __shfl_xor_sync(0xffffffffu, t.m2, o);
  return r;
}

// The block's threads reduce their states; thread 0 gets the result.
FK_DEVICE Top2 top2_block(Top2 t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) top2_merge(t, top2_shfl(t, o));
  __shared__ float sm[32], sm2[32];
  __shared__ int si[32];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm[w] = t.m;
    si[w] = t.i;
    sm2[w] = t.m2;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < (int)(blockDim.x >> 5); ++k) top2_merge(t, Top2{sm[k], si[k], sm2[k]});
  }
  return t;
}

FK_DEVICE void top2_scan(Top2& t, const float* row, int c0, int c1, bool vec) {
  if (vec) {
    for (int c = c0 + threadIdx.x * 4; c < c1; c += blockDim.x * 4) {
      if (c + 4 <= c1) {
        const float4 v = *reinterpret_cast<const float4*>(row + c);
        top2_push(t, v.x, c);
        top2_push(t, v.y, c + 1);
        top2_push(t, v.z, c + 2);
        top2_push(t, v.w, c + 3);
      } else {
        for (int e = c; e < c1; ++e) top2_push(t, row[e], e);
      }
    }
  } else {
    for (int c = c0 + threadIdx.x; c < c1; c += blockDim.x) top2_push(t, row[c], c);
  }
}

FK_DEVICE void top2_store(const Top2& t, int r, int32_t* out, int32_t* out2, float* margin) {
  const int best = t.i == 0x7fffffff ? 0 : t.i;
  out[r] = best;
  if (out2) out2[r] = best;
  if (margin) margin[r] = t.m - t.m2;
}

__global__ void argmax_kernel(const float* __restrict__ z, int R, int V, int ldz, int32_t* __restrict__ out,
                              int32_t* __restrict__ out2, float* __restrict__ margin) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  if (r >= R) return;
  Top2 t{-INFINITY, 0x7fffffff, -INFINITY};
  top2_scan(t, z + (size_t)r * ldz, 0, V, (V & 3) == 0 && (ldz & 3) == 0);
  t = top2_block(t);
  if (threadIdx.x == 0) top2_store(t, r, out, out2, margin);
}

// The same for few rows split across blocks: block (s, r) scans one column
// chunk of row r and records its state; the last block of a row (arrival
// counter, reset after use) merges the chunk states in chunk order, so the
// result does not depend on scheduling.
constexpr int kArgmaxSplits = 32;
__global__ void argmax_split_kernel(const float* __restrict__ z, int V, int ldz, int32_t* __restrict__ out,
                                    int32_t* __restrict__ out2, float* __restrict__ margin, float* part_m,
                                    int* part_i, float* part_m2, unsigned* counters) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.y, sp = blockIdx.x;
  const int chunk = ((V + kArgmaxSplits - 1) / kArgmaxSplits + 1023) / 1024 * 1024;
  const int c0 = sp * chunk, c1 = min(V, c0 + chunk);
  Top2 t{-INFINITY, 0x7fffffff, -INFINITY};
  top2_scan(t, z + (size_t)r * ldz, c0, c1, true);
  t = top2_block(t);
  __shared__ int last;
  if (threadIdx.x == 0) {
    part_m[r * kArgmaxSplits + sp] = t.m;
    part_i[r * kArgmaxSplits + sp] = t.i;
    part_m2[r * kArgmaxSplits + sp] = t.m2;
    __threadfence();
    last = atomicAdd(&counters[r], 1u) == kArgmaxSplits - 1;
  }
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  Top2 b{-INFINITY, 0x7fffffff, -INFINITY};
  for (int i = 0; i < kArgmaxSplits; ++i)
    top2_merge(b, Top2{__ldcg(part_m + r * kArgmaxSplits + i), __ldcg(part_i + r * kArgmaxSplits + i),
                       __ldcg(part_m2 + r * kArgmaxSplits + i)});
  top2_store(b, r, out, out2, margin);
  counters[r] = 0;
}

// copy the last position of each sequence: dst[b] = src[b*S + S-1]
__global__ void gather_last_rows_kernel(const __nv_bfloat16* src, int ld, int S, int H, int B,
                                        __nv_bfloat16* dst) {
  const int b = blockIdx.x;
  if (b >= B) return;
  const __nv_bfloat16* s = src + ((size_t)b * S + S - 1) * ld;
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8)
    *reinterpret_cast<uint4*>(dst + (size_t)b * H + c) = *reinterpret_cast<const uint4*>(s + c);
}

// bf16 -> IEEE f16 copy (8 elements per 16-byte load), for the f16 copies of
// the weights of GEMMs whose input activations are stored as f16
__global__ void bf16_to_f16_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n8) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 u = src[i];
    dst[i] = make_uint4(pack_f16x2(bf16_lo(u.x), bf16_hi(u.x)), pack_f16x2(bf16_lo(u.y), bf16_hi(u.y)),
                        pack_f16x2(bf16_lo(u.z), bf16_hi(u.z)), pack_f16x2(bf16_lo(u.w), bf16_hi(u.w)));
  }
}

__global__ void set_int_kernel(int* p, int value) { *p = value; }
__global__ void inc_int_kernel(int* p) {
  pdl_wait();
  *p += 1;
}

constexpr int kRowThreads = 256;  // 8 rows per block
inline int row_blocks(long rows) { return (int)((rows + 7) / 8); }

}  // namespace

cudaError_t launch_embed_norm(const int32_t* ids, const void* E, int T, int H, int V, float scale, const void* w,
                              float eps, float* x, void* u, unsigned* dev_err, cudaStream_t st, int u_f16) {
  if (T == 0) return cudaSuccess;
  return fk_launch(embed_norm_kernel, row_blocks(T), kRowThreads, 0, st, ids, static_cast<const __nv_bfloat16*>(E), T, H,
                   V, scale, static_cast<const __nv_bfloat16*>(w), eps, x, static_cast<uint16_t*>(u), dev_err, u_f16);
}

cudaError_t launch_rmsnorm(const float* x, int ldx, int T, int H, const void* w, float eps, void* u, int ldu,
                           cudaStream_t st, int u_f16) {
  if (T == 0) return cudaSuccess;
  if (H <= kRowsThreads * 4 * kRowsMaxVec) {
    return fk_launch(rmsnorm_rows_kernel, T, kRowsThreads, 0, st, x, ldx, H, static_cast<const __nv_bfloat16*>(w), eps,
                     static_cast<uint16_t*>(u), ldu, u_f16);
  }
  return fk_launch(rmsnorm_kernel, row_blocks(T), kRowThreads, 0, st, x, ldx, T, H, static_cast<const __nv_bfloat16*>(w),
                   eps, static_cast<uint16_t*>(u), ldu, u_f16);
}

cudaError_t launch_rmsnorm_f32(const float* x, int T, int H, const void* w, float eps, float* y, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  rmsnorm_f32_kernel<<<row_blocks(T), kRowThreads, 0, st>>>(x, T, H, static_cast<const __nv_bfloat16*>(w), eps, y);
  return cudaGetLastError();
}

cudaError_t launch_post_norm_residual(const float* a, const float* x_in, float* x_out, int T, int H,
                                      const void* w_post, const void* w_next, float eps, void* u, cudaStream_t st,
                                      int u_f16) {
  if (T == 0) return cudaSuccess;
  return fk_launch(post_norm_residual_kernel, row_blocks(T), kRowThreads, 0, st, a, x_in, x_out, T, H,
                   static_cast<const __nv_bfloat16*>(w_post), static_cast<const __nv_bfloat16*>(w_next), eps,
                   static_cast<uint16_t*>(u), u_f16);
}

cudaError_t launch_rope_qkv(void* qkv, int ldqkv, int T, int S, int pos0, int Hq, int Hkv, int hd,
                            const float2* rope, int qk_norm, const void* q_norm, const void* k_norm, float eps,
                            void* kcache, void* vcache, int cap, cudaStream_t st, int f16) {
  if (T == 0) return cudaSuccess;
  if (ldqkv % 8) return cudaErrorInvalidValue;  // rows 16-byte aligned
  {
    const dim3 grid((S + kVTile - 1) / kVTile, Hkv, T / S);
    const auto* src = static_cast<const __nv_bfloat16*>(qkv);
    auto* vdst = static_cast<__nv_bfloat16*>(vcache);
    cudaError_t e = cudaErrorInvalidValue;
    if (hd == 64) e = fk_launch(v_cache_kernel<64>, grid, 256, 0, st, src, ldqkv, S, pos0, Hq, Hkv, vdst, cap);
    if (hd == 128) e = fk_launch(v_cache_kernel<128>, grid, 256, 0, st, src, ldqkv, S, pos0, Hq, Hkv, vdst, cap);
    if (hd == 256) e = fk_launch(v_cache_kernel<256>, grid, 256, 0, st, src, ldqkv, S, pos0, Hq, Hkv, vdst, cap);
    if (e != cudaSuccess) return e;
  }
  const int hpw = 512 / hd;  // heads per warp
  const long warps = (long)T * ((Hq + Hkv + hpw - 1) / hpw);
  const int blocks = (int)((warps + 7) / 8);
  auto* q = static_cast<uint16_t*>(qkv);
  auto* qn = static_cast<const __nv_bfloat16*>(q_norm);
  auto* kn = static_cast<const __nv_bfloat16*>(k_norm);
  auto* kc = static_cast<uint16_t*>(kcache);
  switch (hd) {
    case 64:
      return fk_launch(rope_qkv_kernel<1>, blocks, 256, 0, st, q, ldqkv, T, S, pos0, Hq, Hkv, rope, qk_norm, qn,
                       kn, eps, kc, cap, f16);
    case 128:
      return fk_launch(rope_qkv_kernel<2>, blocks, 256, 0, st, q, ldqkv, T, S, pos0, Hq, Hkv, rope, qk_norm, qn,
                       kn, eps, kc, cap, f16);
    case 256:
      return fk_launch(rope_qkv_kernel<4>, blocks, 256, 0, st, q, ldqkv, T, S, pos0, Hq, Hkv, rope, qk_norm, qn,
                       kn, eps, kc, cap, f16);
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_argmax(const float* z, int R, int V, int ldz, int32_t* out, cudaStream_t st, int32_t* out2,
                          void* scratch, float* margin) {
  if (R == 0) return cudaSuccess;
  if (scratch && R <= kArgmaxMaxSplitRows && (ldz & 3) == 0) {
    constexpr int n = kArgmaxMaxSplitRows * kArgmaxSplits;
    float* pm = static_cast<float*>(scratch);
    int* pi = reinterpret_cast<int*>(pm + n);
    float* pm2 = reinterpret_cast<float*>(pi + n);
    unsigned* cnt = reinterpret_cast<unsigned*>(pm2 + n);
    return fk_launch(argmax_split_kernel, dim3(kArgmaxSplits, R), 256, 0, st, z, V, ldz, out, out2, margin, pm, pi,
                     pm2, cnt);
  }
  return fk_launch(argmax_kernel, R, 256, 0, st, z, R, V, ldz, out, out2, margin);
}

cudaError_t launch_bf16_to_f16(const void* src, void* dst, size_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  if (n % 8 || (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) return cudaErrorInvalidValue;
  const size_t n8 = n / 8;
  const int blocks = (int)std::min<size_t>((n8 + 255) / 256, 4096);
  bf16_to_f16_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), n8);
  return cudaGetLastError();
}

cudaError_t launch_set_int(int* p, int value, cudaStream_t st) {
  set_int_kernel<<<1, 1, 0, st>>>(p, value);
  return cudaGetLastError();
}

cudaError_t launch_inc_int(int* p, cudaStream_t st) {
  return fk_launch(inc_int_kernel, 1, 1, 0, st, p);
}

cudaError_t launch_gather_last_rows(const void* src, int ld, int S, int H, int B, void* dst, cudaStream_t st) {
  if (B == 0) return cudaSuccess;
  gather_last_rows_kernel<<<B, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(src), ld, S, H, B,
                                             static_cast<__nv_bfloat16*>(dst));
  return cudaGetLastError();
}

}  // namespace fk
