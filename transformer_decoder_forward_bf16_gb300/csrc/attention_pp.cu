// Causal GQA flash attention for prefill with two query tiles per CTA
// ("N7 · model/forward-parity", Thm 1: causal multi-head/GQA attention;
// Thm 2 and "pegainfer #878": sliding-window local layers), head_dim 64/128.
//
// One CTA per (256 queries, head, sequence), one CTA per SM; key blocks of 128
// positions. The two 128-query tiles take turns on the tensor core: while one
// softmax warpgroup turns its scores into probabilities, the tensor core runs
// the other tile's products, so neither waits for the other's exponentials.
//   warp 0     TMA producers: lane 0 streams both query tiles once and the K
//              blocks (two 64-row boxes each, so a block may straddle the
//              wrap of a sliding-window ring), lane 1 the Vᵀ blocks; 2-deep
//              rings, 128-byte swizzle, K-major.
//   warp 1     TMEM allocator and single-thread MMA issuer. TMEM: S/P of
//              tile i at columns 128 i, O of tile i at 256 + HD i. Order per
//              block j: O0 += P0(j) V_j, S0(j+1) = Q0 K_{j+1}ᵀ, O1 += P1(j) V_j,
//              S1(j+1) = Q1 K_{j+1}ᵀ. A tile's next S is issued after its PV,
//              so the tensor core reads P_i(j) before S_i(j+1) overwrites it,
//              and the completion of S_i(j+1) implies PV_i(j) is done.
//   warps 2-9  softmax of tile 0, warps 10-17 of tile 1: two warps per TMEM
//              lane quarter (32 query rows, TMEM lane = row), one per 64-key
//              half of the block. The running max m (exp2 domain) is raised
//              lazily, only when a row's maximum grows by more than 2^8, so
//              each warp first forms P = exp2(S - m) against the current m in
//              one pipelined pass over its 64 score columns (mask: causal,
//              window, sequence end), keeping P packed to 16 bits in
//              registers, and only then exchanges its row maxima with the
//              partner warp through shared memory. If some row's maximum
//              outgrew m (and on a row's first visible block) both warps
//              recompute P from the scores, still intact in TMEM, against
//              the new m and rescale their half of the rows' O (idle: the S
//              completion implies the previous PV). P goes to the first 32 of
//              the half's own 64 score columns; at the end the output O / l.
// q, K, Vᵀ and P are bf16, or all IEEE f16 (F16); the output bf16 or f16.
// Every mbarrier wait is bounded (FK_DEVERR_PIPE_TIMEOUT on expiry); every
// tcgen05.ld/st is executed by whole warps (decisions that touch TMEM are
// taken warp-wide).
#include <algorithm>
#include <type_traits>

#include "fk_common.cuh"
#include "fk_internal.h"

namespace fk {

namespace {

constexpr int kSoftmaxWarps = 8;  // per query tile: two warps per TMEM lane quarter, one per half of the keys
constexpr int kPPThreads = 64 + 2 * 32 * kSoftmaxWarps;
constexpr int BQ = 128, BKV = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyRescale = 8.0f;  // log2 units

template <int HD>
struct PPCfg {
  static constexpr int Q_BYTES = BQ * HD * 2;   // one query tile: HD/64 column blocks of [128 rows][128 B]
  static constexpr int K_BYTES = BKV * HD * 2;  // HD/64 column blocks of [128 keys][128 B]
  static constexpr int V_BYTES = HD * BKV * 2;  // 2 key halves of [HD rows][64 keys x 2 B]
  static constexpr int STAGES = 2;
  // tiles, then 256 bytes for 16 barriers and two words; the dynamic window
  // starts 1024-byte aligned (checked on entry)
  // tiles, 4 KB of row partials exchanged between the two warps of a row
  // (max, then sum; [tile][key half][row] floats), 256 bytes of barriers
  static constexpr int XCHG_BYTES = 2 * 2 * BQ * 4 * 2;
  static constexpr int SMEM = 2 * Q_BYTES + STAGES * (K_BYTES + V_BYTES) + XCHG_BYTES + 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = 2 * BKV;
};

// 16 consecutive fp32 columns of this thread's TMEM lane, without the wait:
// the registers may be read only after tmem_wait_ld16 on the same array
FK_DEVICE void tmem_ld16_async(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// wait for the outstanding TMEM loads; r is passed through so that no use of
// the loaded registers can be scheduled before the wait
FK_DEVICE void tmem_wait_ld16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (32x32b shape, .x16), then a wait
FK_DEVICE void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

FK_DEVICE void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
FK_DEVICE void tmem_st_wait_pp() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] · B[smem]ᵀ (A operand read from TMEM)
FK_DEVICE void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// max(a, b, c) in one instruction
FK_DEVICE float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

FK_DEVICE float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Key-block range [lo, hi] of query tile i (empty: lo > hi).
struct TileRange {
  int lo, hi;
  int qp_lo, qp_hi;  // first and last query position of the tile
};

FK_DEVICE TileRange tile_range(int i, int q_lo, int S, int pos0, int window) {
  TileRange t;
  const int t_lo = q_lo + BQ * i;
  if (t_lo >= S) {
    t.lo = 1;
    t.hi = 0;
    t.qp_lo = t.qp_hi = 0;
    return t;
  }
  t.qp_lo = pos0 + t_lo;
  t.qp_hi = pos0 + min(S, t_lo + BQ) - 1;
  const int k_lo = window > 0 ? max(0, t.qp_lo - window + 1) : 0;
  t.lo = k_lo / BKV;
  t.hi = t.qp_hi / BKV;
  return t;
}

template <int HD, bool F16>
__global__ void __launch_bounds__(kPPThreads, 1)
    attn_pp_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, int S, int pos0, int Hq, int Hkv, int cap, int window,
                   float scale_log2, uint16_t* __restrict__ out, unsigned* dev_err, int out_f16) {
  using C = PPCfg<HD>;
  constexpr int io_f16 = F16 ? 1 : 0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0 && dev_err) atomicOr(dev_err, FK_DEVERR_PIPE_TIMEOUT);
    return;
  }
  uint8_t* sQ = smem_raw;                     // [2 tiles][Q_BYTES]
  uint8_t* sK = sQ + 2 * C::Q_BYTES;          // [STAGES][K_BYTES]
  uint8_t* sV = sK + C::STAGES * C::K_BYTES;  // [STAGES][V_BYTES]
  float* xmax = reinterpret_cast<float*>(sV + C::STAGES * C::V_BYTES);  // [tile][half][row]
  float* xsum = xmax + 2 * 2 * BQ;                                       // [tile][half][row]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + C::STAGES * C::V_BYTES + C::XCHG_BYTES);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;    // [stage]
  uint64_t* k_empty = bars + 3;   // [stage]
  uint64_t* v_full = bars + 5;    // [stage]
  uint64_t* v_empty = bars + 7;   // [stage]
  uint64_t* s_full = bars + 9;    // [tile]
  uint64_t* p_full = bars + 11;   // [tile]
  uint64_t* pv_done = bars + 13;  // [tile]
  uint64_t* mma_done = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hb = blockIdx.x;  // (head, sequence), fastest: the first wave covers every head
  const int h = hb % Hq, b = hb / Hq;
  const int nsb = (S + 2 * BQ - 1) / (2 * BQ);
  const int q_lo = (nsb - 1 - (int)blockIdx.y) * 2 * BQ;  // longest (latest) query blocks first
  const int g = h / (Hq / Hkv);
  const int kv_len = pos0 + S;
  const TileRange tr0 = tile_range(0, q_lo, S, pos0, window);
  const TileRange tr1 = tile_range(1, q_lo, S, pos0, window);
  const int j_begin = tr0.lo;
  const int j_end = tr1.hi >= tr1.lo ? max(tr0.hi, tr1.hi) : tr0.hi;
  const int nblk = j_end - j_begin + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 32 * kSoftmaxWarps);
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
      // ---------------- TMA producers: lane 0 Q and K, lane 1 Vᵀ ----------------
      const bool is_k = lane == 0;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      if (is_k) {
        mbar_arrive_expect_tx(q_full, 2 * C::Q_BYTES);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int blk = 0; blk < HD / 64; ++blk)
            tma_load_2d(&tmQ, q_full, sQ + i * C::Q_BYTES + blk * BQ * 128, h * HD + blk * 64, b * S + q_lo + BQ * i);
      }
      const int krow = (b * Hkv + g) * cap;
      const int vrow = (b * Hkv + g) * HD;
      int issued[2] = {0, 0};
      for (int n = 0; n < nblk; ++n) {
        const int st = n & 1;
        if (!mbar_wait(&empty[st], ((n >> 1) & 1) ^ 1, abort_flag, dev_err)) break;
        const int p0 = (j_begin + n) * BKV;  // first key position of the block
        if (is_k) {
          mbar_arrive_expect_tx(&full[st], C::K_BYTES);
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int blk = 0; blk < HD / 64; ++blk)
              tma_load_2d(&tmK, &full[st], sK + st * C::K_BYTES + blk * BKV * 128 + half * 64 * 128, blk * 64,
                          krow + (p0 + 64 * half) % cap);
        } else {
          mbar_arrive_expect_tx(&full[st], C::V_BYTES);
#pragma unroll
          for (int half = 0; half < 2; ++half)
            tma_load_2d(&tmV, &full[st], sV + st * C::V_BYTES + half * HD * 128, (p0 + 64 * half) % cap, vrow);
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
      auto in = [&](int i, int j) -> bool {
        const TileRange& t = i ? tr1 : tr0;
        return j >= t.lo && j <= t.hi;
      };
      auto issue_s = [&](int i, int n) {  // K block n already landed
        const int st = n & 1;
        const uint32_t d = tmem + (uint32_t)(i * BKV);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint64_t ad = smem_desc_sw128(sQ + i * C::Q_BYTES + (k >> 2) * BQ * 128) + 2 * (k & 3);
          const uint64_t bd = smem_desc_sw128(sK + st * C::K_BYTES + (k >> 2) * BKV * 128) + 2 * (k & 3);
          umma_bf16(d, ad, bd, idesc_s, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[i]);
      };
      int npv[2] = {0, 0};
      auto issue_pv = [&](int i, int n) -> bool {
        if (!mbar_wait(&p_full[i], npv[i] & 1, abort_flag, dev_err)) return false;
        tc_fence_after();
        const int st = n & 1;
#pragma unroll
        for (int k = 0; k < BKV / 16; ++k) {
          const uint64_t bd = smem_desc_sw128(sV + st * C::V_BYTES + (k >> 2) * HD * 128) + 2 * (k & 3);
          // P of keys 16k..16k+15: key half k/4 keeps its P pairs in the first
          // 32 of its 64 score columns
          umma_ts(tmem + C::O_COL + (uint32_t)(i * HD), tmem + (uint32_t)(i * BKV + 64 * (k >> 2) + 8 * (k & 3)), bd,
                  idesc_o, (npv[i] > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&pv_done[i]);
        ++npv[i];
        return true;
      };
      bool ok = mbar_wait(q_full, 0, abort_flag, dev_err) && mbar_wait(&k_full[0], 0, abort_flag, dev_err);
      if (ok) {
        tc_fence_after();
        if (in(0, j_begin)) issue_s(0, 0);
        if (in(1, j_begin)) issue_s(1, 0);
        umma_commit(&k_empty[0]);
      }
      for (int n = 0; n < nblk && ok; ++n) {
        const int j = j_begin + n, st = n & 1;
        const bool next = n + 1 < nblk;
        if (!mbar_wait(&v_full[st], (n >> 1) & 1, abort_flag, dev_err)) break;
        tc_fence_after();
        if (in(0, j) && !issue_pv(0, n)) break;
        if (next) {
          if (!mbar_wait(&k_full[(n + 1) & 1], ((n + 1) >> 1) & 1, abort_flag, dev_err)) break;
          tc_fence_after();
          if (in(0, j + 1)) issue_s(0, n + 1);
        }
        if (in(1, j) && !issue_pv(1, n)) break;
        umma_commit(&v_empty[st]);
        if (next) {
          if (in(1, j + 1)) issue_s(1, n + 1);
          umma_commit(&k_empty[(n + 1) & 1]);
        }
      }
      umma_commit(mma_done);
      const uint32_t a = smem_u32(mma_done);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else {
    // ---------------- softmax: warps 2-9 tile 0, warps 10-17 tile 1 ----------------
    // warp k of a tile takes TMEM lane quarter (warp % 4), i.e. 32 query rows,
    // and key half k / 4 (64 of the block's 128 columns); the two warps of a
    // row combine their row maxima through shared memory (a named barrier of
    // those two warps per block) and keep partial row sums, added at the end
    const int i = (warp - 2) / kSoftmaxWarps;
    const int kw = (warp - 2) % kSoftmaxWarps;
    const int half = kw >> 2;
    const TileRange tr = i ? tr1 : tr0;
    const int q4 = warp & 3;       // TMEM lane quarter this warp may access
    const int r = q4 * 32 + lane;  // query row of this thread within the tile = TMEM lane
    const int qp = tr.qp_lo + r;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t s_col = (uint32_t)(i * BKV) + half * 64;                     // this warp's 64 score columns
    const uint32_t p_col = s_col;  // its 32 columns of P pairs: the first half of its own score columns
    const uint32_t o_col = C::O_COL + (uint32_t)(i * HD) + half * (HD / 2);   // its half of O
    float* my_max = xmax + (i * 2 + half) * BQ;
    const float* other_max = xmax + (i * 2 + (half ^ 1)) * BQ;
    // named barrier of the two warps that share these 32 rows (ids 1..8)
    const int bar_id = 1 + i * 4 + q4;
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory"); };
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    int ns = 0;
    for (int j = tr.lo; j <= tr.hi; ++j, ++ns) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[i], ns & 1, abort_flag, dev_err))) ok = false;
      // both warps of every row take the same path (the barrier below is per tile)
      if (!ok) break;
      tc_fence_after();
      const int key0 = j * BKV + half * 64;  // first key of this warp's columns
      const bool edge = (j * BKV + BKV - 1 > tr.qp_lo) || (j * BKV + BKV > kv_len) ||
                        (window > 0 && tr.qp_hi - j * BKV >= window);
      auto visible = [&](int k) { return k <= qp && k < kv_len && (window == 0 || qp - k < window); };
      // P against the current m (0 where masked), 16-bit pairs in registers;
      // the row maximum of the visible raw scores on the way. Four 16-column
      // TMEM loads, each issued while the previous one is turned into P.
      // (With no m yet the values are discarded below.)
      uint32_t pk[32];
      float mx = -INFINITY, l0 = 0.f, l1 = 0.f;
      // the masked and unmasked versions are separate loops (edge is warp-uniform)
      auto p_pass_as = [&](auto edge_c, auto want_max_c, float neg_m) {
        constexpr bool kEdge = decltype(edge_c)::value, kMax = decltype(want_max_c)::value;
        uint32_t sa[16], sb[16];
        tmem_ld16_async(lane_base + s_col, sa);
        tmem_wait_ld16(sa);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t* cur = (c & 1) ? sb : sa;
          uint32_t* nxt = (c & 1) ? sa : sb;
          if (c + 1 < 4) tmem_ld16_async(lane_base + s_col + (c + 1) * 16, nxt);
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float x0 = __uint_as_float(cur[e]), x1 = __uint_as_float(cur[e + 1]);
            float p0 = ex2(fmaf(x0, scale_log2, neg_m));
            float p1 = ex2(fmaf(x1, scale_log2, neg_m));
            if constexpr (kEdge) {
              const bool v0 = visible(key0 + c * 16 + e), v1 = visible(key0 + c * 16 + e + 1);
              if constexpr (kMax) {
                if (v0) mx = fmaxf(mx, x0);
                if (v1) mx = fmaxf(mx, x1);
              }
              if (!v0) p0 = 0.f;
              if (!v1) p1 = 0.f;
            } else if constexpr (kMax) {
              mx = max3(mx, x0, x1);
            }
            l0 += p0;
            l1 += p1;
            pk[(c * 16 + e) >> 1] = pack_16x2(p0, p1, io_f16);
          }
          if (c + 1 < 4) tmem_wait_ld16(nxt);
        }
      };
      using kT = std::true_type;
      using kF = std::false_type;
      auto p_pass = [&](float neg_m, auto want_max_c) {
        if (edge) p_pass_as(kT{}, want_max_c, neg_m);
        else p_pass_as(kF{}, want_max_c, neg_m);
      };
      if (ns == 0) {
        // the tile's first block: no row has an m yet, so P is formed only
        // after the exchange below; this pass takes the row maxima alone
        auto max_pass = [&](auto edge_c) {
          constexpr bool kEdge = decltype(edge_c)::value;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t sv[16];
            tmem_ld16(lane_base + s_col + c * 16, sv);
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const float x0 = __uint_as_float(sv[e]), x1 = __uint_as_float(sv[e + 1]);
              if constexpr (kEdge) {
                if (visible(key0 + c * 16 + e)) mx = fmaxf(mx, x0);
                if (visible(key0 + c * 16 + e + 1)) mx = fmaxf(mx, x1);
              } else {
                mx = max3(mx, x0, x1);
              }
            }
          }
        };
        if (edge) max_pass(kT{});
        else max_pass(kF{});
      } else {
        p_pass(m == -INFINITY ? 0.f : -m, kT{});
      }
      my_max[r] = mx;
      // both warps of the row have published their maxima
      pair_sync();
      // scale_log2 > 0: the maximum of the scaled scores is the scaled maximum
      const float m_new = fmaxf(m, fmaxf(mx, other_max[r]) * scale_log2);
      const bool first = m == -INFINITY;  // nothing accumulated in this row yet (O and l are 0)
      const bool raise = first || m_new > m + kLazyRescale;
      // the two warps of these rows see the same maxima: they take the same path
      if (__any_sync(0xffffffffu, raise)) {
        const float m_use = raise ? m_new : m;
        if (__any_sync(0xffffffffu, raise && !first)) {
          const float corr = raise && !first ? ex2(m - m_use) : 1.f;
          l *= corr;
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {  // this warp's half of the row's O, 16 columns at a time
            uint32_t o[16];
            tmem_ld16(lane_base + o_col + c * 16, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
            tmem_st16(lane_base + o_col + c * 16, o);
          }
          tmem_st_wait_pp();
        }
        // m_use is -inf only if no key of this or an earlier block is visible
        // to the row: then every P is masked to 0 (an edge block)
        m = m_use;
        l0 = l1 = 0.f;
        p_pass(-m_use, kF{});
      }
      l += l0 + l1;
      tmem_st16(lane_base + p_col, pk);
      tmem_st16(lane_base + p_col + 16, pk + 16);
      tmem_st_wait_pp();
      tc_fence_before();
      mbar_arrive(&p_full[i]);
      // the maxima are read again only after the next block's barrier
    }
    // epilogue: O / l -> 16 bits, each warp its half of the columns
    if (ns > 0) {
      xsum[(i * 2 + half) * BQ + r] = l;
      pair_sync();
      const float l_row = l + xsum[(i * 2 + (half ^ 1)) * BQ + r];
      const bool have = __all_sync(0xffffffffu, ok && mbar_wait(&pv_done[i], (ns - 1) & 1, abort_flag, dev_err));
      tc_fence_after();
      const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
      const int qi = q_lo + BQ * i + r;
      uint16_t* orow = out + ((size_t)b * S + qi) * ((size_t)Hq * HD) + (size_t)h * HD + half * (HD / 2);
#pragma unroll 1
      for (int c = 0; c < HD / 64; ++c) {
        float v[32];
        tmem_ld32(lane_base + o_col + c * 32, v);
        if (have && qi < S) {
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            *reinterpret_cast<uint4*>(orow + c * 32 + e) = make_uint4(
                pack_16x2(v[e] * inv, v[e + 1] * inv, out_f16), pack_16x2(v[e + 2] * inv, v[e + 3] * inv, out_f16),
                pack_16x2(v[e + 4] * inv, v[e + 5] * inv, out_f16), pack_16x2(v[e + 6] * inv, v[e + 7] * inv, out_f16));
        }
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
fk_status launch_pp(const void* q, int ldq, const void* kc, const void* vc, int cap, int B, int S, int pos0, int Hq,
                    int Hkv, int window, float scale, void* o, unsigned* dev_err, cudaStream_t st, int io_f16,
                    int out_f16) {
  using C = PPCfg<HD>;
  static DeviceOnce once;
  const cudaError_t attr = once.run([] {
    cudaError_t e = cudaFuncSetAttribute(attn_pp_kernel<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_pp_kernel<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    return e;
  });
  if (attr != cudaSuccess) return cuda_fail(attr, "cudaFuncSetAttribute(attn_pp)");
  CUtensorMap tQ, tK, tV;
  fk_status s = make_tmap_bf16(&tQ, q, (int64_t)B * S, ldq, ldq, BQ);
  if (s == FK_OK) s = make_tmap_bf16(&tK, kc, (int64_t)B * Hkv * cap, HD, HD, 64);
  if (s == FK_OK) s = make_tmap_bf16(&tV, vc, (int64_t)B * Hkv * HD, cap, cap, HD);
  if (s != FK_OK) return s;
  const int nsb = (S + 2 * BQ - 1) / (2 * BQ);
  auto kernel = io_f16 ? attn_pp_kernel<HD, true> : attn_pp_kernel<HD, false>;
  kernel<<<dim3(Hq * B, nsb), kPPThreads, C::SMEM, st>>>(tQ, tK, tV, S, pos0, Hq, Hkv, cap, window, scale * kLog2e,
                                                         static_cast<uint16_t*>(o), dev_err, out_f16);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "attn_pp_kernel launch");
  return FK_OK;
}

}  // namespace

fk_status attention_prefill_pp(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B, int S,
                               int pos0, int Hq, int Hkv, int hd, int window, float scale, void* o,
                               unsigned* dev_err, cudaStream_t st, int io_f16, int out_f16) {
  if (hd == 64)
    return launch_pp<64>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, dev_err, st, io_f16,
                         out_f16);
  if (hd == 128)
    return launch_pp<128>(q, ldq, kcache, vcache, cap, B, S, pos0, Hq, Hkv, window, scale, o, dev_err, st, io_f16,
                          out_f16);
  return fail(FK_ERR_INVALID_ARG, "two-tile prefill attention: head_dim 64 or 128");
}

}  // namespace fk
