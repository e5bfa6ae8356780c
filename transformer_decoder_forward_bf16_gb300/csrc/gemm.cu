// bf16 GEMM on the 5th-generation tensor cores: out = epilogue(A · Bᵀ).
//
// "N9 · metalgemm", Theorem 1 defines the operation (Y = X·Wᵀ with float
// accumulation; the Apple MPS lane there is prior art, not the design).
//
// Design (sm_103a):
//   * persistent kernel, one CTA per SM, 128 x BN output tiles walked in
//     groups of 16 M-blocks so that a wave of CTAs shares A and B tiles in L2
//     (BN = 256, with 256-row tiles once there are two per SM; 128; or 64
//     for few rows, so that more CTAs stream the weights);
//   * warp 0: TMA producer (128-byte swizzled 128x64 A boxes and 64x64 B
//     boxes into a STAGES-deep ring, completion on mbarriers);
//   * warp 1: TMEM allocator and single-thread tcgen05.mma issuer
//     (M=128, N=BN, K=16 per instruction, fp32 accumulators in TMEM, two
//     accumulator buffers so the epilogue of tile i overlaps the MMAs of
//     tile i+1);
//   * warps 2-5: epilogue, tcgen05.ld 32x32b (one TMEM lane = one output
//     row per thread) then a fused store: bf16, fp32 (+softcap), fp32
//     residual add, or the gated activation act(gate)*up of the FFN.
//   * the weight operand may be up to three matrices stacked along N (Q|K|V
//     without a repacked copy) or a gate/up pair interleaved per tile;
//   * fp32 outputs (plain, softcapped or residual-added) are staged per
//     32 x 32 block in 128-byte-swizzled shared memory and written by TMA
//     bulk tensor stores (whole 128-byte lines, no per-row scatter from the
//     epilogue threads), except blocks that cross the end of the rows (of
//     their group) or of the columns; a residual add in place (res == out)
//     stores each whole block by a TMA reduce-add, so the residual is never
//     loaded into the SM and the epilogue does not wait on its latency;
//   * grouped mode (the experts of a MoE layer): A holds the rows of every
//     group back to back, group g at rows [off[g], off[g+1]) (offsets read
//     from device memory at kernel start), and each group's rows multiply
//     that group's matrix of a stacked operand. Tiles never span two groups:
//     each group's rows are cut into 128-row blocks of their own, and rows
//     past the group's end are computed but not stored.
#include <algorithm>

#include "fk_common.cuh"
#include "fk_internal.h"

namespace fk {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kEpiWarps = 8;  // two warps per TMEM lane quarter, each taking half the columns
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int A_BYTES = BM * BK * 2;  // 16 KiB

struct GemmArgs {
  int M, K, n_virtual;  // n_virtual: rows of the (virtual) B operand
  int nseg, glu;
  int seg_start[4];
  int seg_rows[3];
  int n_out;
  int epi, act;
  void* out;
  int ldo;
  const float* res;
  int ldr;
  float softcap;
  unsigned* dev_err;
  int ab_f16;   // A and B are IEEE f16 (else bf16)
  int out_f16;  // 16-bit outputs stored as f16 (else bf16)
  int res_inplace;  // EPI_ADD_F32 with res == out: whole staged blocks are added by TMA reductions
  const int* group_off;  // grouped mode: groups + 1 row offsets into A
  int groups;
  int group_rows;        // B rows of one group in each map
};

// MT = 128-row sub-tiles per CTA tile. MT == 2 makes a 256 x BN tile: two
// M=128 accumulators share every B tile, a third fewer L2->SM bytes per FLOP
// than MT == 1, at the price of a single accumulator set (the epilogue of a
// tile no longer overlaps the next tile's MMAs).
// SO: fp32 output blocks staged in shared memory (OUT_SLOTS 4 KiB 32 x 32
// blocks per epilogue warp) and stored by TMA; one operand stage fewer to
// make room (256-row tiles keep their three stages and one slot per warp).
// AR: few-row mode (a call of at most AR rows, MT == 1). The TMA writes only
// the AR valid rows of each A stage, and a stage's A slot is only that big:
// the MMA still reads 128 rows from the slot's start, the rows past AR being
// whatever the next slots hold. Those rows' outputs are never stored, and each
// output row depends on its own A row alone, so the stored rows are the same
// bits as with whole A tiles. The shared memory saved deepens the weight ring.
constexpr int kSmemBudget = 232448;  // dynamic shared memory of one CTA (227 KiB)
template <int BN, int MT = 1, bool SO = false, int AR = 0>
struct Cfg {
  static_assert(AR == 0 || MT == 1, "few-row mode takes 128-row tiles");
  static constexpr int A_STAGE = AR ? (AR * BK * 2 + 1023) / 1024 * 1024 : MT * A_BYTES;  // slot stride
  static constexpr int A_TX = AR ? AR * BK * 2 : MT * A_BYTES;                          // bytes loaded
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int OUT_SLOTS = MT == 2 ? 1 : 2;
  static constexpr int OUT_BYTES = SO ? kEpiWarps * OUT_SLOTS * 4096 : 0;
  // mbarriers (two per stage and five), TMEM address, abort flag: the deep
  // rings of few-row mode need more than 256 bytes
  static constexpr int BAR_BYTES = AR ? 512 : 256;
  static constexpr int AR_STAGES = (kSmemBudget - OUT_BYTES - 1024 - BAR_BYTES) / (A_STAGE + B_BYTES);
  static constexpr int STAGES =
      AR ? (AR_STAGES < 24 ? AR_STAGES : 24)
         : (MT == 2 ? 3 : (BN == 64 ? (SO ? 6 : 8) : (SO ? ((BN == 256) ? 3 : 4) : ((BN == 256) ? 4 : 6))));
  static constexpr int SMEM = STAGES * (A_STAGE + B_BYTES) + OUT_BYTES + 1024 /*align*/ + BAR_BYTES;
  static_assert((2 * STAGES + 5) * 8 + 8 <= BAR_BYTES, "barrier area");
  static_assert(SMEM <= kSmemBudget, "shared memory");
  static_assert(AR == 0 || STAGES * B_BYTES >= A_BYTES, "a slot's 128-row read stays inside the operand ring");
  static constexpr int NACC = MT == 1 ? 2 : 1;  // accumulator sets (double buffer when they fit)
  static constexpr uint32_t TMEM_COLS = NACC * MT * BN;
};

FK_DEVICE void tile_coords(int t, int m_blocks, int n_blocks, int& mb, int& nb) {
  constexpr int G = 16;
  const int group = t / (G * n_blocks);
  const int first_m = group * G;
  const int gsize = min(m_blocks - first_m, G);
  const int r = t - group * G * n_blocks;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

// SiLU g * sigmoid(g) with the hardware 2^x (ex2.approx) and fast division:
// both far more accurate than the bf16 rounding of the product that follows.
FK_DEVICE float act_silu(float g) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-g * 1.4426950408889634f));
  return __fdividef(g, 1.0f + e);
}
FK_DEVICE float act_gelu_tanh(float g) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * g * (1.0f + tanhf(k0 * (g + 0.044715f * g * g * g)));
}

// Source of the i-th 64-row box of B for output block nb (gbase: first row
// of the tile's group in every map, 0 outside grouped mode).
template <int BN>
FK_DEVICE void b_box_source(const GemmArgs& a, int nb, int i, int gbase, int& map, int& row, bool& valid) {
  if (a.glu) {
    constexpr int half = BN >= 128 ? BN / 128 : 1;  // boxes per half tile (gated tiles have BN >= 128)
    map = (i < half) ? 0 : 1;
    row = nb * (BN / 2) + (i % half) * 64;
    valid = row < a.seg_rows[map];
  } else {
    const int v = nb * BN + i * 64;
    map = 0;
    if (a.nseg > 1 && v >= a.seg_start[1]) map = 1;
    if (a.nseg > 2 && v >= a.seg_start[2]) map = 2;
    row = v - a.seg_start[map];
    valid = v < a.n_virtual;
  }
  row += gbase;
}

// A rows of a tile: [row0, row_end) are stored; g is the tile's group.
struct TileRows {
  int row0, row_end, g;
};
// Grouped mode: m-block mb (of TM rows) of the tile order is block
// mb - mstart[g] of the group g with mstart[g] <= mb < mstart[g+1] (empty
// groups have no blocks). mstart is 16-bit: at most 65535 m-blocks.
FK_DEVICE TileRows grouped_rows(const int* goff, const unsigned short* mstart, int groups, int mb, int TM) {
  int lo = 0, hi = groups;  // mstart[lo] <= mb < mstart[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int)mstart[mid] <= mb) lo = mid;
    else hi = mid;
  }
  return TileRows{goff[lo] + (mb - (int)mstart[lo]) * TM, goff[lo + 1], lo};
}

template <int BN, int MT, bool GROUPED, bool SO, int AR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmOut, const GemmArgs args) {
  using C = Cfg<BN, MT, SO, AR>;
  constexpr int TM = BM * MT;  // rows per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_STAGE;
  uint8_t* sOut = sB + C::STAGES * C::B_BYTES;  // SO: staged output blocks (1024-byte aligned)
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + C::OUT_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int m_blocks = (args.M + TM - 1) / TM;
  const int n_blocks = args.glu ? (args.n_out + BN / 2 - 1) / (BN / 2) : (args.n_virtual + BN - 1) / BN;
  const int nk = (args.K + BK - 1) / BK;

  // grouped mode: the group offsets and the first m-block of every group
  __shared__ int s_goff[GROUPED ? kMoeMaxExperts + 1 : 1];
  __shared__ unsigned short s_mstart[GROUPED ? kMoeMaxExperts + 1 : 1];
  if constexpr (GROUPED) {
    for (int i = threadIdx.x; i <= args.groups; i += blockDim.x) s_goff[i] = args.group_off[i];
    __syncthreads();
    if (warp == 2) {  // exclusive prefix of ceil(rows / TM) over the groups
      int carry = 0;
      for (int g0 = 0; g0 < args.groups; g0 += 32) {
        const int g = g0 + lane;
        int v = g < args.groups ? (s_goff[g + 1] - s_goff[g] + TM - 1) / TM : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += n;
        }
        if (g < args.groups) s_mstart[g + 1] = (unsigned short)(carry + v);
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) s_mstart[0] = 0;
    }
  }
  auto rows_of = [&](int mb) -> TileRows {
    if constexpr (GROUPED) return grouped_rows(s_goff, s_mstart, args.groups, mb, TM);
    return TileRows{mb * TM, args.M, 0};
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 32 * kEpiWarps);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    if (args.nseg > 1) tma_prefetch_desc(&tmB1);
    if (args.nseg > 2) tma_prefetch_desc(&tmB2);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if constexpr (GROUPED) m_blocks = s_mstart[args.groups];
  const int tiles = m_blocks * n_blocks;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      const CUtensorMap* maps[3] = {&tmB0, &tmB1, &tmB2};
      int fills[C::STAGES];
      for (int s = 0; s < C::STAGES; ++s) fills[s] = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, m_blocks, n_blocks, mb, nb);
        const TileRows tr = rows_of(mb);
        const int gbase = tr.g * args.group_rows;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, args.dev_err)) {
            ok = false;
            break;
          }
          uint32_t bytes = C::A_TX;
#pragma unroll
          for (int i = 0; i < BN / 64; ++i) {
            int map, row;
            bool valid;
            b_box_source<BN>(args, nb, i, gbase, map, row, valid);
            if (valid) bytes += 64 * BK * 2;
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
          for (int sub = 0; sub < MT; ++sub)
            tma_load_2d(&tmA, &full[stage], sA + stage * C::A_STAGE + sub * A_BYTES, kb * BK, tr.row0 + sub * BM);
          // (few-row mode: the map's box is AR rows high, so this writes A_TX bytes)
#pragma unroll
          for (int i = 0; i < BN / 64; ++i) {
            int map, row;
            bool valid;
            b_box_source<BN>(args, nb, i, gbase, map, row, valid);
            if (valid) tma_load_2d(maps[map], &full[stage], sB + stage * C::B_BYTES + i * 64 * BK * 2, kb * BK, row);
          }
          ++fills[stage];
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // let every copy this thread issued land before the CTA unwinds
        for (int s = 0; s < C::STAGES; ++s) {
          if (fills[s] == 0) continue;
          const uint32_t a = smem_u32(&full[s]);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(a, (fills[s] - 1) & 1) && globaltimer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = idesc_16b_f32(BM, BN, args.ab_f16);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++local) {
        const int acc = local % C::NACC;
        const uint32_t aphase = (local / C::NACC) & 1;
        if (!mbar_wait(&tempty[acc], aphase ^ 1, abort_flag, args.dev_err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * MT * BN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, args.dev_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = smem_desc_sw128(sB + stage * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
#pragma unroll
            for (int sub = 0; sub < MT; ++sub) {
              const uint64_t ad = smem_desc_sw128(sA + stage * C::A_STAGE + sub * A_BYTES);
              umma_bf16(d + sub * BN, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
            }
          umma_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) umma_commit(&tfull[acc]);
      }
      // every MMA issued by this thread has completed once mma_done fires
      // (a grouped CTA may have had no tile and issued none)
      if (local > 0) {
        umma_commit(mma_done);
        const uint32_t a = smem_u32(mma_done);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(a, 0) && globaltimer_ns() - t0 < 100000000ull) {
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which half of the tile's columns it stores
    int oslot = 0;                     // SO: which of the warp's two staging blocks is next
    int local = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++local) {
      int mb, nb;
      tile_coords(t, m_blocks, n_blocks, mb, nb);
      const TileRows tr = rows_of(mb);
      const int acc = local % C::NACC;
      const uint32_t aphase = (local / C::NACC) & 1;
      // warp-uniform: the tcgen05.ld below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], aphase, abort_flag, args.dev_err))) break;
      tc_fence_after();
#pragma unroll 1
      for (int sub = 0; sub < MT; ++sub) {
      const int row = tr.row0 + sub * BM + q * 32 + lane;
      const bool row_ok = row < tr.row_end;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (acc * MT + sub) * BN;
      float v[32];
      if constexpr (SO && BN == 256) {
        // 16-bit outputs: this warp's 32 rows x 64-column boxes (two for a
        // plain output, one for the gated one), staged and stored by TMA
        if (args.epi == EPI_BF16 || args.epi == EPI_GLU_BF16) {
          const bool glu = args.epi == EPI_GLU_BF16;
          const int r0 = tr.row0 + sub * BM + q * 32;
          const int f = args.out_f16;
#pragma unroll 1
          for (int bx = 0; bx < (glu ? 1 : 2); ++bx) {
            const int ocol0 = glu ? nb * (BN / 2) + half * 64 : nb * BN + half * (BN / 2) + bx * 64;
            uint32_t pk[32];
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {  // two 32-column TMEM loads per box
              float x[32];
              if (glu) {
                float g[32];
                tmem_ld32(taddr + (half * 2 + hc) * 32, g);
                tmem_ld32(taddr + BN / 2 + (half * 2 + hc) * 32, x);
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = (args.act ? act_gelu_tanh(g[j]) : act_silu(g[j])) * x[j];
              } else {
                tmem_ld32(taddr + half * (BN / 2) + bx * 64 + hc * 32, x);
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) pk[hc * 16 + j] = pack_16x2(x[2 * j], x[2 * j + 1], f);
            }
            if (r0 + 32 <= tr.row_end && ocol0 + 64 <= args.n_out) {  // warp-uniform: a whole box
              uint8_t* buf = sOut + ((warp - 2) * C::OUT_SLOTS + oslot) * 4096;
              if (lane == 0) bulk_wait_group_read<C::OUT_SLOTS - 1>();
              __syncwarp();
              // row `lane`: 16-byte chunk j at chunk position j ^ (row % 8) (128-byte swizzle)
#pragma unroll
              for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmOut, buf, ocol0, r0);
                bulk_commit_group();
              }
              oslot = (oslot + 1) % C::OUT_SLOTS;
            } else if (row_ok) {
              uint16_t* o = reinterpret_cast<uint16_t*>(args.out) + (size_t)row * args.ldo + ocol0;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                if (ocol0 + 2 * j < args.n_out) o[2 * j] = (uint16_t)(pk[j] & 0xFFFFu);
                if (ocol0 + 2 * j + 1 < args.n_out) o[2 * j + 1] = (uint16_t)(pk[j] >> 16);
              }
            }
          }
          continue;  // next sub-tile
        }
      }
      if (args.epi == EPI_GLU_BF16) {
        for (int c = half * (BN / 128); c < (half + 1) * (BN / 128); ++c) {
          float u[32];
          tmem_ld32(taddr + c * 32, v);
          tmem_ld32(taddr + BN / 2 + c * 32, u);
          const int col0 = nb * (BN / 2) + c * 32;
          if (!row_ok) continue;
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = (args.act ? act_gelu_tanh(v[j]) : act_silu(v[j])) * u[j];
          uint16_t* o = reinterpret_cast<uint16_t*>(args.out) + (size_t)row * args.ldo + col0;  // bf16 or f16
          if (col0 + 32 <= args.n_out) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              const int f = args.out_f16;
              uint4 pk = make_uint4(pack_16x2(v[j], v[j + 1], f), pack_16x2(v[j + 2], v[j + 3], f),
                                    pack_16x2(v[j + 4], v[j + 5], f), pack_16x2(v[j + 6], v[j + 7], f));
              *reinterpret_cast<uint4*>(o + j) = pk;
            }
          } else {
            for (int j = 0; j < 32 && col0 + j < args.n_out; ++j) store_16(o + j, v[j], args.out_f16);
          }
        }
      } else {
        for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
          const int col0 = nb * BN + c * 32;
          // in-place residual add of a whole staged block: the TMA reduction
          // adds it to the output, so the residual is never loaded here
          const bool red_blk = SO && args.res_inplace && tr.row0 + sub * BM + q * 32 + 32 <= tr.row_end &&
                               col0 + 32 <= args.n_out;  // warp-uniform
          // residual add: the chunk's residual loads go out before the TMEM load's wait
          float4 rv[8];
          const bool res_full = args.epi == EPI_ADD_F32 && !red_blk && row_ok && col0 + 32 <= args.n_out;
          if (res_full) {
            const float4* r4 = reinterpret_cast<const float4*>(args.res + (size_t)row * args.ldr + col0);
#pragma unroll
            for (int j = 0; j < 8; ++j) rv[j] = r4[j];
          }
          tmem_ld32(taddr + c * 32, v);
          if constexpr (SO) {
            // a whole 32 x 32 fp32 block inside the output: stage it, store it by TMA
            const int r0 = tr.row0 + sub * BM + q * 32;
            if (r0 + 32 <= tr.row_end && col0 + 32 <= args.n_out) {  // warp-uniform
              if (args.epi == EPI_ADD_F32 && !red_blk) {  // res_full holds for every row of the block
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  v[4 * j] += rv[j].x;
                  v[4 * j + 1] += rv[j].y;
                  v[4 * j + 2] += rv[j].z;
                  v[4 * j + 3] += rv[j].w;
                }
              } else if (args.softcap > 0.f) {
                const float c_ = args.softcap, inv = 1.0f / args.softcap;
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = c_ * tanhf(v[j] * inv);
              }
              uint8_t* buf = sOut + ((warp - 2) * C::OUT_SLOTS + oslot) * 4096;
              // the store issued from this slot OUT_SLOTS blocks ago has read it
              if (lane == 0) bulk_wait_group_read<C::OUT_SLOTS - 1>();
              __syncwarp();
              // row `lane` of the block: 16-byte chunk j at chunk position j ^ (row % 8) (128-byte swizzle)
#pragma unroll
              for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                    make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (red_blk)
                  tma_reduce_add_2d(&tmOut, buf, col0, r0);
                else
                  tma_store_2d(&tmOut, buf, col0, r0);
                bulk_commit_group();
              }
              oslot = (oslot + 1) % C::OUT_SLOTS;
              continue;
            }
          }
          if (!row_ok || col0 >= args.n_out) continue;
          const bool full_chunk = col0 + 32 <= args.n_out;
          if (args.epi == EPI_BF16) {
            uint16_t* o = reinterpret_cast<uint16_t*>(args.out) + (size_t)row * args.ldo + col0;  // bf16 or f16
            if (full_chunk) {
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                const int f = args.out_f16;
                uint4 pk = make_uint4(pack_16x2(v[j], v[j + 1], f), pack_16x2(v[j + 2], v[j + 3], f),
                                      pack_16x2(v[j + 4], v[j + 5], f), pack_16x2(v[j + 6], v[j + 7], f));
                *reinterpret_cast<uint4*>(o + j) = pk;
              }
            } else {
              for (int j = 0; j < 32 && col0 + j < args.n_out; ++j) store_16(o + j, v[j], args.out_f16);
            }
          } else {
            float* o = reinterpret_cast<float*>(args.out) + (size_t)row * args.ldo + col0;
            if (args.epi == EPI_ADD_F32) {
              const float* r = args.res + (size_t)row * args.ldr + col0;
              if (res_full) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  v[4 * j] += rv[j].x;
                  v[4 * j + 1] += rv[j].y;
                  v[4 * j + 2] += rv[j].z;
                  v[4 * j + 3] += rv[j].w;
                }
              } else {
                for (int j = 0; j < 32 && col0 + j < args.n_out; ++j) v[j] += r[j];
              }
            } else if (args.softcap > 0.f) {
              const float c_ = args.softcap, inv = 1.0f / args.softcap;
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = c_ * tanhf(v[j] * inv);
            }
            if (full_chunk) {
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(o + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            } else {
              for (int j = 0; j < 32 && col0 + j < args.n_out; ++j) o[j] = v[j];
            }
          }
        }
      }
      }  // sub-tiles
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
    if constexpr (SO) {
      // the staged stores must finish before the CTA's shared memory goes away
      if (lane == 0) bulk_wait_group_all();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <int BN, int MT, bool GROUPED = false, bool SO = false, int AR = 0>
fk_status launch_bn(const CUtensorMap& tA, const GemmWeights& w, const GemmArgs& a, int sm_count, cudaStream_t st,
                    const CUtensorMap* tOut = nullptr) {
  using C = Cfg<BN, MT, SO, AR>;
  static DeviceOnce once;
  const cudaError_t attr_err = once.run([] {
    return cudaFuncSetAttribute(gemm_tc_kernel<BN, MT, GROUPED, SO, AR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::SMEM);
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(gemm)");
  // grouped: the m-block count is known on the device only; each group adds
  // at most one partial block to the M / 128 full ones
  const int m_blocks = (a.M + BM * MT - 1) / (BM * MT) + (GROUPED ? a.groups : 0);
  const int n_blocks = a.glu ? (a.n_out + BN / 2 - 1) / (BN / 2) : (a.n_virtual + BN - 1) / BN;
  const int tiles = m_blocks * n_blocks;
  const int grid = std::min(tiles, sm_count);
  gemm_tc_kernel<BN, MT, GROUPED, SO, AR><<<grid, kThreads, C::SMEM, st>>>(
      tA, w.map[0], w.nseg > 1 ? w.map[1] : w.map[0], w.nseg > 2 ? w.map[2] : w.map[0], tOut ? *tOut : w.map[0], a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "gemm_tc_kernel launch");
  return FK_OK;
}

}  // namespace

fk_status gemm_weights_init(GemmWeights* g, const void* const* mats, const int* rows, int nseg, int K, int glu,
                            int f16) {
  if (nseg < 1 || nseg > 3 || (glu && nseg != 2) || K <= 0 || K % 8) return fail(FK_ERR_INVALID_ARG, "gemm weights");
  *g = GemmWeights();
  g->nseg = nseg;
  g->glu = glu;
  g->f16 = f16 ? 1 : 0;
  g->K = K;
  int start = 0;
  for (int s = 0; s < nseg; ++s) {
    if (!mats[s] || rows[s] <= 0) return fail(FK_ERR_INVALID_ARG, "gemm weights: null or empty matrix");
    if (nseg > 1 && !glu && s < nseg - 1 && rows[s] % 64)
      return fail(FK_ERR_INVALID_ARG, "stacked weight matrices need row counts that are multiples of 64");
    fk_status st = make_tmap_bf16(&g->map[s], mats[s], rows[s], K, K, 64);
    if (st != FK_OK) return st;
    g->seg_start[s] = start;
    g->seg_rows[s] = rows[s];
    start += rows[s];
  }
  g->seg_start[nseg] = start;
  if (glu) {
    if (rows[0] != rows[1]) return fail(FK_ERR_INVALID_ARG, "gate/up row counts differ");
    g->n_out = rows[0];
  } else {
    g->n_out = start;
  }
  return FK_OK;
}

fk_status gemm_weights_init_grouped(GemmWeights* g, const void* const* mats, int nseg, int groups, int rows_per_group,
                                    int K, int glu, int f16) {
  if ((glu ? nseg != 2 : nseg != 1) || groups < 1 || rows_per_group <= 0 || rows_per_group % 64 || K <= 0 || K % 8)
    return fail(FK_ERR_INVALID_ARG, "grouped gemm weights");
  *g = GemmWeights();
  g->nseg = nseg;
  g->glu = glu;
  g->f16 = f16 ? 1 : 0;
  g->K = K;
  g->groups = groups;
  g->group_rows = rows_per_group;
  for (int s = 0; s < nseg; ++s) {
    if (!mats[s]) return fail(FK_ERR_INVALID_ARG, "grouped gemm weights: null matrix");
    fk_status st = make_tmap_bf16(&g->map[s], mats[s], (int64_t)groups * rows_per_group, K, K, 64);
    if (st != FK_OK) return st;
    g->seg_rows[s] = rows_per_group;
  }
  // one group's rows: the whole virtual operand of a tile
  g->seg_start[0] = 0;
  g->seg_start[1] = rows_per_group;
  g->n_out = rows_per_group;
  return FK_OK;
}

// Operand checks and kernel arguments shared by the plain and grouped GEMMs.
static fk_status gemm_args(const void* A, int M, int lda, const GemmWeights& w, const GemmOut& o, unsigned* dev_err,
                           CUtensorMap* tA, GemmArgs* a, int* sm_count) {
  if (!A || !o.out || M < 0 || lda < w.K || lda % 8 || o.ldo % (o.epi == EPI_BF16 || o.epi == EPI_GLU_BF16 ? 8 : 4))
    return fail(FK_ERR_INVALID_ARG, "gemm_run: bad operand");
  if (o.epi == EPI_ADD_F32 && (!o.res || o.ldr % 4)) return fail(FK_ERR_INVALID_ARG, "gemm_run: residual");
  fk_status s = check_device(sm_count);
  if (s != FK_OK) return s;
  s = make_tmap_bf16(tA, A, M, w.K, lda, BM);
  if (s != FK_OK) return s;
  *a = GemmArgs{};
  a->M = M;
  a->K = w.K;
  a->n_virtual = w.seg_start[w.nseg];
  a->nseg = w.nseg;
  a->glu = w.glu;
  for (int i = 0; i < 4; ++i) a->seg_start[i] = w.seg_start[i];
  for (int i = 0; i < 3; ++i) a->seg_rows[i] = w.seg_rows[i];
  a->n_out = w.n_out;
  a->epi = o.epi;
  a->act = o.act;
  a->out = o.out;
  a->ldo = o.ldo;
  a->res = o.res;
  a->ldr = o.ldr;
  a->softcap = o.softcap;
  a->dev_err = dev_err;
  a->ab_f16 = w.f16;
  a->out_f16 = o.out_f16;
  a->res_inplace = o.epi == EPI_ADD_F32 && o.res == o.out && o.ldr == o.ldo;
  return FK_OK;
}

fk_status gemm_run_grouped(const void* A, int M, int lda, const GemmWeights& w, const GemmOut& o,
                           const int* group_off, unsigned* dev_err, cudaStream_t st) {
  if (M == 0) return FK_OK;
  if (w.groups < 1 || w.groups > kMoeMaxExperts || !group_off)
    return fail(FK_ERR_INVALID_ARG, "gemm_run_grouped: not a grouped operand");
  if (w.glu ? w.nseg != 2 : w.nseg != 1) return fail(FK_ERR_INVALID_ARG, "gemm_run_grouped: operand layout");
  if (o.epi == EPI_ADD_F32) return fail(FK_ERR_INVALID_ARG, "gemm_run_grouped: no residual epilogue");
  CUtensorMap tA;
  GemmArgs a;
  int sm_count = 0;
  fk_status s = gemm_args(A, M, lda, w, o, dev_err, &tA, &a, &sm_count);
  if (s != FK_OK) return s;
  a.group_off = group_off;
  a.groups = w.groups;
  a.group_rows = w.group_rows;
  if ((M + BM - 1) / BM + w.groups > 65535) return fail(FK_ERR_INVALID_ARG, "gemm_run_grouped: too many rows");
  // 256-row tiles (two M=128 accumulators sharing each B tile: a third less
  // operand traffic per FLOP) once they give every SM two tiles; then
  // 128 x 256; else 128-wide. Outputs of 256-wide tiles are staged and stored
  // by TMA (blocks crossing a group's last row are stored directly).
  const int nb256 = w.glu ? (w.n_out + 127) / 128 : (a.n_virtual + 255) / 256;
  const bool big = ((M + 2 * BM - 1) / (2 * BM)) * nb256 >= 2 * sm_count;
  const bool wide = ((M + BM - 1) / BM) * nb256 >= sm_count;
  if (big || wide || o.epi == EPI_F32) {
    CUtensorMap tOut;
    s = o.epi == EPI_F32 ? make_tmap_f32_out(&tOut, o.out, M, w.n_out, o.ldo)
                         : make_tmap_16_out(&tOut, o.out, M, w.n_out, o.ldo);
    if (s != FK_OK) return s;
    if (big) return launch_bn<256, 2, true, true>(tA, w, a, sm_count, st, &tOut);
    if (wide) return launch_bn<256, 1, true, true>(tA, w, a, sm_count, st, &tOut);
    return launch_bn<128, 1, true, true>(tA, w, a, sm_count, st, &tOut);
  }
  return launch_bn<128, 1, true>(tA, w, a, sm_count, st);
}

fk_status gemm_run(const void* A, int M, int lda, const GemmWeights& w, const GemmOut& o, unsigned* dev_err,
                   cudaStream_t st, void* scratch, size_t scratch_bytes, size_t counter_region, const NormIn* norm) {
  if (M == 0) return FK_OK;
  if (w.groups) return fail(FK_ERR_INVALID_ARG, "gemm_run: grouped operand needs gemm_run_grouped");
  if (M <= kSkinnyMaxTokens && scratch)
    return gemm_run_skinny(A, M, lda, w, o, scratch, scratch_bytes, dev_err, st, true, counter_region, norm);
  if (norm) return fail(FK_ERR_INVALID_ARG, "gemm_run: a fused input norm needs the few-token path");

  CUtensorMap tA;
  GemmArgs a;
  int sm_count = 0;
  fk_status s = gemm_args(A, M, lda, w, o, dev_err, &tA, &a, &sm_count);
  if (s != FK_OK) return s;
  // 256x256 tiles while they give every SM at least two tiles; then 128x256;
  // else 128-wide. fp32 outputs: staged blocks, TMA stores.
  const int m_blocks = (M + BM - 1) / BM;
  const int nb256 = w.glu ? (w.n_out + 127) / 128 : (a.n_virtual + 255) / 256;
  const bool big = ((M + 2 * BM - 1) / (2 * BM)) * nb256 >= 2 * sm_count, wide = m_blocks * nb256 >= sm_count;
  // few rows (a short forward or prefill chunk): 128 x 64 tiles while 128-wide
  // ones would leave SMs without a tile, so that more CTAs stream the weights
  // (not for the gated operand, whose halves are 64-row boxes each)
  const bool narrow = !w.glu && m_blocks * ((a.n_virtual + 127) / 128) < sm_count;
  if (M <= 64 && !big && !wide) {
    // few rows: the A map's box holds only the valid rows (16 or 64), and the
    // shared memory of the rest deepens the weight ring (Cfg, AR)
    const int ar = M <= 16 ? 16 : 64;
    s = make_tmap_bf16(&tA, A, M, w.K, lda, ar);
    if (s != FK_OK) return s;
    if (o.epi == EPI_F32 || o.epi == EPI_ADD_F32) {
      CUtensorMap tOut;
      s = make_tmap_f32_out(&tOut, o.out, M, w.n_out, o.ldo);
      if (s != FK_OK) return s;
      if (narrow)
        return ar == 16 ? launch_bn<64, 1, false, true, 16>(tA, w, a, sm_count, st, &tOut)
                        : launch_bn<64, 1, false, true, 64>(tA, w, a, sm_count, st, &tOut);
      return ar == 16 ? launch_bn<128, 1, false, true, 16>(tA, w, a, sm_count, st, &tOut)
                      : launch_bn<128, 1, false, true, 64>(tA, w, a, sm_count, st, &tOut);
    }
    if (narrow)
      return ar == 16 ? launch_bn<64, 1, false, false, 16>(tA, w, a, sm_count, st)
                      : launch_bn<64, 1, false, false, 64>(tA, w, a, sm_count, st);
    return ar == 16 ? launch_bn<128, 1, false, false, 16>(tA, w, a, sm_count, st)
                    : launch_bn<128, 1, false, false, 64>(tA, w, a, sm_count, st);
  }
  if (o.epi == EPI_F32 || o.epi == EPI_ADD_F32) {
    CUtensorMap tOut;
    s = make_tmap_f32_out(&tOut, o.out, M, w.n_out, o.ldo);
    if (s != FK_OK) return s;
    if (big) return launch_bn<256, 2, false, true>(tA, w, a, sm_count, st, &tOut);
    if (wide) return launch_bn<256, 1, false, true>(tA, w, a, sm_count, st, &tOut);
    if (narrow) return launch_bn<64, 1, false, true>(tA, w, a, sm_count, st, &tOut);
    return launch_bn<128, 1, false, true>(tA, w, a, sm_count, st, &tOut);
  }
  if (big || wide) {  // 16-bit outputs of 256-wide tiles: staged boxes, TMA stores
    CUtensorMap tOut;
    s = make_tmap_16_out(&tOut, o.out, M, w.n_out, o.ldo);
    if (s != FK_OK) return s;
    if (big) return launch_bn<256, 2, false, true>(tA, w, a, sm_count, st, &tOut);
    return launch_bn<256, 1, false, true>(tA, w, a, sm_count, st, &tOut);
  }
  if (narrow) return launch_bn<64, 1>(tA, w, a, sm_count, st);
  return launch_bn<128, 1>(tA, w, a, sm_count, st);
}

}  // namespace fk

extern "C" fk_status fk_gemm_bf16(const void* d_x, const void* d_w, int32_t P, int32_t K, int32_t N, void* d_y,
                                  int32_t y_fp32, void* stream) {
  using namespace fk;
  if (!d_x || !d_w || !d_y || P < 0 || K <= 0 || N <= 0) return fail(FK_ERR_INVALID_ARG, "fk_gemm_bf16: bad argument");
  if (K % 8 || N % 8) return fail(FK_ERR_INVALID_ARG, "fk_gemm_bf16: K and N must be multiples of 8");
  if ((reinterpret_cast<uintptr_t>(d_x) | reinterpret_cast<uintptr_t>(d_w) | reinterpret_cast<uintptr_t>(d_y)) & 15)
    return fail(FK_ERR_INVALID_ARG, "fk_gemm_bf16: buffers must be 16-byte aligned");
  int sm = 0;
  fk_status s = check_device(&sm);
  if (s != FK_OK) return s;
  GemmWeights w;
  const void* mats[1] = {d_w};
  int rows[1] = {N};
  s = gemm_weights_init(&w, mats, rows, 1, K, 0);
  if (s != FK_OK) return s;
  unsigned* ctl = nullptr;
  s = op_control_block(&ctl);
  if (s != FK_OK) return s;
  GemmOut o;
  o.epi = y_fp32 ? EPI_F32 : EPI_BF16;
  o.out = d_y;
  o.ldo = N;
  return gemm_run(d_x, P, K, w, o, ctl, static_cast<cudaStream_t>(stream));
}
