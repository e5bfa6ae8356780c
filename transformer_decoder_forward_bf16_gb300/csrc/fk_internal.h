// Host-side internal declarations shared by the fk translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/fk.h"

namespace fk {

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
void set_error(const std::string& msg);
fk_status fail(fk_status s, const std::string& msg);
fk_status cuda_fail(cudaError_t e, const char* what);
#define FK_CUDA_TRY(expr)                                       \
  do {                                                          \
    cudaError_t _e = (expr);                                    \
    if (_e != cudaSuccess) return ::fk::cuda_fail(_e, #expr);   \
  } while (0)

// Current device is an sm_103 GB300-class GPU (cached per device).
fk_status check_device(int* sm_count);

// ---------------------------------------------------------------------------
// kernel timing: RAII scope recording events around the launches inside it
// ---------------------------------------------------------------------------
bool profiling_enabled();
struct ProfScope {
  int slot = -1;
  cudaStream_t st = nullptr;
  ProfScope(const char* name, cudaStream_t stream);
  ~ProfScope();
};

// ---------------------------------------------------------------------------
// TMA descriptors
// ---------------------------------------------------------------------------
// 2-D bf16 row-major tensor [rows, cols] with row stride ld (elements), boxes
// of box_rows x 64 columns, 128-byte swizzle, out-of-bounds elements read as 0.
fk_status make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                         int box_rows);

// ---------------------------------------------------------------------------
// GEMM (tcgen05): out = epilogue(A[M,K] · Bᵀ)
// ---------------------------------------------------------------------------
enum GemmEpi : int {
  EPI_BF16 = 0,     // out bf16 [M, ldo]
  EPI_F32 = 1,      // out fp32 [M, ldo], optional softcap c*tanh(z/c)
  EPI_ADD_F32 = 2,  // out fp32 = res + acc (res may alias out)
  EPI_GLU_BF16 = 3  // out bf16 [M, ldo] = act(gate) * up over interleaved gate/up tiles
};

// The weight operand: one matrix, up to three stacked along the output rows
// (Q|K|V), or a gate/up pair read tile-interleaved (GLU).
struct GemmWeights {
  CUtensorMap map[3];      // boxes of 64 rows x 64 columns
  int nseg = 0;            // number of stacked matrices (1..3); 2 for GLU
  int seg_start[4] = {0};  // first output row of each stacked matrix; seg_start[nseg] = total rows
  int seg_rows[3] = {0};
  int glu = 0;             // 1: virtual rows interleave gate/up per tile
  int K = 0;
  int n_out = 0;           // output columns (GLU: rows of one matrix)
};

fk_status gemm_weights_init(GemmWeights* g, const void* const* mats, const int* rows, int nseg, int K, int glu);

struct GemmOut {
  int epi = EPI_BF16;
  void* out = nullptr;
  int ldo = 0;             // elements
  const float* res = nullptr;
  int ldr = 0;
  float softcap = 0.f;
  int act = 0;             // GLU activation: 0 SiLU, 1 GELU (tanh form)
};

// A: bf16 [M, K] with row stride lda (elements, multiple of 8). With M <=
// kSkinnyMaxTokens and a large enough scratch buffer (skinny_scratch_bytes)
// the weight-streaming split-K kernel runs instead of the tiled one.
// counter_region: bytes at the start of the scratch reserved for the split-K
// arrival counters of every GEMM sharing the scratch (0: this GEMM's own).
fk_status gemm_run(const void* A, int M, int lda, const GemmWeights& w, const GemmOut& o, unsigned* dev_err,
                   cudaStream_t st, void* scratch = nullptr, size_t scratch_bytes = 0, size_t counter_region = 0);

// Skinny (few-token) GEMM: swap-AB tcgen05 split-K + ordered reduction.
constexpr int kSkinnyMaxTokens = 64;
struct SkinnyPlan {
  int splits = 1, kb_per_split = 1, n_tiles = 1, nk = 1;
  bool direct = false;       // one split, epilogue straight from TMEM (small operands)
  size_t counter_bytes = 0;  // per-group arrival counters at the start of the scratch
  size_t part_bytes = 0;     // whole scratch: counters + fp32 partial sums
};
// allow_direct: the operand may take the single-split direct epilogue (not a
// gate/up pair, whose halves are combined by the reduction).
SkinnyPlan skinny_plan(int M, int K, int n_rows, int sm_count, bool allow_direct);
// Scratch of one skinny GEMM at up to M tokens: its arrival counters and its
// fp32 partial sums (the partials of a smaller M never take more).
size_t skinny_counter_bytes(const GemmWeights& w, int M, int sm_count);
size_t skinny_partial_bytes(const GemmWeights& w, int M, int sm_count);
// The scratch holds [counters: counter_region bytes (0 = this GEMM's own)]
// [partial sums]. GEMMs that share a scratch share one counter region, sized
// for the one with the most tiles, so no GEMM's partials overlap another's
// counters. counters_zeroed: the counters are known to be zero (a session
// clears them once; every launch leaves them zero again).
fk_status gemm_run_skinny(const void* A, int M, int lda, const GemmWeights& w, const GemmOut& o, void* scratch,
                          size_t scratch_bytes, unsigned* dev_err, cudaStream_t st, bool counters_zeroed = true,
                          size_t counter_region = 0);

// tcgen05 flash attention for prefill (head_dim 64 or 128; caches as in the
// session layout, V transposed, cap a multiple of 64).
bool attention_prefill_tc_supported(int hd, int ldq, int cap);
fk_status attention_prefill_tc(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B, int S,
                               int pos0, int Hq, int Hkv, int hd, int window, float scale, void* o,
                               unsigned* dev_err, cudaStream_t st);

}  // namespace fk
