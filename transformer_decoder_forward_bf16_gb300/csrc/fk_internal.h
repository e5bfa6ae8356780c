// Host-side internal declarations shared by the fk translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
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

// Per-device one-time set-up: kernel attributes (shared-memory size, cluster
// permissions) belong to a device's context, so they are set once on every
// device that launches the kernel, with that device current.
constexpr int kMaxDevices = 64;
struct DeviceOnce {
  std::mutex mu;
  uint64_t done = 0;
  cudaError_t err[kMaxDevices] = {};
  template <typename F>
  cudaError_t run(F&& init) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!((done >> dev) & 1ull)) {
      err[dev] = init();
      done |= 1ull << dev;
    }
    return err[dev];
  }
};

// Device control block: word 0 holds the error bits (FK_DEVERR_*); words 1
// and 2 are test controls read by the pipelined kernels (word 1: a wait limit
// in microseconds replacing the default, 0 = default; word 2: nonzero makes
// the op-level skinny GEMM leave its first pipeline stage unarmed, so its
// consumers' bounded wait runs out). Models keep theirs in the model arena;
// op-level calls share one per device, owned by the library.
constexpr size_t kCtlWords = 4;
// The op-level control block of the current device (resolved once per device).
fk_status op_control_block(unsigned** out);

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
// 2-D fp32 row-major output [rows, cols] with row stride ld (elements), boxes
// of 32 x 32, 128-byte swizzle: the target of TMA stores of staged tiles.
fk_status make_tmap_f32_out(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld);
// The same for a 16-bit (bf16 or f16: TMA moves the bits) output, boxes of
// 32 rows x 64 columns.
fk_status make_tmap_16_out(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld);

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
  int f16 = 0;             // the matrices (and so the A operand) are IEEE f16, else bf16
  int K = 0;
  int n_out = 0;           // output columns (GLU: rows of one matrix)
  int groups = 0;          // grouped (expert) operand: `groups` matrices stacked per map, 0 = plain
  int group_rows = 0;      // rows of one group's matrix in each map
};

// f16: the matrices hold IEEE f16 (copies made by the model), else bf16.
fk_status gemm_weights_init(GemmWeights* g, const void* const* mats, const int* rows, int nseg, int K, int glu,
                            int f16 = 0);

// Grouped operand: each map holds `groups` matrices of rows_per_group x K
// stacked along the rows (the experts of a MoE layer); nseg 2 with glu 1 is a
// gate/up pair, nseg 1 a single matrix per group.
fk_status gemm_weights_init_grouped(GemmWeights* g, const void* const* mats, int nseg, int groups, int rows_per_group,
                                    int K, int glu, int f16 = 0);

struct GemmOut {
  int epi = EPI_BF16;
  void* out = nullptr;
  int ldo = 0;             // elements
  const float* res = nullptr;
  int ldr = 0;
  float softcap = 0.f;
  int act = 0;             // GLU activation: 0 SiLU, 1 GELU (tanh form)
  int out_f16 = 0;         // EPI_BF16 / EPI_GLU_BF16 store IEEE f16 instead of bf16
  // few-token EPI_ADD_F32 with the fused split-K reduction (skinny_fused_tail):
  // per 128-feature group sums of squares of each stored row, [M][ceil(n_out/128)]
  float* ssq = nullptr;
};

// RMSNorm of the input fused into the few-token GEMM: the A operand becomes
// 16-bit(x[t] * rsqrt(mean(x[t]^2) + eps) * w) of fp32 rows x [M, K] (row
// stride ldx) and bf16 weights w [K]; for M <= kNormFuseMaxTokens.
constexpr int kNormFuseMaxTokens = 2;
// ssq (optional): per 128-feature group sums of squares of x's rows, [M][n_ssq],
// from the GemmOut.ssq of the GEMM that produced x (else the rows are read whole).
struct NormIn {
  const float* x = nullptr;
  int ldx = 0;
  const void* w = nullptr;
  float eps = 0.f;
  const float* ssq = nullptr;
  int n_ssq = 0;
};

// A: bf16 [M, K] with row stride lda (elements, multiple of 8). With M <=
// kSkinnyMaxTokens and a large enough scratch buffer (skinny_scratch_bytes)
// the weight-streaming split-K kernel runs instead of the tiled one.
// counter_region: bytes at the start of the scratch reserved for the split-K
// arrival counters of every GEMM sharing the scratch (0: this GEMM's own).
// norm: fused input RMSNorm (few-token path only; A is then not read).
fk_status gemm_run(const void* A, int M, int lda, const GemmWeights& w, const GemmOut& o, unsigned* dev_err,
                   cudaStream_t st, void* scratch = nullptr, size_t scratch_bytes = 0, size_t counter_region = 0,
                   const NormIn* norm = nullptr);

// Grouped GEMM: rows [group_off[g], group_off[g+1]) of A (M rows in all)
// multiply group g of the grouped operand w; group_off (device, groups + 1
// entries, nondecreasing, group_off[groups] <= M) is read by the kernel.
fk_status gemm_run_grouped(const void* A, int M, int lda, const GemmWeights& w, const GemmOut& o,
                           const int* group_off, unsigned* dev_err, cudaStream_t st);

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
// The few-token GEMM of M <= kNormFuseMaxTokens rows finishes an epi output in
// its own last CTAs (and can then write GemmOut.ssq).
bool skinny_fused_tail(const GemmWeights& w, int M, int sm_count, int epi);
size_t skinny_partial_bytes(const GemmWeights& w, int M, int sm_count);
// The scratch holds [counters: counter_region bytes (0 = this GEMM's own)]
// [partial sums]. GEMMs that share a scratch share one counter region, sized
// for the one with the most tiles, so no GEMM's partials overlap another's
// counters. counters_zeroed: the counters are known to be zero (a session
// clears them once; every launch leaves them zero again).
fk_status gemm_run_skinny(const void* A, int M, int lda, const GemmWeights& w, const GemmOut& o, void* scratch,
                          size_t scratch_bytes, unsigned* dev_err, cudaStream_t st, bool counters_zeroed = true,
                          size_t counter_region = 0, const NormIn* norm = nullptr);

// The op-level few-row GEMM (fk_gemm_bf16_splitk) over a given scratch buffer.
fk_status gemm_splitk_op(const void* d_x, const void* d_w, int P, int K, int N, void* d_y, int y_fp32,
                         void* d_scratch, size_t scratch_bytes, cudaStream_t st);

// tcgen05 flash attention for prefill (head_dim 64, 128 or 256; caches as in
// the session layout, V transposed, cap a multiple of 64, ldq a multiple of 8).
// The same with two 128-query tiles per CTA taking turns on the tensor core
// (head_dim 64 or 128); attention_prefill_tc dispatches those head sizes here.
fk_status attention_prefill_pp(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B, int S,
                               int pos0, int Hq, int Hkv, int hd, int window, float scale, void* o,
                               unsigned* dev_err, cudaStream_t st, int io_f16, int out_f16);
// io_f16: q, the caches and the probabilities are IEEE f16 (else bf16);
// out_f16: the output is stored as f16.
fk_status attention_prefill_tc(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B, int S,
                               int pos0, int Hq, int Hkv, int hd, int window, float scale, void* o,
                               unsigned* dev_err, cudaStream_t st, int io_f16 = 0, int out_f16 = 0);

// ---------------------------------------------------------------------------
// Mixture-of-experts FFN
// ---------------------------------------------------------------------------
constexpr int kMoeMaxExperts = 256;
constexpr int kMoeMaxK = 16;
constexpr int kMoeFewMaxTokens = 64;  // calls of up to this many tokens may take the split-K expert GEMM
struct MoeWeights {
  GemmWeights router;   // [E, H], fp32 logits
  GemmWeights gate_up;  // grouped gate/up pair, E groups of [Ie, H]
  GemmWeights down;     // grouped, E groups of [H, Ie]
  int E = 0, k = 0, Ie = 0, H = 0;
  int norm_topk = 1;
  int act = 0;          // 0 SiLU, 1 GELU (tanh form)
  int act_f16 = 0;      // the gated activation is stored as f16 (else bf16)
};
// Scratch of one MoE FFN call over up to T tokens (layout from moe_scratch).
struct MoeScratch {
  float* z = nullptr;        // [T, E] router logits
  int32_t* ids = nullptr;    // [T, k]
  float* w = nullptr;        // [T, k]
  float* margin = nullptr;   // [T]
  int32_t* counts = nullptr; // [blocks, E] tokens per expert per routing block
  int32_t* base = nullptr;   // [blocks, E] first sorted row of each block's tokens of each expert
  int32_t* group_off = nullptr;  // [E + 1] first sorted row of each expert
  int32_t* active = nullptr;     // [kMoeMaxExperts + 1] experts with rows in id order, then their number
  unsigned* exp_counters = nullptr;  // few-token expert GEMMs: arrival counters, zero between launches
  size_t exp_counters_bytes = 0;
  float* exp_part = nullptr;         // few-token expert GEMMs: split partial sums
  int32_t* pos = nullptr;    // [T, k] sorted row of each (token, slot)
  int32_t* src = nullptr;    // [T*k] token of each sorted row
  void* xs = nullptr;        // [T*k, H] 16-bit: gathered FFN inputs, sorted by expert
  void* hs = nullptr;        // [T*k, Ie] 16-bit: gated activations
  float* ys = nullptr;       // [T*k, H] expert outputs
};
// Bytes of the scratch for T tokens; with base != NULL also fills *s.
size_t moe_scratch(const MoeWeights& mw, long T, MoeScratch* s, uint8_t* base);
// The MoE FFN of u [T, H] (16-bit, the type of mw.router): out = res + d when
// res is given (res may not alias out), else out = d. forced: NULL or int32
// [T, k] expert ids; trace_ids / trace_margin: NULL or outputs of the routing.
// few: up to kMoeFewMaxTokens tokens run the expert GEMMs as a split-K weight
// stream (its arrival counters, s.exp_counters, must be zero between calls;
// each call leaves them zero). gemv/gemv_bytes/gemv_counter: split-K scratch
// for the router GEMM of few tokens (NULL: tiled GEMM).
// next_norm: NULL, or the RMSNorm of out for the next consumer (the next
// layer's Q|K|V projection or the LM head), made by the combine step.
struct NormOut {
  const void* w = nullptr;  // bf16 [H]
  float eps = 0.f;
  void* u = nullptr;        // 16-bit [T, H]
  int f16 = 0;              // u holds IEEE f16 (else bf16)
};
fk_status moe_ffn_run(const MoeWeights& mw, const void* u, int T, const MoeScratch& s, const int32_t* forced,
                      int32_t* trace_ids, float* trace_margin, float* out, const float* res, unsigned* dev_err,
                      cudaStream_t st, bool few = false, void* gemv = nullptr, size_t gemv_bytes = 0,
                      size_t gemv_counter = 0, const NormOut* next_norm = nullptr);
// The routing step alone (fk_op_moe_route): ids, weights, margins, and per
// routing block expert counts when counts != NULL.
fk_status moe_route_launch(const float* z, int T, int E, int ld, int k, int norm_topk, const int32_t* forced,
                           int32_t* ids, float* w, float* margin, int32_t* counts, unsigned* dev_err,
                           cudaStream_t st);

}  // namespace fk
