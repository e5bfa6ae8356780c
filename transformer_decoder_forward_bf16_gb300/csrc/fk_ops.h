// Launchers of the non-GEMM kernels (host side, internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fk {

// u_f16 / f16: the 16-bit activations a kernel writes (and, for RoPE, reads)
// are IEEE f16 instead of bf16 (the model's storage site for them).
cudaError_t launch_embed_norm(const int32_t* ids, const void* E, int T, int H, int V, float scale, const void* w,
                              float eps, float* x, void* u, unsigned* dev_err, cudaStream_t st, int u_f16);
cudaError_t launch_rmsnorm(const float* x, int ldx, int T, int H, const void* w, float eps, void* u, int ldu,
                           cudaStream_t st, int u_f16);
cudaError_t launch_rmsnorm_f32(const float* x, int T, int H, const void* w, float eps, float* y, cudaStream_t st);
cudaError_t launch_post_norm_residual(const float* a, const float* x_in, float* x_out, int T, int H,
                                      const void* w_post, const void* w_next, float eps, void* u, cudaStream_t st,
                                      int u_f16);
// Prefill chunks: pos0 is the position of the first of S tokens per sequence
// (decode steps apply RoPE inside the attention kernel).
// q is rotated in place, k written to the cache, v transposed into the cache.
cudaError_t launch_rope_qkv(void* qkv, int ldqkv, int T, int S, int pos0, int Hq, int Hkv, int hd,
                            const float2* rope, int qk_norm, const void* q_norm, const void* k_norm, float eps,
                            void* kcache, void* vcache, int cap, cudaStream_t st, int f16);
// Per-row argmax (lowest index on ties) of z [R][ldz]; out2 (optional): a
// second copy of the ids; margin (optional): fp32 top-1 minus top-2 value per
// row. With `scratch` (argmax_scratch_bytes, its trailing counters zeroed
// once) and R <= kArgmaxMaxSplitRows, each row is split across blocks.
constexpr int kArgmaxMaxSplitRows = 64;
inline size_t argmax_counter_offset() { return (size_t)kArgmaxMaxSplitRows * 32 * 12; }
inline size_t argmax_scratch_bytes() { return argmax_counter_offset() + kArgmaxMaxSplitRows * 4; }
cudaError_t launch_argmax(const float* z, int R, int V, int ldz, int32_t* out, cudaStream_t st,
                          int32_t* out2 = nullptr, void* scratch = nullptr, float* margin = nullptr);
// dst[i] = f16(src[i]) for n bf16 values (n % 8 == 0, 16-byte aligned)
cudaError_t launch_bf16_to_f16(const void* src, void* dst, size_t n, cudaStream_t st);
// *p = value (one thread), and *p += 1
cudaError_t launch_set_int(int* p, int value, cudaStream_t st);
cudaError_t launch_inc_int(int* p, cudaStream_t st);
cudaError_t launch_gather_last_rows(const void* src, int ld, int S, int H, int B, void* dst, cudaStream_t st);

// One query per sequence at position ctx-1 (ctx = keys in the cache; if
// d_ctx is non-null, ctx = *d_ctx + 1, *d_ctx being the length before the
// new token). Split-KV over a cluster of n_splits CTAs per (sequence, kv
// head), merged on chip in a fixed order. decode_attention_splits picks
// n_splits (a power of two <= 16) for a batch, head_dim and longest context.
int decode_attention_splits(int B, int Hkv, int hd, int max_ctx, int sm_count);
cudaError_t launch_attention_decode(const void* q, int ldq, const void* kcache, const void* vcache, int cap, int B,
                                    int ctx, const int* d_ctx, int Hq, int Hkv, int hd, int window, float scale,
                                    int n_splits, void* o, unsigned* dev_err, cudaStream_t st, int io_f16 = 0,
                                    int out_f16 = 0);
// A session's decode step (S == 1, length *d_ctx before the new token): takes
// the token's qkv row (ldqkv = its stride), applies [QK-norm and] RoPE at
// position *d_ctx to q and k as launch_rope_qkv does, writes k and v into the
// caches and attends, all in one kernel. Launched after the QKV projection
// with programmatic dependent launch, it reads the caches' earlier positions
// before waiting for the projection.
cudaError_t launch_attention_decode_rope(const void* qkv, int ldqkv, void* kcache, void* vcache, int cap, int B,
                                         const int* d_ctx, int Hq, int Hkv, int hd, int window, float scale,
                                         const float2* rope, int qk_norm, const void* q_norm, const void* k_norm,
                                         float eps, int n_splits, void* o, unsigned* dev_err, cudaStream_t st,
                                         int io_f16, int out_f16);

}  // namespace fk
