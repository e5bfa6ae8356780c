// Allocation-free variant of the decode-attention entry point.
//
// Some callers cannot hand the library a scratch buffer: their device memory
// is owned entirely by someone else (a framework's caching allocator that must
// stay the single owner of the heap, an embedding runtime that forbids driver
// allocations after start-up), or they run on a latency-critical path that must
// never enter the driver's allocation code. This entry point needs only its
// inputs and outputs: the decode kernel splits each (sequence, kv head) across
// a thread-block cluster and merges the split partials in the cluster's
// shared memory, so no device memory beyond the caller's tensors is touched
// and nothing is shared between calls (calls on different streams may
// overlap).
#include "fk_internal.h"

namespace fk {
fk_status attention_decode_plan(int B, int Hkv, int hd, int ctx, int* splits);
fk_status attention_decode_run(const void* q, const void* kc, const void* vc, int B, int Hq, int Hkv, int hd, int cap,
                               int ctx, int window, int splits, void* out, cudaStream_t st);
}  // namespace fk

// No device memory is reserved for this entry point.
extern "C" size_t fk_attention_decode_noalloc_limit(void) { return 0; }

extern "C" fk_status fk_attention_decode_noalloc(const void* d_q, const void* d_kcache, const void* d_vcache,
                                                 int32_t batch, int32_t n_q_heads, int32_t n_kv_heads,
                                                 int32_t head_dim, int32_t cap, int32_t ctx, int32_t window,
                                                 void* d_out, void* stream) {
  using fk::fail;
  if (!d_q || !d_kcache || !d_vcache || !d_out) return fail(FK_ERR_INVALID_ARG, "attention decode: null pointer");
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads || n_q_heads / n_kv_heads > 8)
    return fail(FK_ERR_INVALID_ARG, "attention decode: need batch >= 1 and 1..8 query heads per kv head");
  if (head_dim != 64 && head_dim != 128 && head_dim != 256)
    return fail(FK_ERR_INVALID_ARG, "attention decode: head_dim 64/128/256");
  if (ctx < 1 || ctx > cap || window < 0 || cap % 64)
    return fail(FK_ERR_INVALID_ARG, "attention decode: need 1 <= ctx <= cap, cap a multiple of 64");
  if ((reinterpret_cast<uintptr_t>(d_q) | reinterpret_cast<uintptr_t>(d_kcache) |
       reinterpret_cast<uintptr_t>(d_vcache)) & 15)
    return fail(FK_ERR_INVALID_ARG, "attention decode: q and caches must be 16-byte aligned");
  int splits = 1;
  fk_status s = fk::attention_decode_plan(batch, n_kv_heads, head_dim, ctx, &splits);
  if (s != FK_OK) return s;
  return fk::attention_decode_run(d_q, d_kcache, d_vcache, batch, n_q_heads, n_kv_heads, head_dim, cap, ctx, window,
                                  splits, d_out, static_cast<cudaStream_t>(stream));
}
