// Allocation-free variant of the decode-attention entry point.
//
// Some callers cannot hand the library a scratch buffer: their device memory
// is owned entirely by someone else (a framework's caching allocator that must
// stay the single owner of the heap, an embedding runtime that forbids driver
// allocations after start-up), or they run on a latency-critical path that must
// never enter the driver's allocation code. For them this entry point keeps the
// split-KV partial results in a fixed array in the library's own device image,
// so a call needs only its inputs and outputs.
//
// Limit: the array holds kNoAllocScratchBytes (4 MiB). Every GPU that loads the
// library reserves it until the process exits. Calls whose partial results
// would not fit are rejected with FK_ERR_WORKSPACE before anything is launched.
//
// Sharing: every call on a device uses the same array, and the array keeps
// whatever the previous call left in it. Nothing in it needs to start at zero:
// every slot a call reads was written earlier by the same call. Two calls whose
// kernels overlap on the GPU (different streams, or different host threads)
// race on the array and give wrong results; serialise them.
//
// Set-up: the first call on each device looks up the array's device address
// with cudaGetSymbolAddress while that device is current (host code may not
// pass the array's name to a kernel: on the host it is only a stand-in). Make
// that first call before any stream capture begins on the device.
#include <mutex>

#include "fk_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) static unsigned char g_decode_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

fk_status scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fk::cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fk::fail(FK_ERR_INVALID_ARG, "device index out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return fk::cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FK_OK;
}

}  // namespace

namespace fk {
fk_status attention_decode_plan(int B, int Hq, int Hkv, int hd, int ctx, int* chunk, int* splits, size_t* bytes);
fk_status attention_decode_run(const void* q, const void* kc, const void* vc, int B, int Hq, int Hkv, int hd, int cap,
                               int ctx, int window, int chunk, int splits, void* scratch, void* out, cudaStream_t st);
}  // namespace fk

extern "C" size_t fk_attention_decode_noalloc_limit(void) { return kNoAllocScratchBytes; }

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
  int chunk = 0, splits = 0;
  size_t need = 0;
  fk_status s = fk::attention_decode_plan(batch, n_q_heads, n_kv_heads, head_dim, ctx, &chunk, &splits, &need);
  if (s != FK_OK) return s;
  if (need > kNoAllocScratchBytes) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "attention decode (no-alloc): partial results need %zu bytes, more than the fixed %zu-byte array; "
             "use fk_attention_decode with a caller buffer",
             need, kNoAllocScratchBytes);
    return fail(FK_ERR_WORKSPACE, buf);
  }
  void* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != FK_OK) return s;
  return fk::attention_decode_run(d_q, d_kcache, d_vcache, batch, n_q_heads, n_kv_heads, head_dim, cap, ctx, window,
                                  chunk, splits, scratch, d_out, static_cast<cudaStream_t>(stream));
}
