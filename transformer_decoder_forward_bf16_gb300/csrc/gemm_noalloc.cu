// Allocation-free variant of the few-row (split-K) GEMM entry point.
//
// fk_gemm_bf16_splitk needs a scratch buffer from its caller: the fp32 partial
// sums of the K splits and the arrival counters that elect the CTA which adds
// them. Some callers cannot provide one. Their device memory may belong
// entirely to another allocator that must stay the only owner of the heap (a
// framework's caching allocator, an embedded runtime that forbids driver
// allocations after start-up), or they run on a latency-critical path that must
// never enter the driver's allocation code. For them this entry point keeps the
// scratch in a fixed array inside the library's own device image, so a call
// needs only its inputs and outputs and calls no allocator of any kind.
//
// Limit: the array holds kNoAllocScratchBytes (8 MiB). Every GPU that loads the
// library holds it until the process exits. A call whose scratch would not fit
// (fk_gemm_bf16_splitk_scratch_bytes above the limit) is rejected with
// FK_ERR_WORKSPACE before anything is launched.
//
// Sharing: every call on a device uses the same array, and the array keeps
// whatever the previous call left there. The arrival counters must start at
// zero, so each call clears them on its stream before the kernel runs; the
// partial sums need no clearing (every value the reduction reads was written
// by the same call). Two calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on the array and give wrong
// results: serialise them.
//
// Set-up: host code cannot pass the array's name to a kernel (on the host it is
// only a stand-in for the device symbol). The first call on each device looks
// up the array's device address with cudaGetSymbolAddress while that device is
// current and keeps it; make that first call before any stream capture begins
// on the device.
#include <cstdio>
#include <mutex>

#include "fk_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;

__device__ __align__(256) static unsigned char g_splitk_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[fk::kMaxDevices] = {nullptr};

fk_status scratch_for_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fk::cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= fk::kMaxDevices) return fk::fail(FK_ERR_INVALID_ARG, "device index out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_splitk_scratch);
    if (e != cudaSuccess) return fk::cuda_fail(e, "cudaGetSymbolAddress(split-K scratch)");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FK_OK;
}

}  // namespace

extern "C" size_t fk_gemm_bf16_splitk_noalloc_limit(void) { return kNoAllocScratchBytes; }

extern "C" fk_status fk_gemm_bf16_splitk_noalloc(const void* d_x, const void* d_w, int32_t P, int32_t K, int32_t N,
                                                 void* d_y, int32_t y_fp32, void* stream) {
  fk_status s = fk::check_device(nullptr);
  if (s != FK_OK) return s;
  const size_t need = fk_gemm_bf16_splitk_scratch_bytes(P, K, N);
  if (need == 0) return fk::fail(FK_ERR_INVALID_ARG, "fk_gemm_bf16_splitk_noalloc: bad shape (1 <= P <= 64, K, N >= 8)");
  if (need > kNoAllocScratchBytes) {
    char buf[192];
    snprintf(buf, sizeof buf,
             "fk_gemm_bf16_splitk_noalloc: this shape needs %zu bytes of scratch; the built-in array holds %zu "
             "(use fk_gemm_bf16_splitk with a caller buffer)",
             need, kNoAllocScratchBytes);
    return fk::fail(FK_ERR_WORKSPACE, buf);
  }
  void* scratch = nullptr;
  s = scratch_for_current_device(&scratch);
  if (s != FK_OK) return s;
  return fk::gemm_splitk_op(d_x, d_w, P, K, N, d_y, y_fp32, scratch, kNoAllocScratchBytes,
                            static_cast<cudaStream_t>(stream));
}
