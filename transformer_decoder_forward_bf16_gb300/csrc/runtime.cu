// Host runtime shared by the entry points: error reporting, device checks and
// TMA descriptor encoding.
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "fk_internal.h"
#include "fk_launch.h"

namespace fk {

namespace {
thread_local std::string g_last_error;
}

void set_error(const std::string& msg) { g_last_error = msg; }

fk_status fail(fk_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

fk_status cuda_fail(cudaError_t e, const char* what) {
  char buf[512];
  snprintf(buf, sizeof buf, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  g_last_error = buf;
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return FK_ERR_NO_DEVICE;
  return FK_ERR_CUDA;
}

fk_status check_device(int* sm_count) {
  static std::mutex mu;
  static int cached_dev = -1, cached_sms = 0;
  static fk_status cached = FK_OK;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e == cudaErrorInvalidDevice ? cudaErrorNoDevice : e, "cudaGetDevice");
  }
  std::lock_guard<std::mutex> lock(mu);
  if (dev != cached_dev) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return fail(FK_ERR_NO_DEVICE, "cannot query the CUDA device");
    }
    cached_dev = dev;
    cached_sms = sms;
    if (major != 10 || minor != 3) {
      char buf[160];
      snprintf(buf, sizeof buf, "device %d is sm_%d%d; this library is built for sm_103a (GB300) only", dev, major,
               minor);
      set_error(buf);
      cached = FK_ERR_NO_DEVICE;
    } else {
      cached = FK_OK;
    }
  }
  if (cached != FK_OK) return fail(cached, "device is not sm_103 (GB300)");
  if (sm_count) *sm_count = cached_sms;
  return FK_OK;
}

// The op-level control block: one per device that loads the library (16
// bytes). Host code reaches it through its device address, looked up once per
// device with that device current.
namespace {
__device__ __align__(16) unsigned g_op_ctl[kCtlWords];
std::mutex g_ctl_mu;
unsigned* g_ctl_ptr[kMaxDevices] = {nullptr};
}  // namespace

fk_status op_control_block(unsigned** out) {
  *out = nullptr;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e == cudaErrorInvalidDevice ? cudaErrorNoDevice : e, "cudaGetDevice");
  }
  if (dev < 0 || dev >= kMaxDevices) return fail(FK_ERR_INVALID_ARG, "device index out of range");
  std::lock_guard<std::mutex> lock(g_ctl_mu);
  if (!g_ctl_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_op_ctl);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(op control block)");
    e = cudaMemset(p, 0, kCtlWords * sizeof(unsigned));
    if (e != cudaSuccess) return cuda_fail(e, "clear op control block");
    g_ctl_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_ctl_ptr[dev];
  return FK_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return encode;
}

fk_status make_tmap_16_out(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return fail(FK_ERR_NO_DEVICE, "cuTensorMapEncodeTiled is unavailable (no CUDA driver)");
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (ld * 2) % 16 || rows <= 0 || cols <= 0)
    return fail(FK_ERR_INVALID_ARG, "16-bit tensor map: base must be 16-byte aligned, rows 16-byte multiples");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[128];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled (16-bit out) failed (%d)", (int)r);
    return fail(FK_ERR_CUDA, buf);
  }
  return FK_OK;
}

fk_status make_tmap_f32_out(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int64_t ld) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return fail(FK_ERR_NO_DEVICE, "cuTensorMapEncodeTiled is unavailable (no CUDA driver)");
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (ld * 4) % 16 || rows <= 0 || cols <= 0)
    return fail(FK_ERR_INVALID_ARG, "fp32 tensor map: base must be 16-byte aligned, rows 16-byte multiples");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 4)};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[128];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled (fp32) failed (%d)", (int)r);
    return fail(FK_ERR_CUDA, buf);
  }
  return FK_OK;
}

fk_status make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return fail(FK_ERR_NO_DEVICE, "cuTensorMapEncodeTiled is unavailable (no CUDA driver)");
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (ld * 2) % 16 || rows <= 0 || cols <= 0 || box_rows > 256)
    return fail(FK_ERR_INVALID_ARG, "tensor map: base must be 16-byte aligned, rows 16-byte multiples");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[128];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return fail(FK_ERR_CUDA, buf);
  }
  return FK_OK;
}

// ---------------------------------------------------------------------------
// kernel timing
// ---------------------------------------------------------------------------
namespace {
struct ProfClass {
  std::string name;
  int64_t launches = 0;
  double ms = 0.0;
};
struct Pending {
  int cls;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfClass> g_prof_classes;
std::vector<Pending> g_prof_pending;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

void prof_drain_locked() {
  for (const Pending& p : g_prof_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.b) == cudaSuccess && cudaEventElapsedTime(&ms, p.a, p.b) == cudaSuccess) {
      g_prof_classes[p.cls].launches += 1;
      g_prof_classes[p.cls].ms += ms;
    } else {
      cudaGetLastError();
    }
    g_prof_pool.push_back(p.a);
    g_prof_pool.push_back(p.b);
  }
  g_prof_pending.clear();
}
}  // namespace

bool profiling_enabled() { return g_prof_on; }

namespace {
thread_local bool g_pdl = false;
}
bool pdl_enabled() { return g_pdl; }
PdlScope::PdlScope(bool on) : prev(g_pdl) { g_pdl = on; }
PdlScope::~PdlScope() { g_pdl = prev; }

ProfScope::ProfScope(const char* name, cudaStream_t stream) : st(stream) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  int cls = -1;
  for (size_t i = 0; i < g_prof_classes.size(); ++i)
    if (g_prof_classes[i].name == name) cls = (int)i;
  if (cls < 0) {
    g_prof_classes.push_back(ProfClass{name});
    cls = (int)g_prof_classes.size() - 1;
  }
  Pending p{cls, prof_event(), prof_event()};
  cudaEventRecord(p.a, st);
  g_prof_pending.push_back(p);
  slot = (int)g_prof_pending.size() - 1;
}

ProfScope::~ProfScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (slot < (int)g_prof_pending.size()) cudaEventRecord(g_prof_pending[slot].b, st);
}

}  // namespace fk

extern "C" void fk_profile_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(fk::g_prof_mu);
  fk::g_prof_on = on != 0;
}

extern "C" void fk_profile_reset(void) {
  std::lock_guard<std::mutex> lock(fk::g_prof_mu);
  fk::prof_drain_locked();
  fk::g_prof_classes.clear();
}

extern "C" int32_t fk_profile_count(void) {
  std::lock_guard<std::mutex> lock(fk::g_prof_mu);
  fk::prof_drain_locked();
  return (int32_t)fk::g_prof_classes.size();
}

extern "C" fk_status fk_profile_get(int32_t i, const char** name, int64_t* launches, double* total_ms) {
  std::lock_guard<std::mutex> lock(fk::g_prof_mu);
  fk::prof_drain_locked();
  if (i < 0 || i >= (int32_t)fk::g_prof_classes.size()) return fk::fail(FK_ERR_INVALID_ARG, "profile index");
  if (name) *name = fk::g_prof_classes[i].name.c_str();
  if (launches) *launches = fk::g_prof_classes[i].launches;
  if (total_ms) *total_ms = fk::g_prof_classes[i].ms;
  return FK_OK;
}

extern "C" const char* fk_status_string(fk_status s) {
  switch (s) {
    case FK_OK: return "ok";
    case FK_ERR_INVALID_ARG: return "invalid argument";
    case FK_ERR_INVALID_CONFIG: return "invalid config";
    case FK_ERR_TOKEN_RANGE: return "token id out of range";
    case FK_ERR_CONTEXT_FULL: return "session context full";
    case FK_ERR_NO_DEVICE: return "no sm_103 CUDA device";
    case FK_ERR_CUDA: return "CUDA error";
    case FK_ERR_DEVICE_FLAG: return "device error flag set";
    case FK_ERR_TIMEOUT: return "timeout";
    case FK_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

extern "C" const char* fk_last_error(void) { return fk::g_last_error.c_str(); }

extern "C" fk_status fk_debug_set_op_pipe_fault(int32_t stall_first_stage, int32_t wait_limit_us) {
  if (wait_limit_us < 0) return fk::fail(FK_ERR_INVALID_ARG, "wait_limit_us must be >= 0");
  fk_status s = fk::check_device(nullptr);
  if (s != FK_OK) return s;
  unsigned* ctl = nullptr;
  s = fk::op_control_block(&ctl);
  if (s != FK_OK) return s;
  const unsigned w[2] = {(unsigned)wait_limit_us, stall_first_stage ? 1u : 0u};
  cudaError_t e = cudaMemcpy(ctl + 1, w, sizeof w, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fk::cuda_fail(e, "set op control block");
  return FK_OK;
}

extern "C" const char* fk_version(void) { return "fk 0.1 sm_103a"; }
