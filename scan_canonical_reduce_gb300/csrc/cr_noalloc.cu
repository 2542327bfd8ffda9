// cr_reduce_noalloc: the canonical reduction for callers that cannot
// allocate device memory.
//
// Some callers cannot hand libcr a workspace: a plugin running inside a host
// framework that owns every byte of device memory through its own pool, or a
// latency-critical path where a cudaMalloc (which may synchronise the whole
// device) is not acceptable. For them this entry point takes its scratch
// from one file-scope device array of kNoAllocScratchBytes, loaded with the
// library's module on every GPU that uses it and held until the process
// exits. It allocates no device memory and calls no allocating routine.
//
// Host code never passes `g_noalloc_scratch` itself to a kernel: on the host
// that name is only a stand-in for the device symbol. Every call that is not
// being captured into a CUDA graph looks up the symbol's device address with
// cudaGetSymbolAddress (the call's device current) and keeps it; a call made
// while its stream is capturing reuses the address kept for that device, so
// the first call on a device must come before any capture. Looking the
// address up again outside capture keeps it valid after cudaDeviceReset,
// which reloads the module at a new address.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "cr.h"
#include "cr_plan.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per GPU
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.
cr_status scratch_on_current_device(cudaStream_t s, void** ptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CR_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CR_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return CR_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return CR_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  } else if (g_scratch_ptr[dev] == nullptr) {
    return CR_ERR_UNSUPPORTED;  // no call on this device before the capture
  }
  *ptr = g_scratch_ptr[dev];
  return CR_OK;
}

}  // namespace

extern "C" cr_status cr_reduce_noalloc(const void* x, int64_t n, int32_t L,
                                       const void* init_host, cr_dtype dt, void* out_dev,
                                       void* stream) {
  const size_t sz = (dt == CR_F64) ? 8 : (dt == CR_F32) ? 4 : 0;
  if (sz == 0 || n < 0 || L < 1 || init_host == nullptr || out_dev == nullptr)
    return CR_ERR_INVALID_ARG;
  if (n > 0 && x == nullptr) return CR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) % sz) != 0 ||
      (reinterpret_cast<uintptr_t>(out_dev) % sz) != 0)
    return CR_ERR_INVALID_ARG;
  const cr::ReducePlan plan = cr::plan_reduce(1, n, L, 1, n, sz);
  if (plan.ws_bytes > kNoAllocScratchBytes) return CR_ERR_WORKSPACE;  // too large for it
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  const cr_status st = scratch_on_current_device(s, &ws);
  if (st != CR_OK) return st;
  // the array keeps the previous call's contents: clear the status word; the
  // reduce passes initialise every other word they read before reading it
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return CR_ERR_CUDA;
  cudaError_t e;
  if (dt == CR_F64) {
    double init;
    std::memcpy(&init, init_host, sizeof(init));
    e = cr::run_reduce<double>(plan, static_cast<const double*>(x),
                               static_cast<double*>(out_dev), init, static_cast<char*>(ws), s);
  } else {
    float init;
    std::memcpy(&init, init_host, sizeof(init));
    e = cr::run_reduce<float>(plan, static_cast<const float*>(x), static_cast<float*>(out_dev),
                              init, static_cast<char*>(ws), s);
  }
  return e == cudaSuccess ? CR_OK : CR_ERR_CUDA;
}
