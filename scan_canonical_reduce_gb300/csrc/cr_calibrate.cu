// Add-rate calibration: the peak throughput of independent round-to-nearest
// adds and the latency of a dependent chain of them, measured with CUDA
// events on the caller's stream. These are the ALU roofline denominators of
// the kernels whose adds, not their memory traffic, bound them.
#include <cstdint>

#include "cr.h"
#include "cr_device.cuh"

namespace cr {
namespace {

template <class T, int K>
__global__ void add_throughput_kernel(T* sink, T b, int iters) {
  T a[K];
#pragma unroll
  for (int k = 0; k < K; ++k) a[k] = T(threadIdx.x) * T(1e-3) + T(k);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int k = 0; k < K; ++k) a[k] = add_rn(a[k], b);
  }
  T s = a[0];
#pragma unroll
  for (int k = 1; k < K; ++k) s = add_rn(s, a[k]);
  sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

template <class T>
__global__ void add_latency_kernel(T* sink, T b, int iters) {
  T a = T(threadIdx.x);
  for (int it = 0; it < iters; ++it) a = add_rn(a, b);
  sink[threadIdx.x] = a;
}

template <class T>
cr_status measure(void* scratch, size_t bytes, cudaStream_t s, double* rate, double* lat) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CR_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CR_ERR_CUDA;
  const int blocks = sms * 8, threads = 256;
  if (bytes < (size_t)blocks * threads * sizeof(T)) return CR_ERR_WORKSPACE;
  T* sink = static_cast<T*>(scratch);
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return CR_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return CR_ERR_CUDA;
  }
  const int iters = sizeof(T) == 8 ? 2048 : 16384;
  add_throughput_kernel<T, 8><<<blocks, threads, 0, s>>>(sink, T(1e-9), 16);  // warm-up
  cudaEventRecord(e0, s);
  add_throughput_kernel<T, 8><<<blocks, threads, 0, s>>>(sink, T(1e-9), iters);
  cudaEventRecord(e1, s);
  float ms = 0.f;
  cr_status st = CR_OK;
  if (cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
    st = CR_ERR_CUDA;
  if (st == CR_OK && rate) *rate = (double)blocks * threads * 8 * iters / (ms * 1e-3);
  const int chain = 1 << 18;
  if (st == CR_OK) {
    cudaEventRecord(e0, s);
    add_latency_kernel<T><<<1, 1, 0, s>>>(sink, T(1e-9), chain);
    cudaEventRecord(e1, s);
    if (cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      st = CR_ERR_CUDA;
    else if (lat)
      *lat = ms * 1e6 / chain;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st == CR_OK && cudaGetLastError() != cudaSuccess) st = CR_ERR_CUDA;
  return st;
}

}  // namespace
}  // namespace cr

namespace cr {
namespace {
__global__ void add_pairs_int_kernel(const double* a, const double* b, double* out, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = add_rn_int(a[i], b[i]);
}
template <int K>
__global__ void add_int_throughput_kernel(double* sink, double b, int iters) {
  double a[K];
#pragma unroll
  for (int k = 0; k < K; ++k) a[k] = 1.0 + double(threadIdx.x) * 1e-3 + double(k);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int k = 0; k < K; ++k) a[k] = add_rn_int(a[k], b);
  }
  double s = a[0];
#pragma unroll
  for (int k = 1; k < K; ++k) s = add_rn(s, a[k]);
  sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}
}  // namespace
}  // namespace cr

extern "C" cr_status cr_add_pairs_int(const double* a, const double* b, double* out, int64_t n,
                                      void* stream) {
  if (n < 0 || (n > 0 && (!a || !b || !out))) return CR_ERR_INVALID_ARG;
  if (n == 0) return CR_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t blocks = (n + 255) / 256;
  if (blocks > 0x7fffffffLL) return CR_ERR_INVALID_ARG;
  cr::add_pairs_int_kernel<<<(unsigned)blocks, 256, 0, s>>>(a, b, out, n);
  return cudaGetLastError() == cudaSuccess ? CR_OK : CR_ERR_CUDA;
}

extern "C" cr_status cr_measure_int_add_rate(void* scratch_dev, size_t scratch_bytes,
                                             void* stream, double* adds_per_second) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CR_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CR_ERR_CUDA;
  const int blocks = sms * 8, threads = 256;
  if (!scratch_dev || scratch_bytes < (size_t)blocks * threads * 8) return CR_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  double* sink = static_cast<double*>(scratch_dev);
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return CR_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) { cudaEventDestroy(e0); return CR_ERR_CUDA; }
  const int iters = 512;
  cr::add_int_throughput_kernel<8><<<blocks, threads, 0, s>>>(sink, 1e-9, 8);
  cudaEventRecord(e0, s);
  cr::add_int_throughput_kernel<8><<<blocks, threads, 0, s>>>(sink, 1e-9, iters);
  cudaEventRecord(e1, s);
  float ms = 0.f;
  cr_status st = CR_OK;
  if (cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
    st = CR_ERR_CUDA;
  else if (adds_per_second)
    *adds_per_second = (double)blocks * threads * 8 * iters / (ms * 1e-3);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return st;
}

extern "C" size_t cr_measure_add_peak_scratch_bytes(void) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return (size_t)sms * 8 * 256 * sizeof(double);
}

extern "C" cr_status cr_measure_add_peak(cr_dtype dt, void* scratch_dev, size_t scratch_bytes,
                                         void* stream, double* adds_per_second,
                                         double* dependent_latency_ns) {
  if (scratch_dev == nullptr) return CR_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == CR_F64)
    return cr::measure<double>(scratch_dev, scratch_bytes, s, adds_per_second,
                               dependent_latency_ns);
  if (dt == CR_F32)
    return cr::measure<float>(scratch_dev, scratch_bytes, s, adds_per_second,
                              dependent_latency_ns);
  return CR_ERR_INVALID_ARG;
}
