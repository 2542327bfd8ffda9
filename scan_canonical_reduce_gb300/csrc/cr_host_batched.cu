// Host-buffer forms of the batched reduce and the batched inclusive scan
// (contract in include/cr.h): x and out in host memory, a caller-owned
// device buffer for their device copies and the workspace.
//
// The batch is cut into groups of whole sequences. Group g is copied in on
// the host pipeline's copy stream, computed on the caller's stream once it
// has arrived, and copied out on the pipeline's second copy stream once it
// is computed, so that the transfers of one group overlap the kernels and
// transfers of its neighbours. Each group is an independent batched call on
// its sequences: the same kernels, the same results as the device form.
//
// Host layouts: a batch whose sequences are contiguous (elem_stride 1, rows
// at batch_stride >= n) or whose elements k of all sequences are contiguous
// (batch_stride 1, levels at elem_stride >= batch: columns of a level-major
// array). A group is then one rectangle of host memory, moved by one 2-D
// copy into a dense device layout (rows of n, or levels of `batch`).
#include <cstdint>
#include <cstring>
#include <functional>
#include <mutex>

#include "cr.h"
#include "cr_launch.h"
#include "cr_plan.h"
#include "cr_scan.h"

namespace {

size_t esize(cr_dtype dt) { return dt == CR_F64 ? 8 : (dt == CR_F32 ? 4 : 0); }
size_t r256(size_t v) { return (v + 255) & ~size_t(255); }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

enum Layout { kNone, kRows, kCols };

Layout layout_of(int64_t batch, int64_t n, int64_t es, int64_t bs) {
  if (batch == 1) return es == 1 || n <= 1 ? kRows : (es >= 1 ? kCols : kNone);
  if (n == 1) return bs >= 1 ? kRows : kNone;
  if (es == 1 && bs >= n) return kRows;
  if (bs == 1 && es >= batch) return kCols;
  return kNone;
}

// About 16 MB of input a group, 1 to 16 groups, at most one a sequence.
int64_t group_count(int64_t batch, int64_t n, size_t sz) {
  const double bytes = (double)batch * (double)n * (double)sz;
  int64_t g = (int64_t)(bytes / (16.0 * (1 << 20)));
  if (g < 1) g = 1;
  if (g > 16) g = 16;
  if (g > batch) g = batch;
  return g;
}

void group_range(int64_t batch, int64_t G, int64_t g, int64_t& b0, int64_t& b1) {
  b0 = batch * g / G;
  b1 = batch * (g + 1) / G;
}

// The dense device layout of a group: base offset (elements) and strides.
struct DevView {
  int64_t off, es, bs;
};
DevView dev_view(Layout lay, int64_t batch, int64_t n, int64_t b0) {
  if (lay == kRows) return DevView{b0 * n, 1, n};
  return DevView{b0, batch, 1};
}

// One group's rectangle between host (strides es, bs) and the dense device
// layout, `len` elements a sequence.
cudaError_t copy_group(void* dst, const void* src, Layout lay, int64_t batch, int64_t len,
                       int64_t es, int64_t bs, int64_t b0, int64_t b1, size_t sz, bool to_dev,
                       cudaStream_t st) {
  const int64_t nb = b1 - b0;
  if (nb <= 0 || len <= 0) return cudaSuccess;
  char* d = static_cast<char*>(dst);
  const char* s = static_cast<const char*>(src);
  size_t width, height, hpitch, dpitch;
  int64_t hoff, doff;  // elements
  if (lay == kRows) {  // nb rows of len elements
    width = (size_t)len * sz;
    height = (size_t)nb;
    hpitch = (size_t)(nb > 1 ? bs : len) * sz;
    dpitch = (size_t)len * sz;
    hoff = b0 * bs;
    doff = b0 * len;
  } else {  // len levels of nb elements
    width = (size_t)nb * sz;
    height = (size_t)len;
    hpitch = (size_t)(len > 1 ? es : batch) * sz;
    dpitch = (size_t)batch * sz;
    hoff = b0;
    doff = b0;
  }
  if (to_dev)
    return cudaMemcpy2DAsync(d + doff * sz, dpitch, s + hoff * sz, hpitch, width, height,
                             cudaMemcpyHostToDevice, st);
  return cudaMemcpy2DAsync(d + hoff * sz, hpitch, s + doff * sz, dpitch, width, height,
                           cudaMemcpyDeviceToHost, st);
}

// The largest workspace any group's plan needs (groups differ by at most
// one sequence).
size_t reduce_group_ws(int64_t batch, int64_t n, int32_t L, size_t sz, int64_t G) {
  size_t w = 0;
  for (int64_t nb : {batch / G, (batch + G - 1) / G}) {
    if (nb < 1) continue;
    // either dense device layout: rows of n, or levels of `batch`
    for (const cr::ReducePlan& pl : {cr::plan_reduce(nb, n, L, 1, n, sz),
                                     cr::plan_reduce(nb, n, L, batch, 1, sz)})
      w = pl.ws_bytes > w ? pl.ws_bytes : w;
  }
  return w > cr::kHeaderBytes ? w : cr::kHeaderBytes;
}
size_t scan_group_ws(int64_t batch, int64_t n, cr_policy p, int64_t B, size_t sz, int64_t G) {
  size_t w = 0;
  for (int64_t nb : {batch / G, (batch + G - 1) / G}) {
    if (nb < 1) continue;
    const size_t b = cr::plan_scan(nb, n, p, B, sz).ws_bytes;  // the plan ignores strides
    w = b > w ? b : w;
  }
  return w > cr::kHeaderBytes ? w : cr::kHeaderBytes;
}

// The pipeline: copies in on pipe.in, group kernels on s, copies out on
// pipe.out, ordered by the pipe's events; returns once out is written.
using GroupFn = std::function<cudaError_t(int64_t, cudaStream_t)>;
cudaError_t pipeline(int64_t G, cudaStream_t s, const GroupFn& copy_in, const GroupFn& compute,
                     const GroupFn& copy_out) {
  cr::HostPipe* pipe = cr::host_pipe();
  if (pipe == nullptr) return cudaErrorInvalidDevice;
  cr::HostPipe& hp = *pipe;
  cudaError_t e;
  if ((e = hp.ensure((int)G)) != cudaSuccess) return e;
  // the caller's stream may hold earlier work on these buffers: start after it
  if ((e = cudaEventRecord(hp.start, s)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(hp.in, hp.start, 0)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(hp.out, hp.start, 0)) != cudaSuccess) return e;
  for (int64_t g = 0; g < G; ++g) {
    if ((e = copy_in(g, hp.in)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(hp.ev_in[g], hp.in)) != cudaSuccess) return e;
  }
  for (int64_t g = 0; g < G; ++g) {
    if ((e = cudaStreamWaitEvent(s, hp.ev_in[g], 0)) != cudaSuccess) return e;
    if ((e = compute(g, s)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(hp.ev_out[g], s)) != cudaSuccess) return e;
  }
  for (int64_t g = 0; g < G; ++g) {
    if ((e = cudaStreamWaitEvent(hp.out, hp.ev_out[g], 0)) != cudaSuccess) return e;
    if ((e = copy_out(g, hp.out)) != cudaSuccess) return e;
  }
  if ((e = cudaStreamSynchronize(hp.out)) != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(hp.in)) != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

// dev_buf of a batched host-buffer call: the workspace first (wsb bytes; its
// status word at dev_buf itself, where cr_sync_status looks), then the device
// copies of x and out.
template <class T>
cudaError_t reduce_batched_host(const T* xh, T* oh, int64_t batch, int64_t n, int64_t es,
                                int64_t bs, Layout lay, int32_t L, T init, char* ws,
                                size_t wsb, cudaStream_t s) {
  const size_t sz = sizeof(T);
  const int64_t G = group_count(batch, n, sz);
  T* xd = reinterpret_cast<T*>(ws + wsb);
  T* od = reinterpret_cast<T*>(ws + wsb + r256((size_t)(batch * n) * sz));
  std::lock_guard<std::mutex> lock(cr::host_pipe_mutex());
  auto in = [&](int64_t g, cudaStream_t st) -> cudaError_t {
    int64_t b0, b1;
    group_range(batch, G, g, b0, b1);
    return copy_group(xd, xh, lay, batch, n, es, bs, b0, b1, sz, true, st);
  };
  auto run = [&](int64_t g, cudaStream_t st) -> cudaError_t {
    int64_t b0, b1;
    group_range(batch, G, g, b0, b1);
    if (b1 <= b0) return cudaSuccess;
    const DevView v = dev_view(lay, batch, n, b0);
    const cr::ReducePlan plan = cr::plan_reduce(b1 - b0, n, L, v.es, v.bs, sz);
    return cr::run_reduce<T>(plan, n > 0 ? xd + v.off : nullptr, od + b0, init, ws, st);
  };
  auto out = [&](int64_t g, cudaStream_t st) -> cudaError_t {
    int64_t b0, b1;
    group_range(batch, G, g, b0, b1);
    if (b1 <= b0) return cudaSuccess;
    return cudaMemcpyAsync(oh + b0, od + b0, (size_t)(b1 - b0) * sz, cudaMemcpyDeviceToHost,
                           st);
  };
  return pipeline(G, s, in, run, out);
}

template <class T>
cudaError_t scan_batched_host(const T* xh, T* oh, int64_t batch, int64_t n, int64_t es,
                              int64_t bs, Layout lay, cr_policy p, int64_t B, char* ws,
                              size_t wsb, cudaStream_t s) {
  const size_t sz = sizeof(T);
  const int64_t G = group_count(batch, n, sz);
  const size_t arr = r256((size_t)(batch * n) * sz);
  T* xd = reinterpret_cast<T*>(ws + wsb);
  T* od = reinterpret_cast<T*>(ws + wsb + arr);
  std::lock_guard<std::mutex> lock(cr::host_pipe_mutex());
  auto in = [&](int64_t g, cudaStream_t st) -> cudaError_t {
    int64_t b0, b1;
    group_range(batch, G, g, b0, b1);
    return copy_group(xd, xh, lay, batch, n, es, bs, b0, b1, sz, true, st);
  };
  auto run = [&](int64_t g, cudaStream_t st) -> cudaError_t {
    int64_t b0, b1;
    group_range(batch, G, g, b0, b1);
    if (b1 <= b0) return cudaSuccess;
    const DevView v = dev_view(lay, batch, n, b0);
    const cr::ScanPlan plan = cr::plan_scan(b1 - b0, n, p, B, sz);
    if (!plan.supported) return cudaErrorNotSupported;
    return cr::run_scan<T>(plan, xd + v.off, od + v.off, v.es, v.bs, v.es, v.bs, T(0), ws, st);
  };
  auto out = [&](int64_t g, cudaStream_t st) -> cudaError_t {
    int64_t b0, b1;
    group_range(batch, G, g, b0, b1);
    return copy_group(oh, od, lay, batch, n, es, bs, b0, b1, sz, false, st);
  };
  return pipeline(G, s, in, run, out);
}

// Byte extent of a host batch (for the overlap check).
size_t extent_bytes(int64_t batch, int64_t n, int64_t es, int64_t bs, size_t sz) {
  return (size_t)((n - 1) * es + (batch - 1) * bs + 1) * sz;
}

bool ranges_meet(const void* a, size_t na, const void* b, size_t nb) {
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

// The call's result once its pipeline has returned: CR_ERR_CUDA for a failed
// step, else the workspace status word (a wait that gave up is reported).
cr_status host_result(cudaError_t e, const void* ws, cudaStream_t s) {
  if (e == cudaErrorNotSupported) return CR_ERR_UNSUPPORTED;
  int status = 0;
  if (e != cudaSuccess || cr::read_status(ws, s, &status) != cudaSuccess) return CR_ERR_CUDA;
  return status == 0 ? CR_OK : CR_ERR_TIMEOUT;
}

}  // namespace

extern "C" {

size_t cr_reduce_batched_host_workspace_bytes(int64_t batch, int64_t n, int32_t L,
                                              cr_dtype dt) {
  const size_t sz = esize(dt);
  if (sz == 0 || batch < 0 || n < 0 || L < 1) return 0;
  if (batch == 0) return cr::kHeaderBytes;
  const int64_t G = group_count(batch, n, sz);
  return r256(reduce_group_ws(batch, n, L, sz, G)) + r256((size_t)(batch * n) * sz) +
         r256((size_t)batch * sz);
}

cr_status cr_reduce_batched_host(const void* x_host, void* out_host, int64_t batch, int64_t n,
                                 int64_t elem_stride, int64_t batch_stride, int32_t L,
                                 const void* init_host, cr_dtype dt, void* dev_buf,
                                 size_t dev_bytes, void* stream) {
  const size_t sz = esize(dt);
  if (sz == 0 || batch < 0 || n < 0 || L < 1 || init_host == nullptr)
    return CR_ERR_INVALID_ARG;
  if (elem_stride < 0 || batch_stride < 0) return CR_ERR_INVALID_ARG;
  if (batch > 0 && out_host == nullptr) return CR_ERR_INVALID_ARG;
  if (batch > 0 && n > 0 && x_host == nullptr) return CR_ERR_INVALID_ARG;
  if ((x_host && !aligned(x_host, sz)) || (out_host && !aligned(out_host, sz)))
    return CR_ERR_INVALID_ARG;
  if (batch > 0 && n > 0 &&
      ranges_meet(x_host, extent_bytes(batch, n, elem_stride, batch_stride, sz), out_host,
                  (size_t)batch * sz))
    return CR_ERR_INVALID_ARG;
  const size_t need = cr_reduce_batched_host_workspace_bytes(batch, n, L, dt);
  if (dev_buf == nullptr || !aligned(dev_buf, 256) || dev_bytes < need) return CR_ERR_WORKSPACE;
  if (batch == 0) return CR_OK;
  const Layout lay = n == 0 ? kRows : layout_of(batch, n, elem_stride, batch_stride);
  if (lay == kNone) return CR_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(dev_buf);
  const size_t wsb = r256(reduce_group_ws(batch, n, L, sz, group_count(batch, n, sz)));
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return CR_ERR_CUDA;
  cudaError_t e;
  if (dt == CR_F64) {
    double init;
    std::memcpy(&init, init_host, sizeof(init));
    e = reduce_batched_host<double>(static_cast<const double*>(x_host),
                                    static_cast<double*>(out_host), batch, n, elem_stride,
                                    batch_stride, lay, L, init, ws, wsb, s);
  } else {
    float init;
    std::memcpy(&init, init_host, sizeof(init));
    e = reduce_batched_host<float>(static_cast<const float*>(x_host),
                                   static_cast<float*>(out_host), batch, n, elem_stride,
                                   batch_stride, lay, L, init, ws, wsb, s);
  }
  return host_result(e, ws, s);
}

size_t cr_inclusive_scan_batched_host_workspace_bytes(int64_t batch, int64_t n, cr_policy p,
                                                      int64_t B, cr_dtype dt) {
  const size_t sz = esize(dt);
  if (sz == 0 || batch < 0 || n < 0 || !cr::scan_args_ok(p, B)) return 0;
  if (batch == 0 || n == 0) return cr::kHeaderBytes;
  const int64_t G = group_count(batch, n, sz);
  return r256(scan_group_ws(batch, n, p, B, sz, G)) + 2 * r256((size_t)(batch * n) * sz);
}

cr_status cr_inclusive_scan_batched_host(const void* x_host, void* out_host, int64_t batch,
                                         int64_t n, int64_t elem_stride, int64_t batch_stride,
                                         cr_policy p, int64_t B, cr_dtype dt, void* dev_buf,
                                         size_t dev_bytes, void* stream) {
  const size_t sz = esize(dt);
  if (sz == 0 || batch < 0 || n < 0 || !cr::scan_args_ok(p, B)) return CR_ERR_INVALID_ARG;
  if (elem_stride < 0 || batch_stride < 0) return CR_ERR_INVALID_ARG;
  if (batch > 0 && n > 0 && (x_host == nullptr || out_host == nullptr))
    return CR_ERR_INVALID_ARG;
  if ((x_host && !aligned(x_host, sz)) || (out_host && !aligned(out_host, sz)))
    return CR_ERR_INVALID_ARG;
  const size_t need = cr_inclusive_scan_batched_host_workspace_bytes(batch, n, p, B, dt);
  if (batch == 0 || n == 0) {
    if (dev_buf == nullptr || !aligned(dev_buf, 256) || dev_bytes < need)
      return CR_ERR_WORKSPACE;
    return CR_OK;
  }
  const Layout lay = layout_of(batch, n, elem_stride, batch_stride);
  if (lay == kNone) return CR_ERR_UNSUPPORTED;  // e.g. a zero stride: outputs would meet
  if (x_host != out_host &&
      ranges_meet(x_host, extent_bytes(batch, n, elem_stride, batch_stride, sz), out_host,
                  extent_bytes(batch, n, elem_stride, batch_stride, sz)))
    return CR_ERR_INVALID_ARG;
  if (dev_buf == nullptr || !aligned(dev_buf, 256) || dev_bytes < need) return CR_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(dev_buf);
  const size_t wsb = r256(scan_group_ws(batch, n, p, B, sz, group_count(batch, n, sz)));
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return CR_ERR_CUDA;
  cudaError_t e;
  if (dt == CR_F64)
    e = scan_batched_host<double>(static_cast<const double*>(x_host),
                                  static_cast<double*>(out_host), batch, n, elem_stride,
                                  batch_stride, lay, p, B, ws, wsb, s);
  else
    e = scan_batched_host<float>(static_cast<const float*>(x_host),
                                 static_cast<float*>(out_host), batch, n, elem_stride,
                                 batch_stride, lay, p, B, ws, wsb, s);
  return host_result(e, ws, s);
}

}  // extern "C"
