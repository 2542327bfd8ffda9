// C ABI front end of libcr: argument checks, workspace sizing and launch
// dispatch. Declarations and the contract of every call are in include/cr.h.
#include <cstdint>
#include <cstring>

#include "cr.h"
#include "cr_launch.h"
#include "cr_plan.h"
#include "cr_scan.h"

namespace {

size_t esize(cr_dtype dt) {
  switch (dt) {
    case CR_F32: return 4;
    case CR_F64: return 8;
    default: return 0;
  }
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

cr_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || !aligned(ws, 256) || ws_bytes < need) return CR_ERR_WORKSPACE;
  return CR_OK;
}

cr_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CR_OK : CR_ERR_CUDA; }

// A batch of `batch` sequences of `len` elements with strides (es, bs) that
// fills its address range exactly: rows (es = 1, bs = len), columns of a
// level-major array (bs = 1, es = batch), or one sequence or element a row.
bool dense_layout(int64_t len, int64_t batch, int64_t es, int64_t bs) {
  if (len <= 0 || batch <= 0 || len > INT64_MAX / batch) return false;
  if (batch == 1) return len == 1 || es == 1;
  if (len == 1) return bs == 1;
  return (es == 1 && bs == len) || (bs == 1 && es == batch);
}

// Do the byte ranges [a, a + na) and [b, b + nb) meet?
bool ranges_meet(const void* a, size_t na, const void* b, size_t nb) {
  const char* pa = static_cast<const char*>(a);
  const char* pb = static_cast<const char*>(b);
  return pa < pb + nb && pb < pa + na;
}

// Every call starts by clearing the workspace status word (see cr_sync_status).
cudaError_t clear_status(void* ws, cudaStream_t s) {
  return cudaMemsetAsync(ws, 0, sizeof(int), s);
}

cr_status reduce_impl(const void* x, void* out, int64_t batch, int64_t n, int64_t es,
                      int64_t bs, int32_t L, const void* init_host, cr_dtype dt, void* ws,
                      size_t ws_bytes, void* stream) {
  const size_t sz = esize(dt);
  if (sz == 0 || n < 0 || batch < 0 || L < 1 || init_host == nullptr) return CR_ERR_INVALID_ARG;
  if (es < 0 || bs < 0) return CR_ERR_INVALID_ARG;
  if (batch > 0 && out == nullptr) return CR_ERR_INVALID_ARG;
  if (batch > 0 && n > 0 && x == nullptr) return CR_ERR_INVALID_ARG;
  if ((x && !aligned(x, sz)) || (out && !aligned(out, sz))) return CR_ERR_INVALID_ARG;
  // several sequences over one dense block of memory: the results must not
  // land on inputs that another sequence may still read
  if (batch >= 2 && n > 0 && dense_layout(n, batch, es, bs) &&
      ranges_meet(x, (size_t)(n * batch) * sz, out, (size_t)batch * sz))
    return CR_ERR_INVALID_ARG;
  const cr::ReducePlan plan = cr::plan_reduce(batch, n, L, es, bs, sz);
  const cr_status ws_ok = check_ws(ws, ws_bytes, plan.ws_bytes);
  if (ws_ok != CR_OK) return ws_ok;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = clear_status(ws, s);
  if (e != cudaSuccess) return CR_ERR_CUDA;
  char* w = static_cast<char*>(ws);
  if (dt == CR_F64) {
    double init;
    std::memcpy(&init, init_host, sizeof(init));
    e = cr::run_reduce<double>(plan, static_cast<const double*>(x), static_cast<double*>(out),
                               init, w, s);
  } else {
    float init;
    std::memcpy(&init, init_host, sizeof(init));
    e = cr::run_reduce<float>(plan, static_cast<const float*>(x), static_cast<float*>(out),
                              init, w, s);
  }
  return from_cuda(e);
}

}  // namespace

extern "C" {

size_t cr_reduce_workspace_bytes(int64_t n, int32_t L, cr_dtype dt) {
  if (esize(dt) == 0 || n < 0 || L < 1) return 0;
  return cr::plan_reduce(1, n, L, 1, n, esize(dt)).ws_bytes;
}

cr_status cr_reduce(const void* x, int64_t n, int32_t L, const void* init_host, cr_dtype dt,
                    void* out_dev, void* ws, size_t ws_bytes, void* stream) {
  if (out_dev == nullptr) return CR_ERR_INVALID_ARG;
  return reduce_impl(x, out_dev, 1, n, 1, n, L, init_host, dt, ws, ws_bytes, stream);
}

size_t cr_reduce_batched_workspace_bytes(int64_t batch, int64_t n, int32_t L, cr_dtype dt) {
  if (esize(dt) == 0 || n < 0 || batch < 0 || L < 1) return 0;
  // the plan does not depend on the strides
  return cr::plan_reduce(batch, n, L, 1, n, esize(dt)).ws_bytes;
}

cr_status cr_reduce_batched(const void* x, void* out_dev, int64_t batch, int64_t n,
                            int64_t elem_stride, int64_t batch_stride, int32_t L,
                            const void* init_host, cr_dtype dt, void* ws, size_t ws_bytes,
                            void* stream) {
  return reduce_impl(x, out_dev, batch, n, elem_stride, batch_stride, L, init_host, dt, ws,
                     ws_bytes, stream);
}

size_t cr_scan_workspace_bytes(int64_t n, cr_policy p, int64_t B, cr_dtype dt) {
  if (esize(dt) == 0 || n < 0) return 0;
  if (!cr::scan_args_ok(p, B)) return 0;
  return cr::plan_scan(1, n, p, B, esize(dt)).ws_bytes;
}

size_t cr_scan_batched_workspace_bytes(int64_t batch, int64_t n, cr_policy p, int64_t B,
                                       cr_dtype dt) {
  if (esize(dt) == 0 || n < 0 || batch < 0) return 0;
  if (!cr::scan_args_ok(p, B)) return 0;
  return cr::plan_scan(batch, n, p, B, esize(dt)).ws_bytes;
}

static bool mode_ok(int mode) { return mode == CR_EXCLUSIVE || mode == CR_INCLUDE_INITIAL; }

size_t cr_scan_ex_workspace_bytes(int64_t n, cr_policy p, int64_t B, cr_scan_mode mode,
                                  cr_dtype dt) {
  if (esize(dt) == 0 || n < 0 || !mode_ok(mode) || !cr::scan_args_ok(p, B)) return 0;
  return cr::plan_scan(1, n, p, B, esize(dt), mode).ws_bytes;
}

size_t cr_scan_ex_batched_workspace_bytes(int64_t batch, int64_t n, cr_policy p, int64_t B,
                                          cr_scan_mode mode, cr_dtype dt) {
  if (esize(dt) == 0 || n < 0 || batch < 0 || !mode_ok(mode) || !cr::scan_args_ok(p, B))
    return 0;
  return cr::plan_scan(batch, n, p, B, esize(dt), mode).ws_bytes;
}

// Shared by every scan entry point. mode 0 = inclusive (out uses x's
// strides, no init); 1-D calls (contiguous) reject partial overlap of the
// input and output ranges; batched calls with out == x need equal strides.
static cr_status scan_impl(const void* x, void* out, int64_t batch, int64_t n, int64_t es,
                           int64_t bs, int64_t oes, int64_t obs, cr_policy p, int64_t B,
                           int mode, const void* init_host, cr_dtype dt, void* ws,
                           size_t ws_bytes, void* stream, bool contiguous) {
  const size_t sz = esize(dt);
  if (sz == 0 || n < 0 || batch < 0 || !cr::scan_args_ok(p, B)) return CR_ERR_INVALID_ARG;
  if (mode != 0 && (!mode_ok(mode) || init_host == nullptr)) return CR_ERR_INVALID_ARG;
  const int64_t m = n + (mode == CR_INCLUDE_INITIAL ? 1 : 0);
  if (es < 0 || bs < 0 || oes < 0 || obs < 0) return CR_ERR_INVALID_ARG;
  // a zero output stride would send two outputs to one element, and so would
  // equal output strides with two or more sequences of two or more outputs
  // (output (b + 1, k) is output (b, k + 1))
  if (batch > 0 && ((m >= 2 && oes == 0) || (batch >= 2 && m >= 1 && obs == 0)))
    return CR_ERR_INVALID_ARG;
  if (batch >= 2 && m >= 2 && oes == obs) return CR_ERR_INVALID_ARG;
  if (batch > 0 && m > 0 && out == nullptr) return CR_ERR_INVALID_ARG;
  if (batch > 0 && n > 0 && x == nullptr) return CR_ERR_INVALID_ARG;
  if ((x && !aligned(x, sz)) || (out && !aligned(out, sz))) return CR_ERR_INVALID_ARG;
  if (contiguous && x != out && n > 0 && m > 0) {
    const char* a = static_cast<const char*>(x);
    const char* o = static_cast<const char*>(out);
    if (a < o + (size_t)m * sz && o < a + (size_t)n * sz) return CR_ERR_INVALID_ARG;
  }
  if (!contiguous && x == out && x != nullptr && (oes != es || obs != bs))
    return CR_ERR_INVALID_ARG;
  // out != x over dense layouts on both sides: any shared byte is a partial
  // overlap (an output would overwrite an input another sequence reads)
  if (!contiguous && x != out && batch > 0 && n > 0 && m > 0 &&
      dense_layout(n, batch, es, bs) && dense_layout(m, batch, oes, obs) &&
      ranges_meet(x, (size_t)(n * batch) * sz, out, (size_t)(m * batch) * sz))
    return CR_ERR_INVALID_ARG;
  const cr::ScanPlan plan = cr::plan_scan(batch, n, p, B, sz, mode);
  const cr_status ws_ok = check_ws(ws, ws_bytes, plan.ws_bytes);
  if (ws_ok != CR_OK) return ws_ok;
  if (!plan.supported) return CR_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = clear_status(ws, s);
  if (e != cudaSuccess) return CR_ERR_CUDA;
  char* w = static_cast<char*>(ws);
  if (dt == CR_F64) {
    double init = 0.0;
    if (mode != 0) std::memcpy(&init, init_host, sizeof(init));
    e = cr::run_scan<double>(plan, static_cast<const double*>(x), static_cast<double*>(out),
                             es, bs, oes, obs, init, w, s);
  } else {
    float init = 0.0f;
    if (mode != 0) std::memcpy(&init, init_host, sizeof(init));
    e = cr::run_scan<float>(plan, static_cast<const float*>(x), static_cast<float*>(out), es,
                            bs, oes, obs, init, w, s);
  }
  return from_cuda(e);
}

cr_status cr_inclusive_scan(const void* x, void* out, int64_t n, cr_policy p, int64_t B,
                            cr_dtype dt, void* ws, size_t ws_bytes, void* stream) {
  return scan_impl(x, out, 1, n, 1, n, 1, n, p, B, 0, nullptr, dt, ws, ws_bytes, stream, true);
}

cr_status cr_inclusive_scan_batched(const void* x, void* out, int64_t batch, int64_t n,
                                    int64_t elem_stride, int64_t batch_stride, cr_policy p,
                                    int64_t B, cr_dtype dt, void* ws, size_t ws_bytes,
                                    void* stream) {
  return scan_impl(x, out, batch, n, elem_stride, batch_stride, elem_stride, batch_stride, p,
                   B, 0, nullptr, dt, ws, ws_bytes, stream, false);
}

cr_status cr_scan_ex(const void* x, void* out, int64_t n, cr_policy p, int64_t B,
                     cr_scan_mode mode, const void* init_host, cr_dtype dt, void* ws,
                     size_t ws_bytes, void* stream) {
  if (!mode_ok(mode)) return CR_ERR_INVALID_ARG;
  const int64_t m = n + (mode == CR_INCLUDE_INITIAL ? 1 : 0);
  return scan_impl(x, out, 1, n, 1, n, 1, m, p, B, mode, init_host, dt, ws, ws_bytes, stream,
                   true);
}

cr_status cr_scan_ex_batched(const void* x, void* out, int64_t batch, int64_t n,
                             int64_t elem_stride, int64_t batch_stride,
                             int64_t out_elem_stride, int64_t out_batch_stride, cr_policy p,
                             int64_t B, cr_scan_mode mode, const void* init_host, cr_dtype dt,
                             void* ws, size_t ws_bytes, void* stream) {
  if (!mode_ok(mode)) return CR_ERR_INVALID_ARG;
  return scan_impl(x, out, batch, n, elem_stride, batch_stride, out_elem_stride,
                   out_batch_stride, p, B, mode, init_host, dt, ws, ws_bytes, stream, false);
}

static size_t r256(size_t v) { return (v + 255) & ~size_t(255); }

// A host-buffer call's result once its work is enqueued: CR_ERR_CUDA for a
// failed step, else the status word of its workspace (the call's copies out
// are then complete, and a wait that gave up is reported here).
static cr_status host_result(cudaError_t e, const void* ws, cudaStream_t s) {
  int status = 0;
  if (e != cudaSuccess || cr::read_status(ws, s, &status) != cudaSuccess) return CR_ERR_CUDA;
  return status == 0 ? CR_OK : CR_ERR_TIMEOUT;
}

// dev_buf of a host-buffer call: the workspace first (its status word at
// dev_buf itself, where cr_sync_status looks), then the device copies.
size_t cr_inclusive_scan_host_workspace_bytes(int64_t n, cr_policy p, int64_t B, cr_dtype dt) {
  const size_t sz = esize(dt);
  if (sz == 0 || n < 0 || !cr::scan_args_ok(p, B)) return 0;
  return r256(cr::plan_scan(1, n, p, B, sz).ws_bytes) + 2 * r256((size_t)n * sz);
}

cr_status cr_inclusive_scan_host(const void* x_host, void* out_host, int64_t n, cr_policy p,
                                 int64_t B, cr_dtype dt, void* dev_buf, size_t dev_bytes,
                                 void* stream) {
  const size_t sz = esize(dt);
  if (sz == 0 || n < 0 || !cr::scan_args_ok(p, B)) return CR_ERR_INVALID_ARG;
  if (n > 0 && (x_host == nullptr || out_host == nullptr)) return CR_ERR_INVALID_ARG;
  const cr::ScanPlan plan = cr::plan_scan(1, n, p, B, sz);
  const size_t arr = r256((size_t)n * sz);
  const size_t wsb = r256(plan.ws_bytes);
  const cr_status ws_ok = check_ws(dev_buf, dev_bytes, wsb + 2 * arr);
  if (ws_ok != CR_OK) return ws_ok;
  if (!plan.supported) return CR_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(dev_buf);
  char* x_dev = ws + wsb;
  char* out_dev = x_dev + arr;
  if (clear_status(ws, s) != cudaSuccess) return CR_ERR_CUDA;
  cudaError_t e;
  if (dt == CR_F64)
    e = cr::run_scan_host<double>(plan, static_cast<const double*>(x_host),
                                  static_cast<double*>(out_host), reinterpret_cast<double*>(x_dev),
                                  reinterpret_cast<double*>(out_dev), ws, s);
  else
    e = cr::run_scan_host<float>(plan, static_cast<const float*>(x_host),
                                 static_cast<float*>(out_host), reinterpret_cast<float*>(x_dev),
                                 reinterpret_cast<float*>(out_dev), ws, s);
  return host_result(e, ws, s);
}

size_t cr_reduce_host_workspace_bytes(int64_t n, int32_t L, cr_dtype dt) {
  const size_t sz = esize(dt);
  if (sz == 0 || n < 0 || L < 1) return 0;
  return r256(cr::plan_reduce(1, n, L, 1, n, sz).ws_bytes) + 256 + r256((size_t)n * sz);
}

cr_status cr_reduce_host(const void* x_host, int64_t n, int32_t L, const void* init_host,
                         cr_dtype dt, void* out_host, void* dev_buf, size_t dev_bytes,
                         void* stream) {
  const size_t sz = esize(dt);
  if (sz == 0 || n < 0 || L < 1 || init_host == nullptr || out_host == nullptr)
    return CR_ERR_INVALID_ARG;
  if (n > 0 && x_host == nullptr) return CR_ERR_INVALID_ARG;
  const cr::ReducePlan plan = cr::plan_reduce(1, n, L, 1, n, sz);
  const size_t wsb = r256(plan.ws_bytes);
  const cr_status ws_ok = check_ws(dev_buf, dev_bytes, wsb + 256 + r256((size_t)n * sz));
  if (ws_ok != CR_OK) return ws_ok;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(dev_buf);
  char* out_dev = ws + wsb;
  char* x_dev = out_dev + 256;
  if (clear_status(ws, s) != cudaSuccess) return CR_ERR_CUDA;
  cudaError_t e;
  if (dt == CR_F64) {
    double init;
    std::memcpy(&init, init_host, sizeof(init));
    e = cr::run_reduce_host<double>(plan, static_cast<const double*>(x_host),
                                    reinterpret_cast<double*>(x_dev),
                                    reinterpret_cast<double*>(out_dev), init, ws, s, n);
  } else {
    float init;
    std::memcpy(&init, init_host, sizeof(init));
    e = cr::run_reduce_host<float>(plan, static_cast<const float*>(x_host),
                                   reinterpret_cast<float*>(x_dev),
                                   reinterpret_cast<float*>(out_dev), init, ws, s, n);
  }
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_host, out_dev, sz, cudaMemcpyDeviceToHost, s);
  return host_result(e, ws, s);
}

cr_status cr_sync_status(void* ws, void* stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return CR_ERR_CUDA;
  if (ws == nullptr) return CR_ERR_WORKSPACE;
  int status = 0;
  if (cr::read_status(ws, s, &status) != cudaSuccess) return CR_ERR_CUDA;
  return status == 0 ? CR_OK : CR_ERR_TIMEOUT;
}

const char* cr_status_string(cr_status s) {
  switch (s) {
    case CR_OK: return "ok";
    case CR_ERR_INVALID_ARG: return "invalid argument";
    case CR_ERR_UNSUPPORTED: return "unsupported request";
    case CR_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case CR_ERR_CUDA: return "CUDA error";
    case CR_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    default: return "unknown status";
  }
}

int cr_version(void) { return 100; }

void cr_debug_skip_publish(int64_t tile) { cr::set_debug_skip_publish(tile); }
void cr_debug_fused_fixup(int mode) { cr::set_debug_fused_mode(mode); }

}  // extern "C"
