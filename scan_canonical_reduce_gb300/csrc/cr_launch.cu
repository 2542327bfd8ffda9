// Launch counting and event-based per-launch timing (see cr_launch.h).
#include <atomic>
#include <mutex>
#include <vector>

#include "cr.h"
#include "cr_launch.h"

namespace cr {
namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_profiling{0};
std::atomic<int> g_profile_only{-1};  // a kernel id, or -1 for every kernel

struct Record {
  int id;
  cudaEvent_t start, stop;
};

std::mutex g_mu;
std::vector<Record> g_records;      // launches recorded since the last collect
std::vector<cudaEvent_t> g_free;    // reusable events

cudaEvent_t take_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

cudaError_t HostPipe::ensure(int chunks) {
  cudaError_t e;
  if (in == nullptr) {
    if ((e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&start, cudaEventDisableTiming)) != cudaSuccess) return e;
  }
  while ((int)ev_in.size() < chunks) {
    cudaEvent_t a, b;
    if ((e = cudaEventCreateWithFlags(&a, cudaEventDisableTiming)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&b, cudaEventDisableTiming)) != cudaSuccess) return e;
    ev_in.push_back(a);
    ev_out.push_back(b);
  }
  return cudaSuccess;
}

namespace {
std::mutex g_pipe_mu;
HostPipe g_pipes[64];
}  // namespace

std::mutex& host_pipe_mutex() { return g_pipe_mu; }

HostPipe* host_pipe() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  return &g_pipes[dev];
}

const char* kernel_name(int id) {
  static const char* names[kKernelCount] = {
      "lane_pass_kernel",      "write_init_kernel",     "scan_up_kernel",
      "scan_down_kernel",      "carry_chain_kernel",    "scan_seq_kernel",
      "chain_tile_sum_kernel", "chain_offsets_kernel",  "chain_prefix_kernel",
      "chain_classify_kernel", "chain_segments_kernel", "chain_walk_kernel",
      "chain_fill_kernel",     "chain_fallback_kernel", "scan_onepass_kernel",
      "scan_local_kernel",     "carry_fixup_kernel",    "scan_pairwise_kernel",
      "apply_init_kernel",     "fill_init_kernel",      "carry_fixup_shift_kernel",
      "scan_seq_block_kernel", "row_reduce_kernel",
      "chain_link_kernel",     "chain_verify_kernel",   "chain_walk_fix_kernel",
      "scan_local_again_kernel", "fixup_again_kernel", "pairwise_tile_prefix_kernel",
      "chain_round_sum_kernel", "scan_seq_left2_kernel"};
  return (id >= 0 && id < kKernelCount) ? names[id] : "unknown";
}

LaunchScope::LaunchScope(int id_, cudaStream_t s) : id(id_), stream(s), slot(-1) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_profiling.load(std::memory_order_relaxed)) return;
  const int only = g_profile_only.load(std::memory_order_relaxed);
  if (only >= 0 && only != id_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  Record r{id_, take_event(), take_event()};
  if (!r.start || !r.stop) return;
  cudaEventRecord(r.start, s);
  g_records.push_back(r);
  slot = (int)g_records.size() - 1;
}

LaunchScope::~LaunchScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (slot < (int)g_records.size()) cudaEventRecord(g_records[slot].stop, stream);
}

cudaError_t read_status(const void* ws, cudaStream_t s, int* status) {
  *status = 0;
  cudaError_t e = cudaMemcpyAsync(status, ws, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e;
}

}  // namespace cr

extern "C" {

uint64_t cr_launch_count(void) { return cr::g_launches.load(); }

void cr_profile_enable(int on) { cr::g_profiling.store(on ? 1 : 0); }

void cr_profile_select(int kernel_id) {
  cr::g_profile_only.store(kernel_id >= 0 && kernel_id < cr::kKernelCount ? kernel_id : -1);
}

int cr_profile_collect(int* kernel_ids, float* ms, int max_records) {
  std::lock_guard<std::mutex> lk(cr::g_mu);
  int n = 0;
  for (const cr::Record& r : cr::g_records) {
    float t = -1.0f;
    if (cudaEventSynchronize(r.stop) == cudaSuccess) cudaEventElapsedTime(&t, r.start, r.stop);
    if (n < max_records) {
      if (kernel_ids) kernel_ids[n] = r.id;
      if (ms) ms[n] = t;
    }
    ++n;
    cr::g_free.push_back(r.start);
    cr::g_free.push_back(r.stop);
  }
  cr::g_records.clear();
  return n;
}

const char* cr_kernel_name(int id) { return cr::kernel_name(id); }

}  // extern "C"
