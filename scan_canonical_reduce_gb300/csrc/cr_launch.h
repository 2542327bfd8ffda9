// Launch bookkeeping of libcr: every kernel launch goes through launch(),
// which counts it and, while profiling is on, brackets it with a pair of CUDA
// events recorded on the launching stream. Reading the events back gives the
// device duration of each launch without an external profiler.
#pragma once

#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

namespace cr {

enum KernelId : int {
  kKLanePass = 0,
  kKWriteInit,
  kKScanUp,
  kKScanDown,
  kKCarryChain,
  kKScanSeq,
  kKChainTileSum,
  kKChainOffsets,
  kKChainPrefix,
  kKChainClassify,
  kKChainSegments,
  kKChainWalk,
  kKChainFill,
  kKChainFallback,
  kKScanOnePass,
  kKScanLocal,
  kKCarryFixup,
  kKScanPairwise,
  kKApplyInit,
  kKFillInit,
  kKCarryFixupShift,
  kKScanSeqBlock,
  kKRowReduce,
  kKChainLink,
  kKChainVerify,
  kKChainWalkFix,
  kKScanLocalAgain,
  kKFixupAgain,
  kKPairwisePrefix,
  kKChainRoundSum,
  kKScanSeqLeft2,
  kKernelCount
};

const char* kernel_name(int id);

struct LaunchScope {
  LaunchScope(int id, cudaStream_t s);
  ~LaunchScope();
  int id;
  cudaStream_t stream;
  int slot;
};

// Streams and events of the host-buffer pipelines (copies in and out
// overlapped with the passes), one set per device, created on first use and
// kept. A call holds host_pipe_mutex() for its whole duration.
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr;
  std::vector<cudaEvent_t> ev_in, ev_out;
  cudaError_t ensure(int chunks);  // streams, and at least `chunks` event pairs
};
std::mutex& host_pipe_mutex();
// The current device's; nullptr when there is no current device or its index
// is 64 or more (the callers then fail with cudaErrorInvalidDevice).
HostPipe* host_pipe();

// Reads the status word at the start of workspace `ws` once the work before
// it on `s` is done (synchronises s): 0, or the code a bounded device-side
// wait recorded when it gave up.
cudaError_t read_status(const void* ws, cudaStream_t s, int* status);

// Usage: CR_LAUNCH(kKScanUp, stream, kernel<<<grid, block, 0, stream>>>(...));
#define CR_LAUNCH(ID, STREAM, ...)                  \
  do {                                              \
    ::cr::LaunchScope cr_launch_scope_((ID), (STREAM)); \
    __VA_ARGS__;                                    \
  } while (0)

}  // namespace cr
