// Host-side launch plans shared by the C ABI front end and the kernels'
// launchers. A plan depends only on the call's sizes, so the workspace size a
// caller queries and the layout a call uses always agree.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

namespace cr {

// Bytes at the start of every workspace: a status word (int32) at offset 0,
// counters used by the scan kernels after it.
constexpr size_t kHeaderBytes = 256;

// Where a pass reads its (segment, row, lane) matrix: the caller's x or a
// workspace buffer; strides in elements.
struct MatRef {
  bool in_ws;
  size_t ws_off;
  int64_t seg, row, lane;
};

// Kernel arguments of one reduce pass (passed by value).
struct PassArgs {
  int64_t R;             // full rows at this level
  int64_t r;             // lanes j < r have one more value, in row R
  int64_t L;             // lanes at this level
  int64_t T;             // rows per chunk = G * P
  int64_t C;             // full chunks reduced by leaf blocks
  int64_t n_leaf_items;  // leaf blocks: batch * C * tiles
  int64_t next_seg;      // segment stride of the next level's matrix
  int64_t m;             // lanes in the cross-lane tree (fused final pass)
  int32_t P;             // rows per thread run
  int32_t G;             // runs per lane in a block
  int32_t W;             // lanes per block
  int32_t tiles;         // blocks across the lanes
  int32_t final_pass;    // everything left is tail; no next level
  int32_t fuse_cross;    // final pass also does the cross-lane tree and init
  int32_t first_level;   // no lane accumulator yet
  int64_t item_base;     // first work item of this launch (leaf items, then tail)
};

struct PassPlan {
  PassArgs a;
  MatRef in;
  size_t next_off, acc_off, has_off;
  int64_t grid;
};

struct ReducePlan {
  int64_t batch = 0;
  std::vector<PassPlan> passes;
  size_t ws_bytes = 0;
  // Many contiguous rows whose lane count is one warp's 16-byte vector
  // width (L = 32 * 16 / sizeof(T)) and a multiple of it as length: one warp
  // per row (row_reduce_kernel) when the rows are 16-byte aligned; else the
  // passes above. rows_lv = register-stack levels, 0 = not applicable.
  int rows_lv = 0;
  int64_t rows_P = 0, rows_bs = 0;
};

ReducePlan plan_reduce(int64_t batch, int64_t n, int64_t L, int64_t elem_stride,
                       int64_t batch_stride, size_t esize);

template <class T>
cudaError_t run_reduce(const ReducePlan& plan, const T* x, T* out, T init, char* ws,
                       cudaStream_t s);

// The same from a host buffer x_host (n elements, page-locked for overlap):
// copied into x_dev in groups of the first pass's chunks on the host
// pipeline's copy stream, each group reduced as soon as it has arrived.
// out (device) is written on s; the caller copies it back and synchronises.
template <class T>
cudaError_t run_reduce_host(const ReducePlan& plan, const T* x_host, T* x_dev, T* out, T init,
                            char* ws, cudaStream_t s, int64_t n);

}  // namespace cr
