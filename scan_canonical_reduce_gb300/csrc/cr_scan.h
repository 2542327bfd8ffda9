// Host-side launch plans of the scan kernels (see cr_scan.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "cr.h"
#include "cr_chain.h"
#include "cr_plan.h"

namespace cr {

constexpr int kMaxLevels = 40;  // global pyramid levels (tiles up to 2^39)

// Kernel arguments of the tiled 1-D scan passes (passed by value).
struct ScanArgs {
  int64_t n;
  int64_t full_tiles;        // tiles of 2048 elements that are complete
  int32_t logB;              // log2 of the block size; 62 = one block
  int32_t pyr_levels;        // global pyramid levels kept (level 0: tile aggregates)
  int32_t carry;             // block_dyadic: apply C_{k-1}
  int32_t totals_level;      // block totals: 0 in-thread, p > 0 tile pyramid level, -1 global
  int32_t emit_last;         // shifted output of n + 1 entries: also write out[n]
  int64_t tile_base;         // tile index of blockIdx.x == 0 (chunked launches)
  int64_t tile_end;          // up pass: one past the last tile of the launch
  int64_t pyr_off[kMaxLevels];  // element offset of each pyramid level
  int64_t cnt_off[kMaxLevels];  // offset of each level's arrival counters
};

struct ScanPlan {
  // kInitOnly: include_initial of empty sequences (out[0] = init only)
  enum Kind { kEmpty, kInitOnly, kPerSequence, kChainOnly, kTiled };
  // tiled 1-D scans: one pass (iterated_pairwise), local scan + carry
  // fix-up (block_dyadic, B <= 2048), up/down passes (block_dyadic, B > 2048)
  enum Mode { kOnePass, kLocalFixup, kUpDown };
  Mode mode = kOnePass;
  // 0: inclusive; CR_EXCLUSIVE / CR_INCLUDE_INITIAL: out[0] = init,
  // out[k] = init op y[k-1] for k < m (m = n or n + 1)
  int out_mode = 0;
  int64_t m = 0;             // outputs per sequence
  bool supported = false;
  Kind kind = kEmpty;
  int64_t batch = 0, n = 0;
  cr_policy policy = CR_LEFT_FOLD;
  int64_t B = 0;
  int stack_levels = 0;      // per-sequence kernel
  int logB = 62;
  int64_t n_tiles = 0, full_tiles = 0;
  int pyr_levels = 0;
  int64_t pyr_off[kMaxLevels] = {};
  int64_t cnt_off[kMaxLevels] = {};
  size_t pyr_ws = 0, cnt_ws = 0, cnt_bytes = 0;
  size_t ypre_ws = 0;        // pairwise: Y_b = W(2048 b) of every complete tile
  // pairwise, binary64: each thread's quad node x[8t..8t+4) and aggregate,
  // written by the up pass and read by the down-sweep (0: none)
  size_t quad_ws = 0;
  size_t tpyr_ws = 0;        // and each full tile's pyramid levels 1 .. 8
  size_t ready_ws = 0, tilectr_ws = 0;  // one pass: node ready flags, tile counter
  size_t zero_ws = 0, zero_bytes = 0;   // cleared once per call
  int64_t K = 0;             // blocks (block_dyadic)
  int totals_level = -1;
  size_t totals_ws = 0, carries_ws = 0;
  // left folds (block carries, 1-D left_fold) longer than this use the
  // exact parallel chain; shorter ones the serial chain kernel
  bool parallel_chain = false;
  ChainPlan chain;
  size_t chain_ws = 0;
  size_t copy_ws = 0;        // 1-D left_fold in place (or shifted): private copy of x
  int64_t chain_n = 0;       // 1-D left_fold: elements the chain folds
  size_t ws_bytes = kHeaderBytes;
};

bool scan_args_ok(cr_policy p, int64_t B);

// Test hook: the one-pass scan's tile with this index does not publish its
// aggregate, so the tiles that need it exhaust their bounded waits and report
// CR_ERR_TIMEOUT (-1 = off).
int64_t debug_skip_publish();
void set_debug_skip_publish(int64_t tile);
// Test hook for the fused carry fix-up: 0 fused where it is used by default
// (B <= 16), 1 the separate chain and fix-up passes, 2 fused for every B
// with a failure raised half-way through the walk (the recovery passes then
// run), 3 fused for every B.
bool fused_fixup_disabled();
bool debug_fused_fail();
bool fused_fixup_forced();
void set_debug_fused_mode(int mode);
// out_mode: 0 inclusive, CR_EXCLUSIVE or CR_INCLUDE_INITIAL.
ScanPlan plan_scan(int64_t batch, int64_t n, cr_policy p, int64_t B, size_t esize,
                   int out_mode = 0);

// Batched scans read x[b*batch_stride + i*elem_stride] and write
// out[b*out_batch_stride + k*out_elem_stride]; init is used by the shifted
// modes only.
template <class T>
cudaError_t run_scan(const ScanPlan& plan, const T* x, T* out, int64_t elem_stride,
                     int64_t batch_stride, int64_t out_elem_stride, int64_t out_batch_stride,
                     T init, char* ws, cudaStream_t s);

// The same inclusive 1-D scan with x and out in host memory: the copies and
// the kernels are pipelined in chunks of tiles over three streams (copy in,
// compute, copy out, ordered by events), so that the transfers overlap the
// passes. x_dev and out_dev: device buffers of n elements; ws as for
// run_scan. Returns when out is written (the streams are synchronised).
template <class T>
cudaError_t run_scan_host(const ScanPlan& plan, const T* x_host, T* out_host, T* x_dev,
                          T* out_dev, char* ws, cudaStream_t s);

// The trees T_k = tree(x[kB .. (k+1)B)) of the n / B complete blocks, for
// reduce<block_dyadic>: the scan's up pass without its outputs. plan =
// plan_scan(1, n, CR_BLOCK_DYADIC, B, sizeof(T)) with n >= B > 1; the values
// land in the plan's totals buffer (K = ceil(n / B) slots, the last one left
// for a ragged block), whose address goes to *totals_out.
template <class T>
cudaError_t run_block_totals(const ScanPlan& plan, const T* x, char* ws, cudaStream_t s,
                             T** totals_out);

}  // namespace cr
