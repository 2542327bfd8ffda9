// Exact parallel left fold C_0 = T_0, C_k = fl(C_{k-1} + T_k) (see cr_chain.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace cr {

struct ChainPlan {
  int64_t K = 0, ntiles = 0, seg_cap = 0;
  size_t tsum_off = 0, toff_off = 0, tmax_off = 0, thr_off = 0, lead_off = 0,
         leadsteps_off = 0, done_off = 0, entry_off = 0, entryrec_off = 0, q_off = 0, meta_off = 0,
         nseg_off = 0, segbase_off = 0, segs_off = 0, min_off = 0, tfix_off = 0, tfoff_off = 0,
         rsum_off = 0, roff_off = 0, vsum_off = 0, voff_off = 0, thrs_off = 0,
         thrr_off = 0, thrv_off = 0, misc_off = 0;
  size_t bytes = 0;  // workspace bytes (offsets are relative to the chain's base)
};

// esize: 8 for binary64, 4 for binary32 (whose classification needs more).
ChainPlan plan_chain(int64_t K, size_t esize);

// dst[k] = C_k for k < K. src and dst must not overlap (the fallback re-reads
// src). ws: plan.bytes of 256-byte aligned device memory. With final_out
// (device, one element) C_{K-1} is also written there; dst may then be
// nullptr (a reduction: every step is still validated, no output written).
template <class T>
cudaError_t run_chain(const ChainPlan& plan, const T* src, T* dst, char* ws, cudaStream_t s,
                      T* final_out = nullptr);

// The same fold evaluated one step after the other by one warp (steps
// streamed through shared memory): for short chains, and for binary32 chains
// too long for the parallel evaluation's error bound. dst may equal src or
// be nullptr when final_out is given.
template <class T>
cudaError_t run_serial_chain(const T* src, T* dst, int64_t K, cudaStream_t s,
                             T* final_out = nullptr);

// The block carries fused with a block scan's fix-up: dst[k] = C_k for
// k < K as run_chain (src: the K block totals of which the chain folds the
// first K, dst: K carries) and out[i] = dst[(i >> logB) - 1] op out[i] for
// 2^logB <= i < n, the fix-up running behind the chain's evaluation. On any
// failure of the parallel evaluation *fail (device) is set and out is left
// partly fixed; the serial chain has then rewritten dst, and the caller
// recomputes out's local values and calls run_fixup_again (both conditional
// on *fail, so nothing runs when it is clear). Chains longer than
// kMaxFusedChain are not accepted (their walk could outlast the waits'
// time limit). With out == nullptr the pass is the chain alone (its fill
// overlapping the walk); the serial chain has then already rewritten dst on
// a failure, and nothing else is needed.
// *fused tells whether the cooperative pass ran. When the device refuses
// the cooperative launch (or debug_refuse asks to act as if it had), the
// chain runs as separate passes (the same values in dst) and out is left
// untouched: the caller then applies the carries with a plain fix-up.
// debug_fail: a test hook; a second warp of the walking block sets *fail
// once the walk is half-way, so that the recovery runs.
template <class T>
cudaError_t run_chain_fixup(const ChainPlan& plan, const T* src, T* dst, char* ws, T* out,
                            int64_t n, int logB, cudaStream_t s, const int** fail,
                            bool* fused, bool debug_fail = false, bool debug_refuse = false);
template <class T>
cudaError_t run_fixup_again(T* out, const T* carries, int64_t n, int logB, const int* fail,
                            cudaStream_t s);
constexpr int64_t kMaxFusedChain = int64_t(1) << 26;
constexpr int64_t kMaxFusedChainAlone = int64_t(1) << 28;


}  // namespace cr
