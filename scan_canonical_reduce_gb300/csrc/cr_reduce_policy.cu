// reduce<E>: the root of a named scan expression (P4229R0 on "Canonical
// Parallel Reduction and Scan", Key Design Points: reduce observes the root,
// scan observes the prefixes, reduce<E>(xs) = root_observation(E(xs))).
//   left_fold            ((x0 op x1) op x2) ...  : the last value of the fold
//   pairwise, iterated   tree(x)                 : the shift-reduce tree of all x
//   block_dyadic<B>      C_{K-1}, C_0 = T_0, C_k = C_{k-1} op T_k over the
//                        block trees T_k = tree(x[kB .. kB+B))
// The tree is the canonical reduction with one lane and init -0.0 (the exact
// identity of IEEE addition, so op(-0.0, R) = R); the block trees come from
// the block_dyadic scan's up pass (without its outputs) plus one reduction
// for a ragged last block; the folds are the carry chain in its reduce-only
// form (every step still validated, no prefix written).
#include <cstdint>
#include <cstring>

#include "cr.h"
#include "cr_chain.h"
#include "cr_launch.h"
#include "cr_plan.h"
#include "cr_scan.h"

namespace cr {
namespace {

constexpr int64_t kParallelChainMinR = 1024;  // shorter folds: the serial chain

struct PolicyReducePlan {
  int kind = 0;  // 0 tree, 1 fold of x, 2 block trees then their fold
  ReducePlan tree, tail;
  ScanPlan blocks;  // kind 2: the up pass that yields the block trees
  int64_t n = 0, B = 0, K = 0, Kf = 0;
  bool parallel = false;
  ChainPlan chain;
  size_t tree_ws = 0, tail_ws = 0, blocks_ws = 0, chain_ws = 0, ws_bytes = 0;
};

size_t r256(size_t v) { return (v + 255) & ~size_t(255); }

PolicyReducePlan plan_policy_reduce(int64_t n, cr_policy p, int64_t B, size_t esize) {
  PolicyReducePlan plan;
  plan.n = n;
  size_t off = kHeaderBytes;
  auto chain_for = [&](int64_t K) {
    plan.parallel = K >= kParallelChainMinR;
    if (plan.parallel) {
      plan.chain = plan_chain(K, esize);
      plan.chain_ws = off;
      off += r256(plan.chain.bytes);
    }
  };
  if (p == CR_PAIRWISE || p == CR_ITERATED_PAIRWISE || (p == CR_BLOCK_DYADIC && B >= n)) {
    plan.kind = 0;
    plan.tree = plan_reduce(1, n, 1, 1, n, esize);
    plan.tree_ws = off;
    off += r256(plan.tree.ws_bytes);
  } else if (p == CR_LEFT_FOLD || B == 1) {
    plan.kind = 1;
    chain_for(n);
  } else {
    plan.kind = 2;
    plan.B = B;
    plan.K = (n + B - 1) / B;
    plan.Kf = n / B;
    plan.blocks = plan_scan(1, n, CR_BLOCK_DYADIC, B, esize);
    plan.blocks_ws = off;
    off += r256(plan.blocks.ws_bytes);
    if (plan.K > plan.Kf) {
      plan.tail = plan_reduce(1, n - plan.Kf * B, 1, 1, n - plan.Kf * B, esize);
      plan.tail_ws = off;
      off += r256(plan.tail.ws_bytes);
    }
    chain_for(plan.K);
  }
  plan.ws_bytes = off;
  return plan;
}

template <class T>
cudaError_t run_policy_reduce(const PolicyReducePlan& plan, const T* x, T* out, char* ws,
                              cudaStream_t s) {
  const T minus_zero = -T(0);
  cudaError_t e;
  auto fold = [&](const T* src, int64_t K) -> cudaError_t {
    if (K == 1) return cudaMemcpyAsync(out, src, sizeof(T), cudaMemcpyDeviceToDevice, s);
    if (plan.parallel) return run_chain<T>(plan.chain, src, nullptr, ws + plan.chain_ws, s, out);
    return run_serial_chain<T>(src, nullptr, K, s, out);
  };
  switch (plan.kind) {
    case 0:
      return run_reduce<T>(plan.tree, x, out, minus_zero, ws + plan.tree_ws, s);
    case 1:
      return fold(x, plan.n);
    default: {
      T* totals = nullptr;
      if ((e = run_block_totals<T>(plan.blocks, x, ws + plan.blocks_ws, s, &totals)) !=
          cudaSuccess)
        return e;
      if (plan.K > plan.Kf &&
          (e = run_reduce<T>(plan.tail, x + plan.Kf * plan.B, totals + plan.Kf, minus_zero,
                             ws + plan.tail_ws, s)) != cudaSuccess)
        return e;
      return fold(totals, plan.K);
    }
  }
}

size_t esize_of(cr_dtype dt) { return dt == CR_F64 ? 8 : dt == CR_F32 ? 4 : 0; }

}  // namespace
}  // namespace cr

extern "C" {

size_t cr_reduce_policy_workspace_bytes(int64_t n, cr_policy p, int64_t B, cr_dtype dt) {
  const size_t sz = cr::esize_of(dt);
  if (sz == 0 || n < 1 || !cr::scan_args_ok(p, B)) return 0;
  return cr::plan_policy_reduce(n, p, B, sz).ws_bytes;
}

cr_status cr_reduce_policy(const void* x, int64_t n, cr_policy p, int64_t B, cr_dtype dt,
                           void* out_dev, void* ws, size_t ws_bytes, void* stream) {
  const size_t sz = cr::esize_of(dt);
  if (sz == 0 || n < 1 || x == nullptr || out_dev == nullptr || !cr::scan_args_ok(p, B))
    return CR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) % sz) != 0 ||
      (reinterpret_cast<uintptr_t>(out_dev) % sz) != 0)
    return CR_ERR_INVALID_ARG;
  const cr::PolicyReducePlan plan = cr::plan_policy_reduce(n, p, B, sz);
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % 256) != 0 || ws_bytes < plan.ws_bytes)
    return CR_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return CR_ERR_CUDA;
  cudaError_t e;
  if (dt == CR_F64)
    e = cr::run_policy_reduce<double>(plan, static_cast<const double*>(x),
                                      static_cast<double*>(out_dev), static_cast<char*>(ws), s);
  else
    e = cr::run_policy_reduce<float>(plan, static_cast<const float*>(x),
                                     static_cast<float*>(out_dev), static_cast<char*>(ws), s);
  return e == cudaSuccess ? CR_OK : CR_ERR_CUDA;
}

}  // extern "C"
