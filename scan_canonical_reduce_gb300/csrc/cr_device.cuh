// Device-side building blocks of the canonical reduce / scan kernels.
//
// The expression being evaluated is fixed by "Canonical Parallel Reduction
// and Scan" (github README andyD123/canonical-reduce), P4016R0 Key Design
// Points: the iterative pairwise (shift-reduce) tree. Any schedule may be
// used as long as every node of that tree is formed from the same two
// operands in the same order, so everything here works on ALIGNED perfect
// subtrees (2^k consecutive operands starting at a multiple of 2^k), which
// are nodes of the tree whatever the sequence length, plus a binary-counter
// stack that reproduces the shift-reduce merge order exactly.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace cr {

// ---------------------------------------------------------------- the op
// IEEE-754 addition, round to nearest even, never contracted into an FMA.
__device__ __forceinline__ double add_rn(double a, double b) { return __dadd_rn(a, b); }
__device__ __forceinline__ float add_rn(float a, float b) { return __fadd_rn(a, b); }

template <class T>
__device__ __forceinline__ T ldg(const T* p) { return __ldg(p); }

// Binary64 addition, round to nearest even, evaluated on the integer pipes
// (written from the IEEE-754 definition of the operation). GB300 executes
// only about 1.7 fp64 adds per clock per SM while its integer pipes idle in
// the fp64 kernels; this add was measured as a second add unit: alone it
// runs at half the FP64 pipe's rate, and mixed into the fp64-bound loops it
// cost more issue slots, registers and divergence than it added, so the
// kernels do not use it (it is exposed through cr_add_pairs_int). Operands are
// ordered by magnitude, the smaller significand is aligned with 9 guard bits
// and a sticky bit, added or subtracted, normalised and rounded to nearest
// even. Zero, subnormal, infinite or NaN operands and results that would be
// subnormal or overflow take the hardware add, so every input gives exactly
// the IEEE result.
__device__ __forceinline__ double add_rn_int(double a, double b) {
  constexpr uint64_t kAbs = 0x7FFFFFFFFFFFFFFFull, kFrac = 0x000FFFFFFFFFFFFFull;
  constexpr uint64_t kHid = 0x0010000000000000ull;
  uint64_t ua = (uint64_t)__double_as_longlong(a), ub = (uint64_t)__double_as_longlong(b);
  uint64_t xa = ua & kAbs, xb = ub & kAbs;
  if (xb > xa) {  // |a| >= |b| from here on
    const uint64_t t = ua; ua = ub; ub = t;
    const uint64_t tx = xa; xa = xb; xb = tx;
  }
  const int ea = (int)(xa >> 52), eb = (int)(xb >> 52);
  if (ea == 0x7FF || eb == 0) return __dadd_rn(a, b);  // inf/nan, zero or subnormal
  const uint64_t A = ((xa & kFrac) | kHid) << 9;        // leading one at bit 61
  const uint64_t Bv = ((xb & kFrac) | kHid) << 9;
  const int d = ea - eb;
  uint64_t Bs;
  if (d == 0) Bs = Bv;
  else if (d < 63) Bs = (Bv >> d) | ((Bv << (64 - d)) != 0 ? 1u : 0u);
  else Bs = 1;  // everything below the guard bits: sticky only
  uint64_t S = ((ua ^ ub) >> 63) ? A - Bs : A + Bs;
  int e = ea;
  if (S >> 62) {  // carry out of the addition
    S = (S >> 1) | (S & 1);
    e += 1;
  } else if (!(S >> 61)) {  // cancellation
    if (S == 0) return 0.0;  // x + (-x) = +0 under round to nearest
    const int sh = __clzll((long long)S) - 2;
    S <<= sh;
    e -= sh;
    if (e <= 0) return __dadd_rn(a, b);  // subnormal result
  }
  const uint64_t low = S & 0x1FF;
  S >>= 9;
  if (low > 0x100 || (low == 0x100 && (S & 1))) S += 1;
  if (S >> 53) {
    S >>= 1;
    e += 1;
  }
  if (e >= 0x7FF) return __dadd_rn(a, b);  // overflow
  return __longlong_as_double(
      (long long)((ua & ~kAbs) | ((uint64_t)e << 52) | (S & kFrac)));
}

// Perfect tree over U (a power of two) register values, operands in index
// order: ((v0 op v1) op (v2 op v3)) op ...
template <class T, int U>
__device__ __forceinline__ T perfect_tree(T (&v)[U]) {
#pragma unroll
  for (int s = 1; s < U; s *= 2) {
#pragma unroll
    for (int i = 0; i < U; i += 2 * s) v[i] = add_rn(v[i], v[i + s]);
  }
  return v[0];
}

// ------------------------------------------------- the shift-reduce stack
// A binary counter of perfect subtrees held in registers: slot[lv] is valid
// when bit lv of `count` is set and then holds the perfect tree over the 2^lv
// operands that end at the current position. Pushing a perfect block of 2^a
// operands (count must be a multiple of 2^a, which keeps the block aligned)
// merges it with the occupied slots a, a+1, ... exactly as the shift-reduce
// combines the two topmost partial trees while they are of equal size.
template <class T, int LV>
struct RegStack {
  T slot[LV];
  uint32_t count;

  __device__ __forceinline__ void reset() { count = 0; }

  __device__ __forceinline__ void push(T v, int a) {
    bool done = false;
#pragma unroll
    for (int lv = 0; lv < LV; ++lv) {
      if (!done && lv >= a) {
        if ((count >> lv) & 1u) {
          v = add_rn(slot[lv], v);  // older (left) block first
        } else {
          slot[lv] = v;
          done = true;
        }
      }
    }
    count += 1u << a;
  }

  // Right-nested fold of the stack onto `acc` (the part to the right):
  // smallest block first, acc = block op acc. If !has, the smallest block
  // starts the fold. Returns the new `has`.
  __device__ __forceinline__ bool fold_onto(T& acc, bool has) const {
#pragma unroll
    for (int lv = 0; lv < LV; ++lv) {
      if ((count >> lv) & 1u) {
        acc = has ? add_rn(slot[lv], acc) : slot[lv];
        has = true;
      }
    }
    return has;
  }
};

// ----------------------------------------- perfect trees over smem runs
// In-place pyramid over runs: v(g) for g in [0, F) are values of aligned,
// consecutive equal-size blocks. After the call, v(o) for every o that
// starts a block of F's binary decomposition holds the perfect tree over
// that block (F = 2^b1 + 2^b2 + ..., blocks largest first). A node at level
// k starting at g is written only when g + 2^k <= F, so no node that the
// decomposition needs is overwritten by a larger one.
// `v(g)` addresses one lane's slot g; every thread of the block must call
// this (it synchronises). Threads with g_self < G take part.
template <class T, class Acc>
__device__ __forceinline__ void smem_pyramid(Acc v, int g_self, int G, int F) {
  for (int s = 1; s < G; s *= 2) {
    if (g_self < G && (g_self % (2 * s)) == 0 && g_self + 2 * s <= F) {
      v(g_self) = add_rn(v(g_self), v(g_self + s));
    }
    __syncthreads();
  }
}

// Right-nested fold of the decomposition blocks of F (prepared by
// smem_pyramid) onto acc, smallest block first.
template <class T, class Acc>
__device__ __forceinline__ bool fold_blocks(Acc v, int F, T& acc, bool has) {
  for (int b = 0; (F >> b) != 0; ++b) {
    if ((F >> b) & 1) {
      const int o = F & ~((2 << b) - 1);  // start of the block of size 2^b
      acc = has ? add_rn(v(o), acc) : v(o);
      has = true;
    }
  }
  return has;
}

// Bounded spin helpers for cross-block waits: never wait forever.
constexpr uint32_t kSpinLimit = 1u << 22;

__device__ __forceinline__ void raise_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

}  // namespace cr
