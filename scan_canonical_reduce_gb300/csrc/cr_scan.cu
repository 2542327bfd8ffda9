// Canonical scan kernels (P4229R0 on "Canonical Parallel Reduction and
// Scan", Summary / Key Design Points): prefix observations of the named
// expressions left_fold, pairwise, iterated_pairwise and block_dyadic<B>.
//
// iterated_pairwise: out[i] = tree(x[0..i]) = N_1 op (N_2 op (... op N_m)),
// N_1..N_m the perfect subtrees over the aligned blocks of the binary
// decomposition of i + 1, largest first. Writing i = (b*256 + t)*8 + e
// (tile b, thread t, element e), the nodes split by bit ranges:
//   out[i] = [tile-level nodes of b] op ([thread-level nodes of t] op w[e]),
// with w[e] the thread-local scan of its 8 elements and each level folded
// from its lowest set bit up (right-nested). A node at level p starting at
// q*2^p is the perfect tree over aligned thread (tile) aggregates.
// pairwise: out[i] = ((N_1 op N_2) op ...) op N_m, the same nodes folded from
// the left (largest first): the up pass builds the node pyramid (binary64:
// keeping each thread's first quad and root and each tile's pyramid), then a
// down-sweep (scan_pairwise_kernel) writes every output.
// block_dyadic<B>: the same restricted to the position inside the block (only
// the bits below log2 B), then out[i] = C_{k-1} op P(i) for blocks k >= 1,
// where C_0 = T_0 and C_k = C_{k-1} op T_k over the block totals T_k.
//
// Passes of a 1-D scan (contiguous x):
//   up    per tile: thread and tile aggregates, block totals of blocks that
//         lie inside a tile; the node pyramid over full tiles is completed
//         by arrival tickets: of two sibling nodes, the block that arrives
//         second computes the parent as left op right (counters only, values
//         never pass through an atomic, nothing waits);
//   chain block_dyadic only: the serial left fold of the block totals - a
//         dependency of the expression itself;
//   down  per tile: local scans, prefix nodes, carry; one write of out.
// Batched / strided scans (e.g. columns of a level-major array, which are
// adjacent in memory) run one thread per sequence with a register
// shift-reduce stack.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "cr_device.cuh"
#include "cr_launch.h"
#include "cr_scan.h"

namespace cr {

constexpr int kScanThreads = 256;
constexpr int kE = 8;                     // elements per thread
constexpr int kTile = kScanThreads * kE;  // 2048 elements per tile
constexpr int kLogE = 3;
constexpr int kLogTile = 11;
constexpr int64_t kParallelChainMin = 1024;  // shorter chains: serial kernel

__device__ __forceinline__ int64_t imin(int64_t a, int64_t b) { return a < b ? a : b; }
__device__ __forceinline__ int64_t imax(int64_t a, int64_t b) { return a > b ? a : b; }

template <int N>
struct Log2 {
  static constexpr int value = 1 + Log2<N / 2>::value;
};
template <>
struct Log2<1> {
  static constexpr int value = 0;
};

// Thread-local scan of E register values in segments of S (S | E): within a
// segment, w[e] = tree(v[segment start .. e]); agg[s] = tree(segment s).
// The loops unroll completely, so every "is this slot occupied" test is a
// compile-time constant and only the adds of the tree are emitted.
template <class T, int E, int S>
__device__ __forceinline__ void local_scan(const T (&v)[E], T (&w)[E], T (&agg)[E / S]) {
  constexpr int LS = Log2<S>::value;
#pragma unroll
  for (int s = 0; s < E / S; ++s) {
    T slot[LS + 1];
#pragma unroll
    for (int e = 0; e < S; ++e) {
      T c = v[s * S + e];
      bool placed = false;
#pragma unroll
      for (int lv = 0; lv <= LS; ++lv) {
        if (!placed) {
          if ((e >> lv) & 1) {
            c = add_rn(slot[lv], c);  // older block is the left operand
          } else {
            slot[lv] = c;
            placed = true;
          }
        }
      }
      const int n1 = e + 1;
      T acc = T(0);
      bool has = false;
#pragma unroll
      for (int lv = 0; lv <= LS; ++lv) {
        if ((n1 >> lv) & 1) {
          acc = has ? add_rn(slot[lv], acc) : slot[lv];
          has = true;
        }
      }
      w[s * S + e] = acc;
    }
    agg[s] = slot[LS];
  }
}

// The trees of a thread's kE elements only (no prefixes): the perfect tree
// over all kE, whose level log2(S) holds the trees of the segments of S
// (the same nodes local_scan builds). Returns the tree over all kE.
template <class T, int S>
__device__ __forceinline__ T tree_aggs(const T (&v)[kE], T (&agg)[kE / S]) {
  T u[kE];
#pragma unroll
  for (int e = 0; e < kE; ++e) u[e] = v[e];
#pragma unroll
  for (int st = 1; st < kE; st *= 2) {
#pragma unroll
    for (int i = 0; i < kE; i += 2 * st) u[i] = add_rn(u[i], u[i + st]);
    if (2 * st == S) {
#pragma unroll
      for (int s = 0; s < kE / S; ++s) agg[s] = u[s * S];
    }
  }
  if (S == kE) agg[0] = u[0];
  return u[0];
}

// w[e] = nd op w[e] for the thread's elements (nd is the left operand).
template <class T>
__device__ __forceinline__ void apply_node(T nd, T (&w)[kE]) {
#pragma unroll
  for (int e = 0; e < kE; ++e) w[e] = add_rn(nd, w[e]);
}

// The node of lane-index bit q (q < 5) for every lane of the warp. Only the
// lanes whose bit q is set need it (8 adds each); done per lane, half of each
// warp instruction would idle. Instead the lanes pair up across bit q: the
// lane with the bit does its elements 0-3, its partner does elements 4-7 of
// it (operands and results travel by shuffles) - the same adds, in the same
// order, on all 32 lanes. `lvl_node(t_hi)` is the level-q node needed by the
// pair's lane with the bit set. Every lane of the warp must call this.
template <class T, class NodeOf>
__device__ __forceinline__ void apply_lane_bit(int q, int t, NodeOf lvl_node, T (&w)[kE]) {
  const unsigned full = 0xffffffffu;
  const int m = 1 << q;
  const bool hi = (t >> q) & 1;
  const T nd = lvl_node(t | m);
  T x[kE / 2];
#pragma unroll
  for (int e = 0; e < kE / 2; ++e) {
    const T other = __shfl_xor_sync(full, w[kE / 2 + e], m);  // partner's upper half
    x[e] = hi ? w[e] : other;
  }
#pragma unroll
  for (int e = 0; e < kE / 2; ++e) x[e] = add_rn(nd, x[e]);
#pragma unroll
  for (int e = 0; e < kE / 2; ++e) {
    const T back = __shfl_xor_sync(full, x[e], m);  // my upper half, done by the partner
    if (hi) {
      w[e] = x[e];
      w[kE / 2 + e] = back;
    }
  }
}

// A thread's 8 consecutive elements: 16-byte vector accesses when the
// address allows it (the common case), else scalar ones; tails are bounded.
template <class T>
__device__ __forceinline__ void load8(const T* p, int64_t cnt, T (&v)[kE]) {
  if (cnt == kE && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    if (sizeof(T) == 8) {
      const double2* q = reinterpret_cast<const double2*>(p);
#pragma unroll
      for (int k = 0; k < kE / 2; ++k) {
        const double2 d = q[k];
        v[2 * k] = (T)d.x;
        v[2 * k + 1] = (T)d.y;
      }
    } else {
      const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
      for (int k = 0; k < kE / 4; ++k) {
        const float4 d = q[k];
        v[4 * k] = (T)d.x; v[4 * k + 1] = (T)d.y; v[4 * k + 2] = (T)d.z; v[4 * k + 3] = (T)d.w;
      }
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < kE; ++e) v[e] = (e < cnt) ? p[e] : T(0);
}
template <class T>
__device__ __forceinline__ void store8(T* p, int64_t cnt, const T (&v)[kE]) {
  if (cnt == kE && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    if (sizeof(T) == 8) {
      double2* q = reinterpret_cast<double2*>(p);
#pragma unroll
      for (int k = 0; k < kE / 2; ++k) q[k] = make_double2((double)v[2 * k], (double)v[2 * k + 1]);
    } else {
      float4* q = reinterpret_cast<float4*>(p);
#pragma unroll
      for (int k = 0; k < kE / 4; ++k)
        q[k] = make_float4((float)v[4 * k], (float)v[4 * k + 1], (float)v[4 * k + 2],
                           (float)v[4 * k + 3]);
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < kE; ++e)  // unrolled: v stays in registers
    if (e < cnt) p[e] = v[e];
}

// The last valid one of a thread's values (cnt >= 1), without dynamic
// indexing so that the values stay in registers.
template <class T>
__device__ __forceinline__ T last_of(const T (&w)[kE], int64_t cnt) {
  T r = w[0];
#pragma unroll
  for (int e = 1; e < kE; ++e)
    if (e == cnt - 1) r = w[e];
  return r;
}

// Shifted write of a thread's results y[i0 .. i0+cnt) for the exclusive and
// include_initial forms: out[i] = f(y[i - 1]) at the thread's own positions
// (so in-place scans stay correct and vector stores stay aligned), and
// out[0] = init, where f(v) = init op v (kInit) or v (in-block values that a
// fix-up pass completes). y[i0 - 1] is the previous lane's last value
// (shuffle), the previous warp's (shared memory) or, for the tile's first
// thread, tile_prev. With a.emit_last the thread holding y[n - 1] also
// writes out[n] = f(y[n - 1]). Every thread of the block must call this: it
// synchronises the block.
template <class T, bool kInit>
__device__ __forceinline__ void emit_shifted(T* out, int64_t i0, int64_t cnt, const T (&w)[kE],
                                             T tile_prev, T init, const ScanArgs& a,
                                             T* s_last) {
  const unsigned full = 0xffffffffu;
  const int t = threadIdx.x, lane = t & 31, wp = t >> 5;
  const T up = __shfl_up_sync(full, w[kE - 1], 1);
  if (lane == 31) s_last[wp] = w[kE - 1];
  __syncthreads();
  const T prev = lane ? up : (wp ? s_last[wp - 1] : tile_prev);
  T o[kE];
  o[0] = (i0 == 0) ? init : (kInit ? add_rn(init, prev) : prev);
#pragma unroll
  for (int e = 1; e < kE; ++e) o[e] = kInit ? add_rn(init, w[e - 1]) : w[e - 1];
  store8(out + i0, cnt, o);
  if (a.emit_last && cnt > 0 && i0 + cnt == a.n) {
    const T yl = last_of(w, cnt);
    out[a.n] = kInit ? add_rn(init, yl) : yl;
  }
}

// In-block pyramid over the 256 thread aggregates, all levels kept:
// level p (p = 0..8) holds 256 >> p nodes at lvl[lvl_base(p) + q].
__device__ __forceinline__ int lvl_base(int p) {
  return 2 * kScanThreads - ((2 * kScanThreads) >> p);
}

// Levels 1-5 of a warp's nodes depend only on that warp's threads, so they
// are built with warp barriers; levels 6-8 combine warps.
template <class T>
__device__ __forceinline__ void build_tile_pyramid(T* lvl, int t, int full_threads,
                                                   int top = 8) {
  const int lane = t & 31, wp = t >> 5;
  __syncwarp();
  for (int p = 1; p <= (top < 5 ? top : 5); ++p) {
    const int per = 32 >> p;  // level-p nodes per warp
    const int q = wp * per + lane;
    if (lane < per && q < (full_threads >> p))  // complete nodes only
      lvl[lvl_base(p) + q] =
          add_rn(lvl[lvl_base(p - 1) + 2 * q], lvl[lvl_base(p - 1) + 2 * q + 1]);
    __syncwarp();
  }
  __syncthreads();
  for (int p = 6; p <= top; ++p) {
    const int c = full_threads >> p;
    if (t < c)
      lvl[lvl_base(p) + t] =
          add_rn(lvl[lvl_base(p - 1) + 2 * t], lvl[lvl_base(p - 1) + 2 * t + 1]);
    __syncthreads();
  }
}

// The same levels with every level's adds on the lowest threads (level p's
// 256 >> p adds fill whole warps while they can): about 12 warp-wide adds a
// tile instead of 43, for block barriers between the levels. An fp64 warp
// add holds the fp64 pipe as long with one lane active as with 32, so the
// binary64 passes take this form (2^28, block_dyadic<256> local pass 2.43 ->
// 2.18 ms, the others 1-3 % faster); binary32 keeps the warp-local levels
// (its adds are cheap and the barriers cost more: 2-9 % slower packed),
// except in the up pass, which gains either way.
template <class T>
__device__ __forceinline__ void build_tile_pyramid_packed(T* lvl, int t, int full_threads,
                                                          int top = 8) {
  __syncthreads();
  for (int p = 1; p <= top; ++p) {
    const int c = full_threads >> p;  // complete nodes only
    // a loop, not an if: a one-add if body is compiled to a predicated add
    // that every warp issues (and an fp64 warp add holds the pipe with its
    // lanes off as with them on); the loop leaves the warps past c out
    for (int q = t; q < c; q += kScanThreads)
      lvl[lvl_base(p) + q] = add_rn(lvl[lvl_base(p - 1) + 2 * q], lvl[lvl_base(p - 1) + 2 * q + 1]);
    __syncthreads();
  }
}

template <bool kPacked, class T>
__device__ __forceinline__ void tile_pyramid(T* lvl, int t, int full_threads, int top = 8) {
  if (kPacked) build_tile_pyramid_packed(lvl, t, full_threads, top);
  else build_tile_pyramid(lvl, t, full_threads, top);
}

// Two consecutive values of a 16-byte aligned pair (one vector access for
// binary64).
template <class T>
__device__ __forceinline__ void store_pair(T* p, T a, T b) {
  if constexpr (sizeof(T) == 8) {
    *reinterpret_cast<double2*>(p) = make_double2((double)a, (double)b);
  } else {
    p[0] = a;
    p[1] = b;
  }
}
template <class T>
__device__ __forceinline__ void load_pair(const T* p, T& a, T& b) {
  if constexpr (sizeof(T) == 8) {
    const double2 d = __ldg(reinterpret_cast<const double2*>(p));
    a = (T)d.x;
    b = (T)d.y;
  } else {
    a = p[0];
    b = p[1];
  }
}

// ------------------------------------------------------------------ up pass
// A block takes kUpTiles consecutive tiles (the next tile's elements in
// flight while the current tile's tree is built) and writes their
// aggregates; for an aligned group of full tiles it also combines them into
// the pyramid levels above (no tickets: the group is one subtree) and climbs
// by arrival tickets from there, once per block instead of once per tile.
// Binary64: at least 6 blocks per SM (40 registers instead of 53), so that
// more tiles in flight cover the tile pyramid's barriers (2^28 pairwise
// 1.84 -> 1.76 ms; 8 blocks per SM spill and gain less, 8 tiles a block
// nothing). Binary32: 8 blocks per SM (32 registers), as it compiles
// unbounded (a bound of 6 lets it take 40 and runs 14 % slower).
// The tiles a block (2^CR_UP_LOG_TILES) can be overridden at compile time:
// that changes which block forms which node of the pyramid, never a node.
#ifndef CR_UP_LOG_TILES
#define CR_UP_LOG_TILES 2
#endif
constexpr int kLogUpTiles = CR_UP_LOG_TILES;
constexpr int kUpTiles = 1 << kLogUpTiles;

template <class T, int S, bool kQuads = false>
__global__ void __launch_bounds__(kScanThreads, sizeof(T) == 8 ? 6 : 8)
scan_up_kernel(const T* __restrict__ x, T* __restrict__ pyr, int* __restrict__ counters,
               T* __restrict__ totals, ScanArgs a, T* __restrict__ quads,
               T* __restrict__ tpyr) {
  __shared__ T lvl[2 * kScanThreads];
  __shared__ T s_agg[kUpTiles];
  constexpr int NS = kE / S;
  constexpr int LS = Log2<S>::value;
  const int t = threadIdx.x;
  const int64_t b0 = a.tile_base + (int64_t)blockIdx.x * kUpTiles;
  const int64_t b_end = b0 + kUpTiles < a.tile_end ? b0 + kUpTiles : a.tile_end;
  T vn[kE];
  {
    const int64_t i0 = b0 * kTile + (int64_t)t * kE;
    load8(x + i0, imax(0, imin(kE, a.n - i0)), vn);
  }
  for (int64_t b = b0; b < b_end; ++b) {
    const int64_t i0 = b * kTile + (int64_t)t * kE;
    const int64_t cnt = imax(0, imin(kE, a.n - i0));
    const int full_threads = (int)imin(kScanThreads, (a.n - b * kTile) / kE);
    T v[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) v[e] = vn[e];
    if (b + 1 < b_end) {  // the next tile, in flight meanwhile
      const int64_t j0 = i0 + kTile;
      load8(x + j0, imax(0, imin(kE, a.n - j0)), vn);
    }
#pragma unroll
    for (int e = 0; e < kE; ++e)
      if (e >= cnt) v[e] = T(0);
    T agg[NS];
    T tagg;
    if (kQuads) {
      // pairwise (S = kE): the same tree, its first quad and root kept for
      // the down pass, which then needs only the pairs 01 and 45 of its own
      const T p01 = add_rn(v[0], v[1]), p23 = add_rn(v[2], v[3]);
      const T p45 = add_rn(v[4], v[5]), p67 = add_rn(v[6], v[7]);
      const T q03 = add_rn(p01, p23), q47 = add_rn(p45, p67);
      tagg = add_rn(q03, q47);
      store_pair(quads + 2 * (b * kScanThreads + t), q03, tagg);
    } else {
      tagg = tree_aggs<T, S>(v, agg);  // trees only: the prefixes are the down pass's
      if (a.totals_level == 0) {  // blocks of B = S <= kE elements inside a thread
#pragma unroll
        for (int s = 0; s < NS; ++s)
          if ((s + 1) * S <= cnt) totals[(i0 >> LS) + s] = agg[s];
      }
    }
    if (t < full_threads) lvl[t] = tagg;
    tile_pyramid<true>(lvl, t, full_threads);
    // pairwise: a full tile's pyramid levels 1 .. 8 kept for the down-sweep
    if (kQuads && full_threads == kScanThreads && t < kScanThreads - 1)
      tpyr[b * (kScanThreads - 1) + t] = lvl[kScanThreads + t];
    // blocks of kE < B < kTile elements: complete nodes of the tile pyramid
    if (a.totals_level > 0) {
      const int p = a.totals_level;
      if (t < (full_threads >> p)) totals[((b * kTile) >> a.logB) + t] = lvl[lvl_base(p) + t];
    }
    if (t == 0) s_agg[b - b0] = lvl[lvl_base(8)];
    __syncthreads();  // lvl is rebuilt for the next tile
  }
  if (a.pyr_levels == 0 || t != 0) return;

  // tile aggregates = level 0 of the global pyramid
  for (int64_t b = b0; b < b_end && b < a.full_tiles; ++b) pyr[a.pyr_off[0] + b] = s_agg[b - b0];
  const int loc = a.pyr_levels - 1 < kLogUpTiles ? a.pyr_levels - 1 : kLogUpTiles;
  int64_t q;
  int p0;
  T node;
  if (b_end - b0 == kUpTiles && (b0 & (kUpTiles - 1)) == 0 && b_end <= a.full_tiles) {
    // an aligned group of full tiles: its subtree's levels 1 .. loc here
    T cur[kUpTiles];
#pragma unroll
    for (int i = 0; i < kUpTiles; ++i) cur[i] = s_agg[i];
    int width = kUpTiles;
    for (int p = 1; p <= loc; ++p) {
      width >>= 1;
      for (int i = 0; i < width; ++i) {
        cur[i] = add_rn(cur[2 * i], cur[2 * i + 1]);
        pyr[a.pyr_off[p] + (b0 >> p) + i] = cur[i];
      }
    }
    if (width != 1) return;  // the pyramid ends below the group's root
    q = b0 >> loc;
    p0 = loc + 1;
    node = cur[0];
  } else {
    // a partial group: each full tile climbs from level 0
    for (int64_t b = b0; b < b_end && b < a.full_tiles; ++b) {
      int64_t qq = b;
      for (int p = 1; p < a.pyr_levels; ++p) {
        const int64_t parent = qq >> 1;
        if (parent >= (a.full_tiles >> p)) break;  // the parent is not a complete node
        __threadfence();
        const int ticket = atomicAdd(counters + a.cnt_off[p] + parent, 1);
        if (ticket == 0) break;  // the sibling is still running; it will climb
        __threadfence();
        const T left = __ldcg(pyr + a.pyr_off[p - 1] + 2 * parent);
        const T right = __ldcg(pyr + a.pyr_off[p - 1] + 2 * parent + 1);
        pyr[a.pyr_off[p] + parent] = add_rn(left, right);
        qq = parent;
      }
    }
    return;
  }
  // climb by arrival tickets from the group's root
  for (int p = p0; p < a.pyr_levels; ++p) {
    const int64_t parent = q >> 1;
    if (parent >= (a.full_tiles >> p)) break;  // the parent is not a complete node
    __threadfence();
    const int ticket = atomicAdd(counters + a.cnt_off[p] + parent, 1);
    if (ticket == 0) break;  // the sibling is still running; it will climb
    __threadfence();
    const T left = __ldcg(pyr + a.pyr_off[p - 1] + 2 * parent);
    const T right = __ldcg(pyr + a.pyr_off[p - 1] + 2 * parent + 1);
    node = add_rn(left, right);
    pyr[a.pyr_off[p] + parent] = node;
    q = parent;
  }
}

// ---------------------------------------------------------------- down pass
template <class T, int S, bool kShift>
__global__ void __launch_bounds__(kScanThreads)
scan_down_kernel(const T* x, T* out, const T* __restrict__ pyr, const T* __restrict__ carries,
                 ScanArgs a, T init) {
  __shared__ T lvl[2 * kScanThreads];
  __shared__ T tile_nodes[64];
  __shared__ T tile_carry;
  __shared__ T s_last[kScanThreads / 32];
  constexpr int NS = kE / S;
  const int t = threadIdx.x;
  const int64_t b = a.tile_base + blockIdx.x;
  const int64_t i0 = b * kTile + (int64_t)t * kE;
  const int64_t cnt = imax(0, imin(kE, a.n - i0));
  const int full_threads = (int)imin(kScanThreads, (a.n - b * kTile) / kE);
  // global pyramid levels that lie inside a block (bits of b below log2(B/kTile))
  const int tile_bits = (int)imin(a.pyr_levels, imax(0, a.logB - kLogTile));
  const int thread_bits = (int)imin(8, imax(0, a.logB - kLogE));

  if (t < tile_bits && ((b >> t) & 1)) tile_nodes[t] = pyr[a.pyr_off[t] + (b >> t) - 1];
  if (t == 0 && a.carry && a.logB >= kLogTile) {
    const int64_t k = (b * kTile) >> a.logB;  // whole tile in block k
    tile_carry = (k >= 1) ? carries[k - 1] : T(0);
  }

  T v[kE];
  load8(x + i0, cnt, v);
  T w[kE], agg[NS];
  local_scan<T, kE, S>(v, w, agg);
  T tagg;
  if (NS == 1) {
    tagg = agg[0];
  } else {
    T vv[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) vv[e] = v[e];
    tagg = perfect_tree<T, kE>(vv);
  }
  if (t < full_threads) lvl[t] = tagg;
  tile_pyramid<sizeof(T) == 8>(lvl, t, full_threads);  // also publishes tile_nodes/tile_carry

  // thread-level prefix nodes, lowest bit first (right-nested): binary64
  // takes the lane bits with the lanes paired across each bit (every lane of
  // the warp takes part, so none leaves before them), then the warp bits
  auto node_of = [&](int p) { return [&, p](int th) { return lvl[lvl_base(p) + (th >> p) - 1]; }; };
  // (binary32: its adds are cheaper than the pairing's shuffles; each lane
  // applies its own bits)
  const int paired = sizeof(T) == 8 ? 5 : 0;
  for (int p = 0; p < paired && p < thread_bits; ++p) apply_lane_bit(p, t, node_of(p), w);
  if (!kShift && cnt == 0) return;
  for (int p = paired; p < thread_bits; ++p) {
    if (((t >> p) & 1) && cnt > 0) {
      const T nd = lvl[lvl_base(p) + (t >> p) - 1];
      apply_node(nd, w);
    }
  }
  // tile-level prefix nodes, lowest bit first
  for (int p = 0; p < tile_bits; ++p) {
    if (((b >> p) & 1) && cnt > 0) {
      const T nd = tile_nodes[p];
      apply_node(nd, w);
    }
  }
  // block carry: out[i] = C_{k-1} op P(i) for blocks k >= 1
  if (a.carry && cnt > 0) {
    if (a.logB >= kLogTile) {
      if (((b * kTile) >> a.logB) >= 1) {
        const T c = tile_carry;
#pragma unroll
        for (int e = 0; e < kE; ++e) w[e] = add_rn(c, w[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < kE; ++e) {
        const int64_t k = (i0 + e) >> a.logB;
        if (k >= 1 && e < cnt) w[e] = add_rn(ldg(carries + k - 1), w[e]);
      }
    }
  }
  if (!kShift) {
    store8(out + i0, cnt, w);
    return;
  }
  // y[2048 b - 1]: blocks span tiles here (B > 2048). At a block start it is
  // C_{k-1}; else C_{k-1} op P with P = tree(x[kB .. 2048 b)), the in-block
  // tile-level nodes folded right-nested (no carry in block 0).
  T tile_prev = T(0);
  if (t == 0 && b > 0) {
    const int64_t k = (b * kTile) >> a.logB;
    if (((b * kTile) & (((int64_t)1 << a.logB) - 1)) == 0) {
      tile_prev = carries[k - 1];
    } else {
      bool has = false;
      for (int p = 0; p < tile_bits; ++p) {
        if ((b >> p) & 1) {
          tile_prev = has ? add_rn(tile_nodes[p], tile_prev) : tile_nodes[p];
          has = true;
        }
      }
      if (k >= 1) tile_prev = add_rn(tile_carry, tile_prev);
    }
  }
  emit_shifted<T, true>(out, i0, cnt, w, tile_prev, init, a, s_last);
}

// ------------------------------------------- one-pass tile protocol
// Tiles take indices in the order they start (a counter), publish their
// aggregate, climb the node pyramid by arrival tickets (the second of two
// siblings to arrive computes the parent, left op right, and publishes it
// with a ready flag), and only then wait for the nodes of earlier tiles that
// their own prefix needs. Every wait is on tiles that started earlier and
// never wait before publishing, so the waits end; each is still bounded and,
// if it gives up, records CR_ERR_TIMEOUT in the workspace status word.

// Publishes tile b's aggregate as level-0 node b and climbs while this tile
// arrives second (one thread).
template <class T>
__device__ __forceinline__ void publish_and_climb(T node, int64_t b, T* pyr, int* counters,
                                                  int* ready, const ScanArgs& a) {
  pyr[a.pyr_off[0] + b] = node;
  __threadfence();
  atomicExch(ready + a.pyr_off[0] + b, 1);
  int64_t q = b;
  for (int p = 1; p < a.pyr_levels; ++p) {
    const int64_t parent = q >> 1;
    if (parent >= (a.full_tiles >> p)) break;  // the parent is not a complete node
    const int ticket = atomicAdd(counters + a.cnt_off[p] + parent, 1);
    if (ticket == 0) break;  // the sibling is still running; it will climb
    __threadfence();
    const T left = __ldcg(pyr + a.pyr_off[p - 1] + 2 * parent);
    const T right = __ldcg(pyr + a.pyr_off[p - 1] + 2 * parent + 1);
    node = add_rn(left, right);
    pyr[a.pyr_off[p] + parent] = node;
    __threadfence();
    atomicExch(ready + a.pyr_off[p] + parent, 1);
    q = parent;
  }
}

// The published pyramid node q of level p, after a bounded wait for its flag.
template <class T>
__device__ __forceinline__ T wait_node(const T* pyr, const int* ready, int* status,
                                       const ScanArgs& a, int p, int64_t q) {
  const volatile int* f = ready + a.pyr_off[p] + q;
  uint32_t spins = 0;
  while (*f == 0) {
    if (++spins > kSpinLimit) {
      raise_status(status, CR_ERR_TIMEOUT);
      break;
    }
    __nanosleep(64);
  }
  __threadfence();
  return __ldcg(pyr + a.pyr_off[p] + q);
}

// ------------------------------------------- iterated_pairwise, one pass
// 8 blocks per SM (32 registers; a few bytes spilled in the inclusive form,
// about 560 in the shifted one): more tiles in flight cover the
// tile-pyramid barriers and the waits (2^28 fp64 against 5 blocks per SM:
// inclusive 8.28 -> 7.90 ms, exclusive 8.92 -> 8.60 ms).
template <class T, bool kShift>
__global__ void __launch_bounds__(kScanThreads, 8)
scan_onepass_kernel(const T* x, T* out, T* pyr, int* counters, int* ready, int* tile_ctr,
                    int* status, ScanArgs a, int64_t skip_publish, T init) {
  __shared__ T lvl[2 * kScanThreads];
  __shared__ T tile_nodes[64];
  __shared__ T s_last[kScanThreads / 32];
  __shared__ int64_t s_tile;
  const int t = threadIdx.x;
  if (t == 0) s_tile = atomicAdd(tile_ctr, 1);
  __syncthreads();
  const int64_t b = s_tile;
  const int64_t i0 = b * kTile + (int64_t)t * kE;
  const int64_t cnt = imax(0, imin(kE, a.n - i0));
  const int full_threads = (int)imin(kScanThreads, (a.n - b * kTile) / kE);

  T v[kE];
  load8(x + i0, cnt, v);
  T w[kE], agg[1];
  local_scan<T, kE, kE>(v, w, agg);
  if (t < full_threads) lvl[t] = agg[0];
  tile_pyramid<sizeof(T) == 8>(lvl, t, full_threads);

  if (t == 0 && b < a.full_tiles && a.pyr_levels > 0 && b != skip_publish)
    publish_and_climb(lvl[lvl_base(8)], b, pyr, counters, ready, a);

  // thread-level prefix nodes (all bits of t), lowest first; lane bits by
  // pairs of lanes, warp bits (uniform across the warp) directly
  auto node_of = [&](int p) { return [&, p](int th) { return lvl[lvl_base(p) + (th >> p) - 1]; }; };
  for (int p = 0; p < 5; ++p) apply_lane_bit(p, t, node_of(p), w);
  for (int p = 5; p < 8; ++p) {
    if (((t >> p) & 1) && cnt > 0) apply_node(lvl[lvl_base(p) + (t >> p) - 1], w);
  }
  // wait for the tile-level nodes this tile needs (bits of b)
  const int tile_bits = a.pyr_levels;
  if (t < tile_bits && ((b >> t) & 1))
    tile_nodes[t] = wait_node(pyr, ready, status, a, t, (b >> t) - 1);
  __syncthreads();
  if (!kShift && cnt == 0) return;
  if (cnt > 0) {
    for (int p = 0; p < tile_bits; ++p) {
      if ((b >> p) & 1) apply_node(tile_nodes[p], w);
    }
  }
  if (!kShift) {
    store8(out + i0, cnt, w);
    return;
  }
  // y[2048 b - 1] = tree(x[0 .. 2048 b)): the tile-level nodes, right-nested
  T tile_prev = T(0);
  if (t == 0 && b > 0) {
    bool has = false;
    for (int p = 0; p < tile_bits; ++p) {
      if ((b >> p) & 1) {
        tile_prev = has ? add_rn(tile_nodes[p], tile_prev) : tile_nodes[p];
        has = true;
      }
    }
  }
  emit_shifted<T, true>(out, i0, cnt, w, tile_prev, init, a, s_last);
}

// ------------------------------------------------------ pairwise, down pass
// out[i] = W(i + 1), where W(m) folds the perfect subtrees over the aligned
// blocks of the binary decomposition of m from the LEFT:
// W(m) = ((N_1 op N_2) op ...) op N_k, largest block first. Equivalently
// W(m) = W(m - lowbit(m)) op N(lowbit(m), m - lowbit(m)), with W(0) empty:
// one add per output given the node tree (a down-sweep). Per tile b:
// Y_b = W(2048 b) and Y_{b+1} from the tile-level nodes; per warp the thread
// prefixes E_{32w} = W(2048 b + 256 w) from the warp-level nodes; per lane
// E_t = W(2048 b + 8 t) by a down-sweep over the lane bits; per thread
// W(8t + r), r = 1..7, from E_t and its own pairs and quads, and
// W(8t + 8) = E_{t+1}.
// Y_b is the innermost (left-most) operand of every output of tile b, so no
// later fix-up can apply it: the node pyramid over complete tiles is built
// first by the up pass (scan_up_kernel), and this pass only reads it. (A
// single pass that waits for the nodes measured 2.5x slower here: a tile's
// own add work is too short to hide the pyramid's completion latency.)
// Y_b = W(2048 b), b = 1 .. full_tiles: the tile-level nodes of b folded
// left-nested, highest bit first (the prefix every output of tile b starts
// from), one thread a tile, all its nodes' loads issued before the folds.
template <class T>
__global__ void __launch_bounds__(256)
pairwise_tile_prefix_kernel(const T* __restrict__ pyr, T* __restrict__ ypre, ScanArgs a) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x + 1;
  if (b > a.full_tiles) return;
  T nd[kMaxLevels];
#pragma unroll
  for (int p = 0; p < kMaxLevels; ++p)
    if (p < a.pyr_levels && ((b >> p) & 1)) nd[p] = pyr[a.pyr_off[p] + (b >> p) - 1];
  T acc = T(0);
  bool has = false;
#pragma unroll
  for (int p = kMaxLevels - 1; p >= 0; --p) {
    if (p < a.pyr_levels && ((b >> p) & 1)) {
      acc = has ? add_rn(acc, nd[p]) : nd[p];
      has = true;
    }
  }
  ypre[b] = acc;
}

template <class T, bool kShift, bool kQuads = false>
__global__ void __launch_bounds__(kScanThreads, 8)
scan_pairwise_kernel(const T* x, T* out, const T* __restrict__ ypre, ScanArgs a, T init,
                     const T* __restrict__ quads, const T* __restrict__ tpyr) {
  __shared__ T lvl[2 * kScanThreads];
  __shared__ T s_last[kScanThreads / 32];
  __shared__ T s_E[kScanThreads + 1];  // E_t = W(8 t) of the tile; E_256 = Y_{b+1}
  const int t = threadIdx.x;
  const int64_t b = a.tile_base + blockIdx.x;
  const int64_t i0 = b * kTile + (int64_t)t * kE;
  const int64_t cnt = imax(0, imin(kE, a.n - i0));
  const int full_threads = (int)imin(kScanThreads, (a.n - b * kTile) / kE);
  const int64_t b1 = b + 1;
  const bool complete = (b1 <= a.full_tiles);  // its last output is W(2048 (b + 1))

  T v[kE];
  load8(x + i0, cnt, v);
  // a full tile's pyramid levels 1 .. 8, when the up pass kept them
  const bool kept = kQuads && full_threads == kScanThreads;
  T tp = T(0);
  if (kept && t < kScanThreads - 1) tp = ldg(tpyr + b * (kScanThreads - 1) + t);
  // the thread's nodes: pairs, quads, its aggregate (the first quad and the
  // aggregate from the up pass when it kept them)
  T p01, q03, p45, tagg;
  if (kQuads) {
    load_pair(quads + 2 * (b * kScanThreads + t), q03, tagg);
    p01 = add_rn(v[0], v[1]);
    p45 = add_rn(v[4], v[5]);
  } else {
    p01 = add_rn(v[0], v[1]);
    const T p23 = add_rn(v[2], v[3]);
    p45 = add_rn(v[4], v[5]);
    const T p67 = add_rn(v[6], v[7]);
    q03 = add_rn(p01, p23);
    tagg = add_rn(q03, add_rn(p45, p67));
  }
  if (t < full_threads) lvl[t] = tagg;
  if (kept) {
    if (t < kScanThreads - 1) lvl[kScanThreads + t] = tp;
    __syncthreads();
  } else {
    tile_pyramid<sizeof(T) == 8>(lvl, t, full_threads);  // ends with a block barrier
  }

  // warp prefixes E_{32 w}: thread w of warp 0 takes Y_b (the tile prefix,
  // computed once for every tile) and folds the warp bits; thread 8 takes
  // Y_{b+1}
  if (t <= kScanThreads / 32) {
    T acc = T(0);
    bool has = false;
    if (t < kScanThreads / 32) {
      if (b > 0) {  // W(0) is empty
        acc = ypre[b];
        has = true;
      }
      const int th = t * 32;  // first thread of warp t
      for (int p = 7; p >= 5; --p) {
        if ((th >> p) & 1) {
          const T nd = lvl[lvl_base(p) + (th >> p) - 1];
          acc = has ? add_rn(acc, nd) : nd;
          has = true;
        }
      }
    } else if (complete) {
      acc = ypre[b1];
    }
    s_E[t * 32] = acc;  // W(0) is empty; E_256 is used only when complete
  }
  __syncthreads();
  // lane levels, highest first: E_t = E_{t - 2^p} op node_p for the threads
  // whose lowest set bit is 2^p (p < 5), the 256 >> (p + 1) adds of a level
  // on the lowest threads (no early exit: values past the end are computed
  // and never stored)
#pragma unroll
  for (int p = 4; p >= 0; --p) {
    for (int i = t; i < (kScanThreads >> (p + 1)); i += kScanThreads) {  // a loop: see above
      const int tt = (2 * i + 1) << p;
      const T nd = lvl[lvl_base(p) + (tt >> p) - 1];
      s_E[tt] = (b == 0 && tt == (1 << p)) ? nd : add_rn(s_E[tt - (1 << p)], nd);
    }
    __syncthreads();
  }
  const T E = s_E[t];
  const T E1 = s_E[t + 1];

  T w[kE];
  if (b == 0 && t == 0) {  // W(0) is empty
    w[0] = v[0];
    w[1] = p01;
    w[3] = q03;
  } else {
    w[0] = add_rn(E, v[0]);
    w[1] = add_rn(E, p01);
    w[3] = add_rn(E, q03);
  }
  w[2] = add_rn(w[1], v[2]);
  w[4] = add_rn(w[3], v[4]);
  w[5] = add_rn(w[3], p45);
  w[6] = add_rn(w[5], v[6]);
  w[7] = E1;
  if (kShift)  // y[2048 b - 1] = W(2048 b) = Y_b
    emit_shifted<T, true>(out, i0, cnt, w, s_E[0], init, a, s_last);
  else
    store8(out + i0, cnt, w);
}

// ------------------------------- block_dyadic, blocks inside a tile (B <= 2048)
// Pass 1: the in-block iterated_pairwise values P(i) and the block totals T_k.
template <class T, int S, bool kShift>
__device__ __forceinline__ void local_tile(const T* x, T* out, T* __restrict__ totals,
                                           const ScanArgs& a, int64_t b) {
  __shared__ T lvl[2 * kScanThreads];
  __shared__ T s_last[kScanThreads / 32];
  constexpr int NS = kE / S;
  constexpr int LS = Log2<S>::value;
  const int t = threadIdx.x;
  const int64_t i0 = b * kTile + (int64_t)t * kE;
  const int64_t cnt = imax(0, imin(kE, a.n - i0));
  const int full_threads = (int)imin(kScanThreads, (a.n - b * kTile) / kE);
  T v[kE];
  load8(x + i0, cnt, v);
  T w[kE], agg[NS];
  local_scan<T, kE, S>(v, w, agg);
  if (a.totals_level == 0) {  // blocks inside a thread
#pragma unroll
    for (int s = 0; s < NS; ++s)
      if ((s + 1) * S <= cnt) totals[(i0 >> LS) + s] = agg[s];
  }
  if (a.logB > kLogE) {  // blocks span threads: build the tile pyramid
    T tagg = agg[0];
    if (t < full_threads) lvl[t] = tagg;
    tile_pyramid<sizeof(T) == 8>(lvl, t, full_threads, a.logB - kLogE);  // levels inside a block
    const int p = a.logB - kLogE;
    if (t < (full_threads >> p)) totals[((b * kTile) >> a.logB) + t] = lvl[lvl_base(p) + t];
    auto node_of = [&](int q) { return [&, q](int th) { return lvl[lvl_base(q) + (th >> q) - 1]; }; };
    for (int q = 0; q < p && q < 5; ++q) apply_lane_bit(q, t, node_of(q), w);
    for (int q = 5; q < p; ++q)
      if (((t >> q) & 1) && cnt > 0) apply_node(lvl[lvl_base(q) + (t >> q) - 1], w);
  }
  if (kShift)  // out[i + 1] = P(i); a tile starts a block, whose start the fix-up writes
    emit_shifted<T, false>(out, i0, cnt, w, T(0), T(0), a, s_last);
  else
    store8(out + i0, cnt, w);
}

template <class T, int S, bool kShift>
__global__ void __launch_bounds__(kScanThreads)
scan_local_kernel(const T* x, T* out, T* __restrict__ totals, ScanArgs a) {
  local_tile<T, S, kShift>(x, out, totals, a, a.tile_base + blockIdx.x);
}

// Pass 1 again, every tile (grid-stride), when *only_if is set: the
// recovery of the fused carry fix-up, whose failure leaves out partly fixed.
template <class T, int S>
__global__ void __launch_bounds__(kScanThreads)
scan_local_again_kernel(const T* x, T* out, T* __restrict__ totals, ScanArgs a,
                        int64_t n_tiles, const int* only_if) {
  if (*only_if == 0) return;
  for (int64_t b = blockIdx.x; b < n_tiles; b += gridDim.x) {
    local_tile<T, S, false>(x, out, totals, a, b);
    __syncthreads();  // the tile's shared arrays are reused by the next
  }
}

// Pass 2: out[i] = C_{k-1} op P(i) for every element of blocks k >= 1.
// Elements [start, end) with start >= B (block 0 has no carry).
template <class T>
__global__ void __launch_bounds__(256)
carry_fixup_kernel(T* out, const T* __restrict__ carries, int64_t start, int64_t n, int logB) {
  const int64_t i0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * kE) + start;
  if (i0 >= n) return;
  if (i0 + kE <= n && logB >= kLogE) {  // one block for all 8 elements
    const T c = ldg(carries + (i0 >> logB) - 1);
    T v[kE];
    load8(out + i0, kE, v);
#pragma unroll
    for (int e = 0; e < kE; ++e) v[e] = add_rn(c, v[e]);
    store8(out + i0, kE, v);
    return;
  }
  for (int e = 0; e < kE && i0 + e < n; ++e) {
    const int64_t i = i0 + e;
    out[i] = add_rn(ldg(carries + (i >> logB) - 1), out[i]);
  }
}

// Pass 2 of the shifted forms: out holds P(j - 1) at j (the local pass wrote
// it one place right). For 0 <= j < m: out[0] = init; at a block start
// j = kB < n, out[j] = init op C_{k-1} (the end of block k - 1); otherwise
// j - 1 lies in block k = (j - 1) >> logB and
// out[j] = init op (C_{k-1} op P(j - 1)), or init op P(j - 1) in block 0.
template <class T>
__global__ void __launch_bounds__(256)
carry_fixup_shift_kernel(T* out, const T* __restrict__ carries, int64_t n, int64_t m, int logB,
                         T init) {
  const int64_t j0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * kE;
  if (j0 >= m) return;
  const int64_t bmask = ((int64_t)1 << logB) - 1;
  if (j0 + kE <= n && logB >= kLogE) {  // j0 .. j0+7 in one block, j0 the only possible start
    const int64_t k = j0 >> logB;
    const T c = k >= 1 ? ldg(carries + k - 1) : T(0);
    T v[kE];
    load8(out + j0, kE, v);
#pragma unroll
    for (int e = 0; e < kE; ++e) v[e] = add_rn(init, k >= 1 ? add_rn(c, v[e]) : v[e]);
    if ((j0 & bmask) == 0) v[0] = (j0 == 0) ? init : add_rn(init, ldg(carries + k - 1));
    store8(out + j0, kE, v);
    return;
  }
  for (int e = 0; e < kE && j0 + e < m; ++e) {
    const int64_t j = j0 + e;
    if (j == 0) {
      out[0] = init;
    } else if ((j & bmask) == 0 && j < n) {
      out[j] = add_rn(init, ldg(carries + (j >> logB) - 1));
    } else {
      const int64_t k = (j - 1) >> logB;
      const T v = out[j];
      out[j] = add_rn(init, k >= 1 ? add_rn(ldg(carries + k - 1), v) : v);
    }
  }
}

// out[0] = init, out[k] = init op out[k] for 0 < k < m (the shifted left
// fold: the chain wrote y[k - 1] to out[k]).
template <class T>
__global__ void __launch_bounds__(256)
apply_init_kernel(T* out, int64_t m, T init) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= m) return;
  out[k] = (k == 0) ? init : add_rn(init, out[k]);
}

// out[q * stride] = init for q < count (include_initial of empty sequences).
template <class T>
__global__ void __launch_bounds__(256)
fill_init_kernel(T* out, int64_t count, int64_t stride, T init) {
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (q < count) out[q * stride] = init;
}

// ------------------------------------------------ batched: thread per sequence
// Sequence q: element k at x[q*bs + k*es]; inclusive results go to
// out[q*obs + k*oes]. Shifted forms (shift = 1): out[q*obs] = init and
// y[k] goes to position k + 1 as init op y[k], for k + 1 < m. The next
// element is loaded before the current result is stored, so that an
// in-place call (out == x, same strides) reads every element first.
template <class T, int LV>
__global__ void __launch_bounds__(256)
scan_seq_kernel(const T* x, T* out, int64_t batch, int64_t n, int64_t es, int64_t bs,
                int64_t oes, int64_t obs, int policy, int64_t B, int shift, int64_t m, T init) {
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= batch) return;
  const T* xp = x + q * bs;
  T* yp = out + q * obs;
  auto put = [&](int64_t k, T v) {  // the result y[k]
    if (!shift) yp[k * oes] = v;
    else if (k + 1 < m) yp[(k + 1) * oes] = add_rn(init, v);
  };
  T cur = xp[0];
  if (shift) yp[0] = init;
  if (policy == CR_LEFT_FOLD) {
    T acc = cur;
    for (int64_t k = 0; k < n; ++k) {
      const T nxt = (k + 1 < n) ? xp[(k + 1) * es] : T(0);
      if (k > 0) acc = add_rn(acc, cur);
      put(k, acc);
      cur = nxt;
    }
    return;
  }
  const int64_t blk = (policy == CR_BLOCK_DYADIC) ? B : n;
  T carry = T(0);
  for (int64_t k0 = 0; k0 < n; k0 += blk) {
    const int64_t len = imin(blk, n - k0);
    RegStack<T, LV> st;
    st.reset();
    for (int64_t e = 0; e < len; ++e) {
      const int64_t k = k0 + e;
      const T nxt = (k + 1 < n) ? xp[(k + 1) * es] : T(0);
      st.push(cur, 0);
      cur = nxt;
      T acc = T(0);
      if (policy == CR_PAIRWISE) {  // maximal subtrees folded from the left
        bool has = false;
#pragma unroll
        for (int lv = LV - 1; lv >= 0; --lv) {
          if ((st.count >> lv) & 1u) {
            acc = has ? add_rn(acc, st.slot[lv]) : st.slot[lv];
            has = true;
          }
        }
      } else {  // tree(prefix): folded from the top down (right-nested)
        st.fold_onto(acc, false);
      }
      put(k, (k0 == 0) ? acc : add_rn(carry, acc));
    }
    if (policy == CR_BLOCK_DYADIC && k0 + blk < n) {
      T tk = T(0);
      st.fold_onto(tk, false);
      carry = (k0 == 0) ? tk : add_rn(carry, tk);
    }
  }
}

// Batched block_dyadic with B = BB <= 16 (BB > 1) and left_fold (BB = 16,
// kLeft): one thread per sequence, one block of BB levels per step. The BB
// loads of a block are issued together (consecutive threads read
// consecutive columns, so each is a coalesced row), the in-block values come
// from the compile-time tree of local_scan (only its adds, none predicated
// off), then the carry. The next block's loads are issued before this
// block's adds and stores, so they are in flight meanwhile (the left fold
// of 90 x 200,000 binary64: 0.063 -> 0.057 ms). Outputs as in
// scan_seq_kernel; in the shifted forms the stores reach one position
// further, and the next block is already loaded, so in-place calls stay
// correct.
template <class T, int BB, bool kLeft>
__global__ void __launch_bounds__(256)
scan_seq_block_kernel(const T* x, T* out, int64_t batch, int64_t n, int64_t es, int64_t bs,
                      int64_t oes, int64_t obs, int shift, int64_t m, T init) {
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= batch) return;
  const T* xp = x + q * bs;
  T* yp = out + q * obs;
  T v[BB];
#pragma unroll
  for (int e = 0; e < BB; ++e) v[e] = (e < n) ? xp[(int64_t)e * es] : T(0);
  if (shift) yp[0] = init;
  T carry = T(0);
  for (int64_t k0 = 0; k0 < n; k0 += BB) {
    const int64_t len = imin(BB, n - k0);
    T nv[BB];  // the next block of levels, in flight during this one
#pragma unroll
    for (int e = 0; e < BB; ++e) nv[e] = (k0 + BB + e < n) ? xp[(k0 + BB + e) * es] : T(0);
    T w[BB];
    if (kLeft) {
      T acc = (k0 == 0) ? v[0] : add_rn(carry, v[0]);
      w[0] = acc;
#pragma unroll
      for (int e = 1; e < BB; ++e) {
        acc = add_rn(acc, v[e]);
        w[e] = acc;
      }
      carry = acc;  // read only when a full block follows
    } else {
      T agg[1];
      local_scan<T, BB, BB>(v, w, agg);
      if (k0 > 0) {
#pragma unroll
        for (int e = 0; e < BB; ++e) w[e] = add_rn(carry, w[e]);
      }
      carry = (k0 == 0) ? agg[0] : add_rn(carry, agg[0]);
    }
#pragma unroll
    for (int e = 0; e < BB; ++e) {
      if (e < len) {
        const int64_t k = k0 + e;
        if (!shift) yp[k * oes] = w[e];
        else if (k + 1 < m) yp[(k + 1) * oes] = add_rn(init, w[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < BB; ++e) v[e] = nv[e];
  }
}

// The binary64 left fold of columns two at a time (inclusive, adjacent
// columns: batch stride 1 in and out, element strides even, x and out
// 16-byte aligned): thread q folds columns 2q and 2q + 1 with one 16-byte
// load and one 16-byte store per level, half the memory instructions of one
// column a thread, and two independent chains in every thread. The next BB
// levels are loaded while the current BB are folded and stored. BB = 4 (56
// registers, every column of 90 x 200,000 resident at once): 0.056 ->
// 0.050 ms against one column a thread; BB = 2, 8 and 16 (16 without the
// loads ahead) measured 0.054, 0.060 and 0.072 ms.
template <int BB, bool kAhead>
__global__ void __launch_bounds__(256)
scan_seq_left2_kernel(const double* x, double* out, int64_t batch, int64_t n, int64_t es,
                      int64_t oes) {
  const int64_t c0 = 2 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x);
  if (c0 >= batch) return;
  const bool two = c0 + 1 < batch;
  auto load = [&](int64_t k, double& a, double& b) {
    if (two) {
      const double2 d = __ldg(reinterpret_cast<const double2*>(x + k * es + c0));
      a = d.x;
      b = d.y;
    } else {
      a = x[k * es + c0];
      b = 0.0;
    }
  };
  double v0[BB], v1[BB];
#pragma unroll
  for (int e = 0; e < BB; ++e) {
    v0[e] = 0.0;
    v1[e] = 0.0;
    if (e < n) load(e, v0[e], v1[e]);
  }
  double acc0 = 0.0, acc1 = 0.0;
  for (int64_t k0 = 0; k0 < n; k0 += BB) {
    double n0[BB], n1[BB];  // the next BB levels, in flight meanwhile
#pragma unroll
    for (int e = 0; e < BB; ++e) {
      n0[e] = 0.0;
      n1[e] = 0.0;
      if (kAhead && k0 + BB + e < n) load(k0 + BB + e, n0[e], n1[e]);
    }
#pragma unroll
    for (int e = 0; e < BB; ++e) {
      const int64_t k = k0 + e;
      if (k < n) {
        acc0 = k == 0 ? v0[e] : add_rn(acc0, v0[e]);
        acc1 = k == 0 ? v1[e] : add_rn(acc1, v1[e]);
        if (two) *reinterpret_cast<double2*>(out + k * oes + c0) = make_double2(acc0, acc1);
        else out[k * oes + c0] = acc0;
      }
    }
#pragma unroll
    for (int e = 0; e < BB; ++e) {
      v0[e] = n0[e];
      v1[e] = n1[e];
      if (!kAhead && k0 + BB + e < n) load(k0 + BB + e, v0[e], v1[e]);
    }
  }
}

// ---------------------------------------------------------------- planning
namespace {
std::atomic<int64_t> g_skip_publish{-1};
}
int64_t debug_skip_publish() { return g_skip_publish.load(); }
void set_debug_skip_publish(int64_t tile) { g_skip_publish.store(tile); }
namespace {
std::atomic<int> g_fused_mode{0};
}
bool fused_fixup_disabled() { return g_fused_mode.load() == 1; }
bool debug_fused_fail() { return g_fused_mode.load() == 2; }
bool debug_coop_refused() { return g_fused_mode.load() == 4; }
bool fused_fixup_forced() { return g_fused_mode.load() >= 2; }
void set_debug_fused_mode(int mode) { g_fused_mode.store(mode); }

bool scan_args_ok(cr_policy p, int64_t B) {
  switch (p) {
    case CR_LEFT_FOLD:
    case CR_PAIRWISE:
    case CR_ITERATED_PAIRWISE: return true;
    case CR_BLOCK_DYADIC: return B >= 1 && (B & (B - 1)) == 0;
    default: return false;
  }
}

namespace {
int ilog2(int64_t v) {
  int l = 0;
  while ((int64_t(1) << (l + 1)) <= v) ++l;
  return l;
}
size_t round256(size_t v) { return (v + 255) & ~size_t(255); }
}  // namespace

ScanPlan plan_scan(int64_t batch, int64_t n, cr_policy p, int64_t B, size_t esize,
                   int out_mode) {
  ScanPlan plan;
  plan.batch = batch;
  plan.n = n;
  plan.policy = p;
  plan.B = (p == CR_BLOCK_DYADIC) ? B : 0;
  plan.out_mode = out_mode;
  const bool shift = out_mode != 0;
  plan.m = n + (out_mode == CR_INCLUDE_INITIAL ? 1 : 0);
  size_t off = kHeaderBytes;
  plan.supported = true;
  if (batch == 0 || plan.m == 0) {
    plan.kind = ScanPlan::kEmpty;
    plan.ws_bytes = off;
    return plan;
  }
  if (n == 0) {  // include_initial of empty sequences
    plan.kind = ScanPlan::kInitOnly;
    plan.ws_bytes = off;
    return plan;
  }
  const bool block = (p == CR_BLOCK_DYADIC);
  if (batch > 1) {
    const int64_t depth_n = block ? (B < n ? B : n) : n;
    plan.kind = ScanPlan::kPerSequence;
    plan.stack_levels = ilog2(depth_n) + 1;
    plan.supported = (p == CR_LEFT_FOLD) || n < (int64_t(1) << 31);
    plan.ws_bytes = off;
    return plan;
  }
  if (p == CR_LEFT_FOLD || (block && B == 1)) {
    // every element is its own block: the left-fold chain (into out + 1 for
    // the shifted forms, then init applied)
    plan.kind = ScanPlan::kChainOnly;
    plan.chain_n = shift ? plan.m - 1 : n;
    if (plan.chain_n >= kParallelChainMin) {
      plan.parallel_chain = true;
      plan.chain = plan_chain(plan.chain_n, esize);
      plan.chain_ws = off;
      off += round256(plan.chain.bytes);
    }
    if (plan.chain_n > 0 && (plan.parallel_chain || shift)) {
      plan.copy_ws = off;  // used only in place (out == x)
      off += round256((size_t)plan.chain_n * esize);
    }
    plan.ws_bytes = off;
    return plan;
  }
  plan.kind = ScanPlan::kTiled;
  const int logB = block ? ilog2(B) : 62;
  plan.logB = logB;
  plan.n_tiles = (n + kTile - 1) / kTile;
  plan.full_tiles = n / kTile;
  // one pass for binary64 iterated_pairwise, whose adds hide the waits for
  // earlier tiles' pyramid nodes; binary32 (adds far cheaper) and pairwise
  // (2 adds per element) would expose them: node pyramid first instead
  if (p == CR_PAIRWISE || (!block && esize == 4)) plan.mode = ScanPlan::kUpDown;
  else if (!block) plan.mode = ScanPlan::kOnePass;
  else if (logB <= kLogTile) plan.mode = ScanPlan::kLocalFixup;
  else plan.mode = ScanPlan::kUpDown;
  // global node pyramid over complete tiles (one pass, up/down): level l has
  // full_tiles >> l nodes; up/down keeps only the levels inside a block
  int levels = 0;
  if (plan.mode != ScanPlan::kLocalFixup && plan.full_tiles >= 1) {
    levels = ilog2(plan.full_tiles) + 1;
    if (block) levels = std::min(levels, std::max(0, logB - kLogTile + 1));
  }
  plan.pyr_levels = levels;
  if (p == CR_PAIRWISE && levels > 32) plan.supported = false;  // 2^43 elements and more
  int64_t pyr_elems = 0, cnt_elems = 0;
  for (int l = 0; l < levels; ++l) {
    plan.pyr_off[l] = pyr_elems;
    plan.cnt_off[l] = cnt_elems;
    pyr_elems += plan.full_tiles >> l;
    if (l >= 1) cnt_elems += plan.full_tiles >> l;
  }
  plan.pyr_ws = off;
  off += round256((size_t)pyr_elems * esize);
  if (p == CR_PAIRWISE) {
    plan.ypre_ws = off;
    off += round256((size_t)(plan.full_tiles + 1) * esize);
    if (esize == 8) {  // binary64: each thread's first quad and aggregate,
      plan.quad_ws = off;  // and each tile's pyramid levels 1 .. 8
      off += round256((size_t)plan.n_tiles * kScanThreads * 2 * esize);
      plan.tpyr_ws = off;
      off += round256((size_t)plan.n_tiles * (kScanThreads - 1) * esize);
    }
  }
  // arrival counters, ready flags (one pass) and the tile counter: one
  // region cleared by a single memset per call
  plan.zero_ws = off;
  plan.cnt_ws = off;
  plan.cnt_bytes = (size_t)cnt_elems * sizeof(int);
  off += round256(plan.cnt_bytes);
  if (plan.mode == ScanPlan::kOnePass) {
    plan.ready_ws = off;
    off += round256((size_t)pyr_elems * sizeof(int));
    plan.tilectr_ws = off;
    off += 256;
  }
  plan.zero_bytes = off - plan.zero_ws;
  if (block) {
    plan.K = (n + B - 1) / B;
    if (logB <= kLogE) plan.totals_level = 0;            // inside a thread
    else if (logB <= kLogTile) plan.totals_level = logB - kLogE;  // tile pyramid level
    else plan.totals_level = -1;                         // global pyramid level
    plan.totals_ws = off;
    off += round256((size_t)plan.K * esize);
    plan.carries_ws = off;
    off += round256((size_t)plan.K * esize);
    if (plan.K - 1 >= kParallelChainMin) {
      plan.parallel_chain = true;
      plan.chain = plan_chain(plan.K - 1, esize);
      plan.chain_ws = off;
      off += round256(plan.chain.bytes);
    }
  } else {
    plan.totals_level = -1;
  }
  plan.ws_bytes = off;
  return plan;
}

template <class T>
cudaError_t launch_fixup(const ScanPlan& plan, T* out, const T* carries, int64_t start,
                         int64_t end, cudaStream_t s);

// Whether the block carries and the fix-up run as one fused pass: inclusive
// local + fix-up scans whose carries take the parallel chain, for B <= 16,
// where the chain's walk is long enough against the fix-up for the overlap
// to win (2^28 binary64 elements: B = 16 1.43 -> 1.21 ms, B = 8 1.97 ->
// 1.67 ms; at B = 256 and 2048 the fused fix-up streams below the plain
// kernel's rate and the walk is short: 0.79 -> 0.90 ms, 0.70 -> 0.77 ms).
bool fused_fixup_ok(const ScanPlan& plan) {
  if (plan.kind != ScanPlan::kTiled || plan.mode != ScanPlan::kLocalFixup ||
      plan.out_mode != 0 || !plan.parallel_chain || plan.K - 1 > kMaxFusedChain)
    return false;
  if (fused_fixup_disabled()) return false;
  return plan.logB <= 4 || fused_fixup_forced();
}

// The passes of a tiled 1-D scan, each over a range of tiles [t0, t1):
// first (one pass / local / up), middle (the carry chain, once), second
// (fix-up / down / pairwise down-sweep; none for the one pass).
template <class T>
struct Tiled {
  const ScanPlan& plan;
  char* ws;
  T init;
  bool block, shift;
  int S;
  ScanArgs a{};
  T *pyr, *ypre, *totals, *carries, *quads, *tpyr;
  int* counters;
  Tiled(const ScanPlan& p, char* w, T i) : plan(p), ws(w), init(i) {
    block = plan.policy == CR_BLOCK_DYADIC;
    shift = plan.out_mode != 0;
    S = block ? (int)(plan.B < kE ? plan.B : kE) : kE;
    a.n = plan.n;
    a.full_tiles = plan.full_tiles;
    a.logB = plan.logB;
    a.pyr_levels = plan.pyr_levels;
    a.carry = block ? 1 : 0;
    a.totals_level = block ? plan.totals_level : -1;
    a.emit_last = plan.out_mode == CR_INCLUDE_INITIAL ? 1 : 0;
    for (int l = 0; l < kMaxLevels; ++l) {
      a.pyr_off[l] = plan.pyr_off[l];
      a.cnt_off[l] = plan.cnt_off[l];
    }
    pyr = reinterpret_cast<T*>(ws + plan.pyr_ws);
    ypre = reinterpret_cast<T*>(ws + plan.ypre_ws);
    quads = plan.quad_ws ? reinterpret_cast<T*>(ws + plan.quad_ws) : nullptr;
    tpyr = plan.quad_ws ? reinterpret_cast<T*>(ws + plan.tpyr_ws) : nullptr;
    counters = reinterpret_cast<int*>(ws + plan.cnt_ws);
    totals = block ? reinterpret_cast<T*>(ws + plan.totals_ws) : nullptr;
    carries = block ? reinterpret_cast<T*>(ws + plan.carries_ws) : nullptr;
  }
  bool has_second() const { return plan.mode != ScanPlan::kOnePass; }
  cudaError_t prepare(cudaStream_t s) {
    if (plan.n_tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (plan.zero_bytes > 0) return cudaMemsetAsync(ws + plan.zero_ws, 0, plan.zero_bytes, s);
    return cudaSuccess;
  }
  cudaError_t first(const T* x, T* out, int64_t t0, int64_t t1, cudaStream_t s) {
    if (t1 <= t0) return cudaSuccess;
    const unsigned grid = (unsigned)(t1 - t0);
    a.tile_base = t0;
    if (plan.mode == ScanPlan::kOnePass) {  // tiles numbered by the counter, in launch order
      int* ready = reinterpret_cast<int*>(ws + plan.ready_ws);
      int* tctr = reinterpret_cast<int*>(ws + plan.tilectr_ws);
      int* status = reinterpret_cast<int*>(ws);
      CR_LAUNCH(kKScanOnePass, s, {
        if (shift)
          scan_onepass_kernel<T, true><<<grid, kScanThreads, 0, s>>>(
              x, out, pyr, counters, ready, tctr, status, a, debug_skip_publish(), init);
        else
          scan_onepass_kernel<T, false><<<grid, kScanThreads, 0, s>>>(
              x, out, pyr, counters, ready, tctr, status, a, debug_skip_publish(), init);
      });
      return cudaGetLastError();
    }
    if (plan.mode == ScanPlan::kLocalFixup) {
#define CR_LOCAL(SS, SH) \
  scan_local_kernel<T, SS, SH><<<grid, kScanThreads, 0, s>>>(x, out, totals, a)
      CR_LAUNCH(kKScanLocal, s, {
        if (shift) {
          if (S == 8) CR_LOCAL(8, true);
          else if (S == 4) CR_LOCAL(4, true);
          else CR_LOCAL(2, true);
        } else {
          if (S == 8) CR_LOCAL(8, false);
          else if (S == 4) CR_LOCAL(4, false);
          else CR_LOCAL(2, false);
        }
      });
#undef CR_LOCAL
      return cudaGetLastError();
    }
    a.tile_end = t1;
    const unsigned ugrid = (unsigned)((t1 - t0 + kUpTiles - 1) / kUpTiles);
    CR_LAUNCH(kKScanUp, s, {  // up pass: pairwise, blocks spanning tiles, binary32 iterated
      if (S == 8 && quads != nullptr)
        scan_up_kernel<T, 8, true><<<ugrid, kScanThreads, 0, s>>>(x, pyr, counters, totals, a, quads, tpyr);
      else if (S == 8) scan_up_kernel<T, 8><<<ugrid, kScanThreads, 0, s>>>(x, pyr, counters, totals, a, nullptr, nullptr);
      else if (S == 4) scan_up_kernel<T, 4><<<ugrid, kScanThreads, 0, s>>>(x, pyr, counters, totals, a, nullptr, nullptr);
      else scan_up_kernel<T, 2><<<ugrid, kScanThreads, 0, s>>>(x, pyr, counters, totals, a, nullptr, nullptr);
    });
    return cudaGetLastError();
  }
  // block carries: C_0..C_{K-2} from the block totals
  cudaError_t middle(cudaStream_t s) {
    if (plan.policy == CR_PAIRWISE) {  // every complete tile's prefix Y_b, once
      if (plan.full_tiles < 1) return cudaSuccess;
      const int64_t blocks = (plan.full_tiles + 255) / 256;
      if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
      CR_LAUNCH(kKPairwisePrefix, s,
                pairwise_tile_prefix_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(pyr, ypre, a));
      return cudaGetLastError();
    }
    if (!block || plan.K < 2) return cudaSuccess;
    const T* src = plan.mode == ScanPlan::kLocalFixup ? totals
                                                       : pyr + plan.pyr_off[plan.logB - kLogTile];
    if (plan.parallel_chain) return run_chain<T>(plan.chain, src, carries, ws + plan.chain_ws, s);
    return run_serial_chain<T>(src, carries, plan.K - 1, s);
  }
  // The carries C_k of the blocks whose elements lie in [e0, e1) (tile-
  // aligned, B <= 2048), after those of every earlier block: a segment of
  // the fold continued from C_{kb-1}, which replaces T_{kb-1} in the totals
  // (no longer read: its own segment has run) so that the segment's first
  // step reproduces it. Local + fix-up mode only.
  cudaError_t middle_segment(int64_t e0, int64_t e1, cudaStream_t s) {
    const int64_t kb = e0 >> plan.logB;
    int64_t ke = (e1 + plan.B - 1) >> plan.logB;  // blocks [kb, ke) start in the range
    if (ke > plan.K - 1) ke = plan.K - 1;         // C_{K-1} is not needed
    if (ke <= kb) return cudaSuccess;
    const int64_t first = kb > 0 ? kb - 1 : 0;    // the segment starts at C_{kb-1}
    const int64_t len = ke - first;
    cudaError_t e;
    if (kb > 0 && (e = cudaMemcpyAsync(totals + first, carries + first, sizeof(T),
                                       cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
      return e;
    if (len < 2) return cudaSuccess;
    const bool par = plan.parallel_chain && len >= kParallelChainMin;
    if (par) {
      const ChainPlan cp = plan_chain(len, sizeof(T));  // no larger than the whole chain's
      return run_chain<T>(cp, totals + first, carries + first, ws + plan.chain_ws, s);
    }
    return run_serial_chain<T>(totals + first, carries + first, len, s);
  }
  // The carries and the fix-up in one cooperative pass (inclusive local +
  // fix-up scans with the parallel chain; out != x, for the recovery
  // recomputes the local pass from x).
  cudaError_t fused_middle_second(const T* x, T* out, cudaStream_t s) {
    const int* fail = nullptr;
    bool fused = false;
    cudaError_t e = run_chain_fixup<T>(plan.chain, totals, carries, ws + plan.chain_ws, out,
                                       plan.n, plan.logB, s, &fail, &fused, debug_fused_fail(),
                                       debug_coop_refused());
    if (e != cudaSuccess) return e;
    if (!fused) return second(x, out, 0, plan.n_tiles, s);  // carries ready: plain fix-up
    a.tile_base = 0;
    const unsigned grid = (unsigned)(plan.n_tiles < 1216 ? plan.n_tiles : 1216);
    CR_LAUNCH(kKScanLocalAgain, s, {
      if (S == 8)
        scan_local_again_kernel<T, 8><<<grid, kScanThreads, 0, s>>>(x, out, totals, a,
                                                                    plan.n_tiles, fail);
      else if (S == 4)
        scan_local_again_kernel<T, 4><<<grid, kScanThreads, 0, s>>>(x, out, totals, a,
                                                                    plan.n_tiles, fail);
      else
        scan_local_again_kernel<T, 2><<<grid, kScanThreads, 0, s>>>(x, out, totals, a,
                                                                    plan.n_tiles, fail);
    });
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return run_fixup_again<T>(out, carries, plan.n, plan.logB, fail, s);
  }
  cudaError_t second(const T* x, T* out, int64_t t0, int64_t t1, cudaStream_t s) {
    if (t1 <= t0 || plan.mode == ScanPlan::kOnePass) return cudaSuccess;
    const unsigned grid = (unsigned)(t1 - t0);
    a.tile_base = t0;
    if (plan.mode == ScanPlan::kLocalFixup) {
      if (shift) {  // every output: init, carries and the shifted in-block values (one range)
        if (t0 != 0 || t1 != plan.n_tiles) return cudaErrorInvalidValue;
        const int64_t threads = (plan.m + kE - 1) / kE;
        const int64_t blocks = (threads + 255) / 256;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        CR_LAUNCH(kKCarryFixupShift, s,
                  carry_fixup_shift_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(
                      out, carries, plan.n, plan.m, plan.logB, init));
        return cudaGetLastError();
      }
      if (plan.K < 2) return cudaSuccess;
      const int64_t e0 = t0 * kTile > plan.B ? t0 * kTile : plan.B;
      const int64_t e1 = t1 * kTile < plan.n ? t1 * kTile : plan.n;
      return launch_fixup<T>(plan, out, carries, e0, e1, s);
    }
    if (plan.policy == CR_PAIRWISE) {
      CR_LAUNCH(kKScanPairwise, s, {
        if (shift && quads != nullptr)
          scan_pairwise_kernel<T, true, true><<<grid, kScanThreads, 0, s>>>(x, out, ypre, a, init, quads, tpyr);
        else if (shift)
          scan_pairwise_kernel<T, true><<<grid, kScanThreads, 0, s>>>(x, out, ypre, a, init, nullptr, nullptr);
        else if (quads != nullptr)
          scan_pairwise_kernel<T, false, true><<<grid, kScanThreads, 0, s>>>(x, out, ypre, a, init, quads, tpyr);
        else
          scan_pairwise_kernel<T, false><<<grid, kScanThreads, 0, s>>>(x, out, ypre, a, init, nullptr, nullptr);
      });
      return cudaGetLastError();
    }
#define CR_DOWN(SS, SH) \
  scan_down_kernel<T, SS, SH><<<grid, kScanThreads, 0, s>>>(x, out, pyr, carries, a, init)
    CR_LAUNCH(kKScanDown, s, {
      if (shift) {
        if (S == 8) CR_DOWN(8, true);
        else if (S == 4) CR_DOWN(4, true);
        else CR_DOWN(2, true);
      } else {
        if (S == 8) CR_DOWN(8, false);
        else if (S == 4) CR_DOWN(4, false);
        else CR_DOWN(2, false);
      }
    });
#undef CR_DOWN
    return cudaGetLastError();
  }
};

// The carry fix-up of elements [start, end), start >= B.
template <class T>
cudaError_t launch_fixup(const ScanPlan& plan, T* out, const T* carries, int64_t start,
                         int64_t end, cudaStream_t s) {
  if (end <= start) return cudaSuccess;
  const int64_t threads = (end - start + kE - 1) / kE;
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  CR_LAUNCH(kKCarryFixup, s,
            carry_fixup_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(out, carries, start, end,
                                                                    plan.logB));
  return cudaGetLastError();
}

template <class T>
cudaError_t run_scan(const ScanPlan& plan, const T* x, T* out, int64_t es, int64_t bs,
                     int64_t oes, int64_t obs, T init, char* ws, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  const bool shift = plan.out_mode != 0;
  switch (plan.kind) {
    case ScanPlan::kEmpty: return cudaSuccess;
    case ScanPlan::kInitOnly: {
      if ((plan.batch + 255) / 256 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
      CR_LAUNCH(kKFillInit, s,
                fill_init_kernel<T><<<(unsigned)((plan.batch + 255) / 256), 256, 0, s>>>(
                    out, plan.batch, obs, init));
      return cudaGetLastError();
    }
    case ScanPlan::kPerSequence: {
      if ((plan.batch + 255) / 256 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
      const unsigned grid = (unsigned)((plan.batch + 255) / 256);
      const int LV = plan.stack_levels;
#define CR_SEQ(LVV)                                                                      \
  CR_LAUNCH(kKScanSeq, s,                                                                \
            scan_seq_kernel<T, LVV><<<grid, 256, 0, s>>>(x, out, plan.batch, plan.n, es, \
                                                         bs, oes, obs, (int)plan.policy, \
                                                         plan.B, shift ? 1 : 0, plan.m,  \
                                                         init))
#define CR_SEQB(BBV, LEFT)                                                                 \
  CR_LAUNCH(kKScanSeqBlock, s,                                                             \
            (scan_seq_block_kernel<T, BBV, LEFT><<<grid, 256, 0, s>>>(                     \
                x, out, plan.batch, plan.n, es, bs, oes, obs, shift ? 1 : 0, plan.m, init)))
      const bool bd = plan.policy == CR_BLOCK_DYADIC;
      const bool left = plan.policy == CR_LEFT_FOLD || (bd && plan.B == 1);
      if (left && sizeof(T) == 8 && !shift && bs == 1 && obs == 1 && es % 2 == 0 &&
          oes % 2 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
          (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
        const int64_t blocks2 = ((plan.batch + 1) / 2 + 255) / 256;
        CR_LAUNCH(kKScanSeqLeft2, s,
                  scan_seq_left2_kernel<4, true><<<(unsigned)blocks2, 256, 0, s>>>(
                      reinterpret_cast<const double*>(x), reinterpret_cast<double*>(out),
                      plan.batch, plan.n, es, oes));
        return cudaGetLastError();
      }
      if (left) CR_SEQB(16, true);
      else if (bd && plan.B == 16) CR_SEQB(16, false);
      else if (bd && plan.B == 8) CR_SEQB(8, false);
      else if (bd && plan.B == 4) CR_SEQB(4, false);
      else if (bd && plan.B == 2) CR_SEQB(2, false);
      else if (LV <= 5) CR_SEQ(5);
      else if (LV <= 9) CR_SEQ(9);
      else if (LV <= 17) CR_SEQ(17);
      else CR_SEQ(32);
#undef CR_SEQB
#undef CR_SEQ
      return cudaGetLastError();
    }
    case ScanPlan::kChainOnly: {
      // inclusive: out[k] = y[k]; shifted: y[k] into out[k + 1], then init
      T* dst = shift ? out + 1 : out;
      const int64_t K = plan.chain_n;
      if (K > 0) {
        const T* src = x;
        // in place, the chain must not overwrite input it has still to read:
        // the parallel chain's fallback re-reads all of it, and a shifted
        // output runs one element ahead of the input. Keep a copy then.
        if (out == x && (plan.parallel_chain || shift)) {
          T* copy = reinterpret_cast<T*>(ws + plan.copy_ws);
          e = cudaMemcpyAsync(copy, x, (size_t)K * sizeof(T), cudaMemcpyDeviceToDevice, s);
          if (e != cudaSuccess) return e;
          src = copy;
        }
        if (!plan.parallel_chain) {
          if ((e = run_serial_chain<T>(src, dst, K, s)) != cudaSuccess) return e;
        } else if (K <= kMaxFusedChainAlone && !fused_fixup_disabled()) {
          // the fill of each tile overlaps the rest of the walk (one
          // cooperative pass); on a failure the serial chain rewrites dst
          const int* fail = nullptr;
          bool fused = false;
          if ((e = run_chain_fixup<T>(plan.chain, src, dst, ws + plan.chain_ws, nullptr, 0, 0, s,
                                      &fail, &fused, debug_fused_fail(),
                                      debug_coop_refused())) != cudaSuccess)
            return e;
        } else if ((e = run_chain<T>(plan.chain, src, dst, ws + plan.chain_ws, s)) !=
                   cudaSuccess) {
          return e;
        }
      }
      if (shift) {
        const int64_t blocks = (plan.m + 255) / 256;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        CR_LAUNCH(kKApplyInit, s,
                  apply_init_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(out, plan.m, init));
        e = cudaGetLastError();
      }
      return e;
    }
    case ScanPlan::kTiled: break;
  }
  Tiled<T> tc(plan, ws, init);
  if ((e = tc.prepare(s)) != cudaSuccess) return e;
  if ((e = tc.first(x, out, 0, plan.n_tiles, s)) != cudaSuccess) return e;
  if (fused_fixup_ok(plan) && out != x) return tc.fused_middle_second(x, out, s);
  if ((e = tc.middle(s)) != cudaSuccess) return e;
  return tc.second(x, out, 0, plan.n_tiles, s);
}

constexpr int64_t kHostChunks = 32;  // 2^28 fp64 from host: 8 14.6, 16 13.8, 32 13.4 ms

template <class T>
cudaError_t run_scan_host(const ScanPlan& plan, const T* x_host, T* out_host, T* x_dev,
                          T* out_dev, char* ws, cudaStream_t s) {
  cudaError_t e;
  const size_t bytes = (size_t)plan.n * sizeof(T);
  if (plan.kind != ScanPlan::kTiled || plan.out_mode != 0) {  // not pipelined
    if (plan.n > 0) {
      if ((e = cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return e;
    }
    if ((e = run_scan<T>(plan, x_dev, out_dev, 1, plan.n, 1, plan.n, T(0), ws, s)) !=
        cudaSuccess)
      return e;
    if (plan.n > 0 &&
        (e = cudaMemcpyAsync(out_host, out_dev, bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
      return e;
    return cudaStreamSynchronize(s);
  }
  // about kHostChunks chunks of whole tiles (at least 256 tiles each): the
  // first chunk's copy in and the last one's copy out overlap nothing
  const int64_t tiles = plan.n_tiles;
  int64_t per = (tiles + kHostChunks - 1) / kHostChunks;
  if (per < 256) per = 256;
  const int64_t nchunks = (tiles + per - 1) / per;
  std::lock_guard<std::mutex> lock(host_pipe_mutex());  // host-buffer calls share the streams
  HostPipe* pipe = host_pipe();
  if (pipe == nullptr) return cudaErrorInvalidDevice;
  HostPipe& hp = *pipe;
  if ((e = hp.ensure((int)nchunks)) != cudaSuccess) return e;
  cudaStream_t cin = hp.in, cout = hp.out;
  // the caller's stream may hold earlier work on these buffers: start after it
  if ((e = cudaEventRecord(hp.start, s)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(cin, hp.start, 0)) != cudaSuccess) return e;
  if ((e = cudaStreamWaitEvent(cout, hp.start, 0)) != cudaSuccess) return e;
  Tiled<T> tc(plan, ws, T(0));
  if ((e = tc.prepare(s)) != cudaSuccess) return e;
  auto range = [&](int64_t c, int64_t& t0, int64_t& t1, int64_t& e0, int64_t& e1) {
    t0 = c * per;
    t1 = t0 + per < tiles ? t0 + per : tiles;
    e0 = t0 * kTile;
    e1 = t1 * kTile < plan.n ? t1 * kTile : plan.n;
  };
  if (plan.mode == ScanPlan::kLocalFixup && nchunks > 1 && plan.K >= 2) {
    // block_dyadic, B <= 2048: blocks do not straddle chunks (tile-aligned)
    // and C_k depends on T_0 .. T_k only, so the carries are folded chunk by
    // chunk (each segment continued from the last carry of the one before)
    // and every chunk is fixed up and copied out as soon as its carries
    // exist: the copies out overlap the copies in.
    for (int64_t c = 0; c < nchunks; ++c) {
      int64_t t0, t1, e0, e1;
      range(c, t0, t1, e0, e1);
      if ((e = cudaMemcpyAsync(x_dev + e0, x_host + e0, (size_t)(e1 - e0) * sizeof(T),
                               cudaMemcpyHostToDevice, cin)) != cudaSuccess)
        return e;
      if ((e = cudaEventRecord(hp.ev_in[c], cin)) != cudaSuccess) return e;
    }
    for (int64_t c = 0; c < nchunks; ++c) {
      int64_t t0, t1, e0, e1;
      range(c, t0, t1, e0, e1);
      if ((e = cudaStreamWaitEvent(s, hp.ev_in[c], 0)) != cudaSuccess) return e;
      if ((e = tc.first(x_dev, out_dev, t0, t1, s)) != cudaSuccess) return e;
      if ((e = tc.middle_segment(e0, e1, s)) != cudaSuccess) return e;
      if ((e = tc.second(x_dev, out_dev, t0, t1, s)) != cudaSuccess) return e;
      if ((e = cudaEventRecord(hp.ev_out[c], s)) != cudaSuccess) return e;
      if ((e = cudaStreamWaitEvent(cout, hp.ev_out[c], 0)) != cudaSuccess) return e;
      if ((e = cudaMemcpyAsync(out_host + e0, out_dev + e0, (size_t)(e1 - e0) * sizeof(T),
                               cudaMemcpyDeviceToHost, cout)) != cudaSuccess)
        return e;
    }
    if ((e = cudaStreamSynchronize(cout)) != cudaSuccess) return e;
    if ((e = cudaStreamSynchronize(cin)) != cudaSuccess) return e;
    return cudaStreamSynchronize(s);
  }
  for (int64_t c = 0; c < nchunks; ++c) {  // copy in, first pass per chunk
    int64_t t0, t1, e0, e1;
    range(c, t0, t1, e0, e1);
    if ((e = cudaMemcpyAsync(x_dev + e0, x_host + e0, (size_t)(e1 - e0) * sizeof(T),
                             cudaMemcpyHostToDevice, cin)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(hp.ev_in[c], cin)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, hp.ev_in[c], 0)) != cudaSuccess) return e;
    if ((e = tc.first(x_dev, out_dev, t0, t1, s)) != cudaSuccess) return e;
    if (!tc.has_second() && (e = cudaEventRecord(hp.ev_out[c], s)) != cudaSuccess) return e;
  }
  if ((e = tc.middle(s)) != cudaSuccess) return e;
  if (tc.has_second()) {
    for (int64_t c = 0; c < nchunks; ++c) {
      int64_t t0, t1, e0, e1;
      range(c, t0, t1, e0, e1);
      if ((e = tc.second(x_dev, out_dev, t0, t1, s)) != cudaSuccess) return e;
      if ((e = cudaEventRecord(hp.ev_out[c], s)) != cudaSuccess) return e;
    }
  }
  for (int64_t c = 0; c < nchunks; ++c) {  // copy out as each chunk completes
    int64_t t0, t1, e0, e1;
    range(c, t0, t1, e0, e1);
    if ((e = cudaStreamWaitEvent(cout, hp.ev_out[c], 0)) != cudaSuccess) return e;
    if ((e = cudaMemcpyAsync(out_host + e0, out_dev + e0, (size_t)(e1 - e0) * sizeof(T),
                             cudaMemcpyDeviceToHost, cout)) != cudaSuccess)
      return e;
  }
  if ((e = cudaStreamSynchronize(cout)) != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(cin)) != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

template <class T>
cudaError_t run_block_totals(const ScanPlan& plan, const T* x, char* ws, cudaStream_t s,
                             T** totals_out) {
  ScanArgs a{};
  a.n = plan.n;
  a.full_tiles = plan.full_tiles;
  a.logB = plan.logB;
  // blocks inside a tile need no node pyramid across tiles
  a.pyr_levels = plan.mode == ScanPlan::kLocalFixup ? 0 : plan.pyr_levels;
  a.carry = 0;
  a.totals_level = plan.totals_level;
  for (int l = 0; l < kMaxLevels; ++l) {
    a.pyr_off[l] = plan.pyr_off[l];
    a.cnt_off[l] = plan.cnt_off[l];
  }
  T* pyr = reinterpret_cast<T*>(ws + plan.pyr_ws);
  int* counters = reinterpret_cast<int*>(ws + plan.cnt_ws);
  T* totals = reinterpret_cast<T*>(ws + plan.totals_ws);
  cudaError_t e;
  if (plan.zero_bytes > 0 && a.pyr_levels > 0 &&
      (e = cudaMemsetAsync(ws + plan.zero_ws, 0, plan.zero_bytes, s)) != cudaSuccess)
    return e;
  if (plan.n_tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  a.tile_base = 0;
  a.tile_end = plan.n_tiles;
  const unsigned grid = (unsigned)((plan.n_tiles + kUpTiles - 1) / kUpTiles);
  const int S = (int)(plan.B < kE ? plan.B : kE);
  CR_LAUNCH(kKScanUp, s, {
    if (S == 8) scan_up_kernel<T, 8><<<grid, kScanThreads, 0, s>>>(x, pyr, counters, totals, a, nullptr, nullptr);
    else if (S == 4) scan_up_kernel<T, 4><<<grid, kScanThreads, 0, s>>>(x, pyr, counters, totals, a, nullptr, nullptr);
    else scan_up_kernel<T, 2><<<grid, kScanThreads, 0, s>>>(x, pyr, counters, totals, a, nullptr, nullptr);
  });
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t Kf = plan.n / plan.B;
  if (plan.logB > kLogTile && Kf > 0) {  // the pyramid level of whole blocks
    e = cudaMemcpyAsync(totals, pyr + plan.pyr_off[plan.logB - kLogTile], (size_t)Kf * sizeof(T),
                        cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return e;
  }
  *totals_out = totals;
  return cudaSuccess;
}

template cudaError_t run_block_totals<double>(const ScanPlan&, const double*, char*,
                                              cudaStream_t, double**);
template cudaError_t run_block_totals<float>(const ScanPlan&, const float*, char*, cudaStream_t,
                                             float**);
template cudaError_t run_scan_host<double>(const ScanPlan&, const double*, double*, double*,
                                           double*, char*, cudaStream_t);
template cudaError_t run_scan_host<float>(const ScanPlan&, const float*, float*, float*, float*,
                                          char*, cudaStream_t);
template cudaError_t run_scan<double>(const ScanPlan&, const double*, double*, int64_t,
                                      int64_t, int64_t, int64_t, double, char*, cudaStream_t);
template cudaError_t run_scan<float>(const ScanPlan&, const float*, float*, int64_t, int64_t,
                                     int64_t, int64_t, float, char*, cudaStream_t);

}  // namespace cr
