// Canonical reduction kernels (P4016R0 on "Canonical Parallel Reduction and
// Scan", Key Design Points):
//   reduce(x, n, L, init) = op(init, tree(R_0 .. R_{m-1})),  m = min(n, L),
//   R_j = tree(x_j, x_{j+L}, ...),  tree = iterative pairwise shift-reduce.
//
// Data view. Lane j of a sequence is column j of a row-major (rows x L)
// matrix: row t holds x[tL .. tL + L). R = floor(n / L) rows are full; lanes
// j < r = n mod L have one more element in row R. Reading a row is a
// coalesced read of L consecutive elements, so each thread owns one lane and
// walks down its column.
//
// Passes. One launch per level h of a pyramid:
//   * leaf blocks: a chunk of T = G * P full rows x W lanes; thread (lane j,
//     group g) reduces its run of P rows to a perfect tree in registers (16
//     loads in flight, then a register shift-reduce stack), the G run values
//     of a lane are combined in shared memory into the perfect tree over the
//     chunk, which becomes one element of the level h+1 matrix. Chunks start
//     at multiples of T, so every value is a node of the lane's tree.
//   * tail blocks (same launch): the rows after the last full chunk. Their
//     shift-reduce stack is folded, smallest block first, onto the lane's
//     running right-hand part `acc` (the finer levels' tails lie to the
//     right), or, when the tail is itself a full chunk (only possible for
//     the lanes that own row R), written as the ragged row of level h+1.
//   * final pass: everything left is tail; then, when one block holds all
//     lanes, the cross-lane tree over R_0..R_{m-1} and op(init, .) follow in
//     the same block. Otherwise the lane results are a new sequence reduced
//     by the same passes with L = 1.
// No value is ever combined with an atomic; the grid shape changes which
// block evaluates a node, never the node.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "cr_device.cuh"
#include "cr_launch.h"
#include "cr_plan.h"

namespace cr {

// Decomposition knobs: the threads of a block (lanes x runs a block holds;
// 128 measured within 1 % of 256), the largest run of rows a thread reduces
// in a leaf pass, and the leaf items a pass aims at (4 per SM of a GB300).
// None changes a result, only which block forms which node (the canonical
// tree is the same for every value; a compile-time override is how the
// tests show it).
#ifndef CR_REDUCE_THREADS
#define CR_REDUCE_THREADS 256
#endif
constexpr int kThreads = CR_REDUCE_THREADS;  // a power of two
constexpr int kLV = 10;  // stack levels: a run of up to 512 operands

#ifndef CR_REDUCE_MAX_RUN
#define CR_REDUCE_MAX_RUN 256
#endif
#ifndef CR_REDUCE_LEAF_ITEMS
#define CR_REDUCE_LEAF_ITEMS 608
#endif
constexpr int64_t kMaxRun = CR_REDUCE_MAX_RUN;  // a power of two, at most 256
constexpr int64_t kLeafItems = CR_REDUCE_LEAF_ITEMS;
static_assert(kMaxRun >= 2 && kMaxRun <= 256 && (kMaxRun & (kMaxRun - 1)) == 0,
              "runs are powers of two up to 256 rows");

template <class T, int U, bool kContig>
__global__ void __launch_bounds__(kThreads)
lane_pass_kernel(const T* __restrict__ in_base, int64_t in_seg, int64_t in_row,
                 int64_t in_lane, T* __restrict__ next, T* __restrict__ acc,
                 int* __restrict__ has, T* __restrict__ out, T init, PassArgs a) {
  constexpr int LOGU = (U == 1) ? 0 : (U == 2) ? 1 : (U == 4) ? 2 : (U == 8) ? 3 : 4;
  __shared__ T vals[kThreads];
  __shared__ T lane_val[kThreads];
  __shared__ int lane_has[kThreads];

  const int tid = threadIdx.x;
  const int jl = tid % a.W;
  const int g = tid / a.W;

  int64_t item = a.item_base + blockIdx.x;
  const bool leaf = item < a.n_leaf_items;
  int64_t b, c;
  int w;
  if (leaf) {
    w = (int)(item % a.tiles);
    const int64_t rest = item / a.tiles;
    c = rest % a.C;
    b = rest / a.C;
  } else {
    item -= a.n_leaf_items;
    w = (int)(item % a.tiles);
    b = item / a.tiles;
    c = a.C;
  }
  const int64_t j = (int64_t)w * a.W + jl;
  const bool lane_ok = (g < a.G) && (j < a.L);
  const int64_t nj = lane_ok ? a.R + (j < a.r ? 1 : 0) : 0;  // values of lane j
  const int64_t run0 = c * a.T + (int64_t)g * a.P;             // first row of my run
  int64_t cnt;
  if (leaf) {
    cnt = lane_ok ? a.P : 0;
  } else {
    cnt = nj - run0;
    cnt = cnt < 0 ? 0 : (cnt > a.P ? a.P : cnt);
  }

  // ---- my run: perfect blocks of U rows, then single rows, into the stack
  RegStack<T, kLV> st;
  st.reset();
  if (cnt > 0) {
    const T* p = in_base + b * in_seg + run0 * in_row + j * in_lane;
    int64_t k = 0;
    constexpr int VW = 16 / sizeof(T);  // elements per 16-byte vector
    // blocks of U rows, the next block's loads in flight while the current
    // block's tree is built (two register buffers)
    if (kContig && U % VW == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
      // one lane (L = 1 and the lane-result passes): the run is contiguous
      auto load = [&](T (&v)[U], int64_t k0) {
        const uint4* q = reinterpret_cast<const uint4*>(p + k0);
#pragma unroll
        for (int u = 0; u < U / VW; ++u) {
          const uint4 d = __ldg(q + u);
#pragma unroll
          for (int e = 0; e < VW; ++e) v[u * VW + e] = reinterpret_cast<const T*>(&d)[e];
        }
      };
      if (k + U <= cnt) {
        T v[U];
        load(v, k);
        for (; k + 2 * U <= cnt; k += U) {
          T w[U];
          load(w, k + U);
          st.push(perfect_tree<T, U>(v), LOGU);
#pragma unroll
          for (int u = 0; u < U; ++u) v[u] = w[u];
        }
        st.push(perfect_tree<T, U>(v), LOGU);
        k += U;
      }
    }
    if (k + U <= cnt) {
      auto load = [&](T (&v)[U], int64_t k0) {
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = ldg(p + (k0 + u) * in_row);
      };
      T v[U];
      load(v, k);
      for (; k + 2 * U <= cnt; k += U) {
        T w[U];
        load(w, k + U);
        st.push(perfect_tree<T, U>(v), LOGU);
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = w[u];
      }
      st.push(perfect_tree<T, U>(v), LOGU);
      k += U;
    }
    for (; k < cnt; ++k) st.push(ldg(p + k * in_row), 0);
  }

  auto V = [&](int gg) -> T& { return vals[gg * a.W + jl]; };

  if (leaf) {
    // all G runs of the chunk are full: perfect tree over them
    if (lane_ok) {
      T v = T(0);
      st.fold_onto(v, false);
      V(g) = v;
    }
    __syncthreads();
    smem_pyramid<T>(V, lane_ok ? g : a.G, a.G, a.G);
    if (lane_ok && g == 0) next[b * a.next_seg + c * a.L + j] = V(0);
    return;
  }

  // ---- tail of this level (and, in the final pass, everything)
  const int64_t tau = lane_ok ? (nj - c * a.T) : 0;  // tail length, 0 <= tau <= T
  const int F = (int)(tau / a.P);                      // full runs
  const int part = (int)(tau % a.P);                   // length of the partial run
  const bool to_next = !a.final_pass && tau == a.T;    // ragged lanes' extra chunk

  if (lane_ok && g < F) {
    T v = T(0);
    st.fold_onto(v, false);
    V(g) = v;
  }
  if (lane_ok && to_next && a.first_level && g == 0) has[b * a.L + j] = 0;  // acc empty
  if (lane_ok && !to_next) {
    // innermost first: the previous levels' part, then my partial run
    const bool writer = part > 0 ? (g == F) : (g == 0);
    if (writer) {
      T av = T(0);  // read only when ah is set
      bool ah = false;
      if (!a.first_level && has[b * a.L + j]) {
        av = acc[b * a.L + j];
        ah = true;
      }
      if (part > 0) ah = st.fold_onto(av, ah);
      lane_val[jl] = av;
      lane_has[jl] = ah ? 1 : 0;
    }
  }
  __syncthreads();
  smem_pyramid<T>(V, lane_ok ? g : a.G, a.G, lane_ok ? F : 0);

  if (lane_ok && g == 0) {
    if (to_next) {
      next[b * a.next_seg + c * a.L + j] = V(0);  // F == G: the chunk's perfect tree
    } else {
      T av = lane_val[jl];
      bool ah = lane_has[jl] != 0;
      ah = fold_blocks<T>(V, F, av, ah);
      if (a.fuse_cross) {
        lane_val[jl] = av;  // R_j (every lane j < m holds at least one operand)
      } else {
        acc[b * a.L + j] = av;
        has[b * a.L + j] = ah ? 1 : 0;
      }
    }
  }
  if (!a.fuse_cross) return;

  // ---- cross-lane tree over R_0..R_{m-1} (all in this block), then init
  __syncthreads();
  auto LVv = [&](int gg) -> T& { return lane_val[gg]; };
  const int mm = (int)a.m;
  int Gp = 1;
  while (Gp < mm) Gp *= 2;
  smem_pyramid<T>(LVv, tid < mm ? tid : Gp, Gp, mm);
  if (tid == 0) {
    T r = T(0);
    fold_blocks<T>(LVv, mm, r, false);
    out[b] = add_rn(init, r);
  }
}

template <class T>
__global__ void write_init_kernel(T* out, int64_t batch, T init) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < batch) out[i] = init;
}

// ------------------------------------------------- rows: one warp per row
template <class T>
struct Vec16;
template <>
struct Vec16<double> {
  using type = double2;
  __device__ static double get(const double2& d, int v) { return v == 0 ? d.x : d.y; }
};
template <>
struct Vec16<float> {
  using type = float4;
  __device__ static float get(const float4& d, int v) {
    return v == 0 ? d.x : (v == 1 ? d.y : (v == 2 ? d.z : d.w));
  }
};

// Batched canonical reduce of contiguous rows with L = 32 V lanes
// (V = 16 / sizeof(T)) and n = P L: lane j of a row holds the columns
// j + L t, t < P, so the V components of a thread's 16-byte loads are V
// consecutive lanes and one warp's load is one row of the (P x L) lane
// matrix. One warp per row: per lane the P-operand tree in a register
// binary-counter stack (perfect trees of 8 positions pushed at level 3, the
// rest one by one), then the perfect tree over the L lane results (in the
// thread, then across lanes by shuffles, lower lane on the left), then
// op(init, root).
template <class T, int LV>
__global__ void __launch_bounds__(256)
row_reduce_kernel(const T* x, T* out, int64_t batch, int64_t P, int64_t bs, T init) {
  constexpr int V = 16 / sizeof(T);
  using Vec = typename Vec16<T>::type;
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= batch) return;  // whole warps
  const Vec* p = reinterpret_cast<const Vec*>(x + row * bs) + lane;  // position t at p[32 t]
  RegStack<T, LV> st[V];
#pragma unroll
  for (int v = 0; v < V; ++v) st[v].reset();
  int64_t t = 0;
  for (; t + 8 <= P; t += 8) {
    Vec d[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) d[u] = __ldcs(p + (t + u) * 32);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      T a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = Vec16<T>::get(d[u], v);
      st[v].push(perfect_tree<T, 8>(a), 3);
    }
  }
  for (; t < P; ++t) {
    const Vec d = __ldcs(p + t * 32);
#pragma unroll
    for (int v = 0; v < V; ++v) st[v].push(Vec16<T>::get(d, v), 0);
  }
  T r[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
    r[v] = T(0);
    st[v].fold_onto(r[v], false);
  }
  T val = perfect_tree<T, V>(r);
#pragma unroll
  for (int sh = 1; sh < 32; sh *= 2) {
    const T other = __shfl_down_sync(full, val, sh);
    if ((lane & (2 * sh - 1)) == 0) val = add_rn(val, other);
  }
  if (lane == 0) out[row] = add_rn(init, val);
}

// ------------------------------------------------------------------ planning
namespace {

int64_t pow2floor(int64_t v) {
  int64_t p = 1;
  while (p * 2 <= v) p *= 2;
  return p;
}
int64_t pow2ceil(int64_t v) {
  int64_t p = 1;
  while (p < v) p *= 2;
  return p;
}

struct Bump {
  size_t off;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~size_t(255);
    return o;
  }
};

// Appends the passes that reduce `batch` sequences held as a (R x Lanes)
// matrix (+ r ragged lanes) to lane results. If the last pass cannot fuse the
// cross-lane tree, recurses with L = 1 over the lane results.
void plan_tree(ReducePlan& plan, Bump& ws, int64_t batch, int64_t R, int64_t r,
               int64_t Lanes, int64_t m, MatRef in, size_t esize) {
  const int W = (int)std::min<int64_t>(Lanes, kThreads);
  const int G = (int)pow2floor(kThreads / W);
  const int tiles = (int)((Lanes + W - 1) / W);
  const size_t acc_off = ws.take(batch * Lanes * esize);
  const size_t has_off = ws.take(batch * Lanes * sizeof(int));
  bool first = true;
  for (;;) {
    PassPlan pp{};
    PassArgs& a = pp.a;
    a.R = R;
    a.r = r;
    a.L = Lanes;
    a.W = W;
    a.G = G;
    a.tiles = tiles;
    a.m = m;
    a.first_level = first ? 1 : 0;
    pp.in = in;
    pp.acc_off = acc_off;
    pp.has_off = has_off;
    const bool final_pass = R * W <= 4096;
    if (final_pass) {
      int64_t T = std::max<int64_t>(G, pow2ceil(R + (r > 0 ? 1 : 0)));
      a.T = T;
      a.P = (int)(T / G);
      a.C = 0;
      a.n_leaf_items = 0;
      a.final_pass = 1;
      a.fuse_cross = tiles == 1 ? 1 : 0;
      a.next_seg = 0;
      pp.next_off = 0;
      pp.grid = batch * tiles;
      plan.passes.push_back(pp);
      if (!a.fuse_cross) {
        // lane results acc[b][0..m) form a new sequence per segment; L = 1
        MatRef acc_in{true, acc_off, Lanes, 1, 1};
        plan_tree(plan, ws, batch, m, 0, 1, 1, acc_in, esize);
      }
      return;
    }
    const int64_t target = std::max<int64_t>(1, kLeafItems / (batch * tiles));
    int64_t P = pow2floor(std::max<int64_t>(1, R / (G * target)));
    P = std::min<int64_t>(P, kMaxRun);
    if ((int64_t)G * P * W < 4096)
      P = std::min<int64_t>(pow2floor(std::max<int64_t>(1, R / G)),
                            pow2ceil((4096 + G * W - 1) / (G * W)));
    if (G * P < 2) P = 2;
    P = std::min<int64_t>(P, kMaxRun);
    const int64_t T = G * P;
    const int64_t C = R / T;
    a.T = T;
    a.P = (int)P;
    a.C = C;
    a.n_leaf_items = batch * C * tiles;
    a.final_pass = 0;
    a.fuse_cross = 0;
    a.next_seg = (C + 1) * Lanes;
    pp.next_off = ws.take(batch * (C + 1) * Lanes * esize);
    pp.grid = a.n_leaf_items + batch * tiles;
    plan.passes.push_back(pp);
    const int64_t r_next = (R % T == T - 1) ? r : 0;
    in = MatRef{true, pp.next_off, a.next_seg, Lanes, 1};
    R = C;
    r = r_next;
    first = false;
  }
}

}  // namespace

ReducePlan plan_reduce(int64_t batch, int64_t n, int64_t L, int64_t elem_stride,
                       int64_t batch_stride, size_t esize) {
  ReducePlan plan;
  Bump ws{kHeaderBytes};
  plan.batch = batch;
  if (n == 0 || batch == 0) {
    plan.ws_bytes = ws.off;
    return plan;
  }
  const int64_t Leff = (L >= n) ? 1 : L;  // L >= n gives the same tree as L = 1
  const int64_t R = n / Leff, r = n % Leff;
  const int64_t m = std::min<int64_t>(n, Leff);
  MatRef x_in{false, 0, batch_stride, Leff * elem_stride, elem_stride};
  plan_tree(plan, ws, batch, R, r, Leff, m, x_in, esize);
  plan.ws_bytes = ws.off;
  const int64_t Lrow = 32 * (16 / (int64_t)esize);
  if (batch >= 2048 && elem_stride == 1 && L == Lrow && n >= L && n % L == 0 &&
      (batch_stride * (int64_t)esize) % 16 == 0) {
    const int64_t P = n / L;
    const int need = (int)std::log2((double)P) + 1;  // stack levels for P operands
    const int lv = need <= 6 ? 6 : need <= 11 ? 11 : need <= 16 ? 16 : need <= 21 ? 21 : 0;
    if (lv && P < (int64_t(1) << 21)) {
      plan.rows_lv = lv;
      plan.rows_P = P;
      plan.rows_bs = batch_stride;
    }
  }
  return plan;
}

// Items [i0, i1) of one pass (leaf items first, then the tail items).
template <class T>
cudaError_t launch_pass(const PassPlan& pp, const T* x, T* out, T init, char* ws,
                        cudaStream_t s, int64_t i0, int64_t i1) {
  if (i1 <= i0) return cudaSuccess;
  const T* in_base = pp.in.in_ws ? reinterpret_cast<const T*>(ws + pp.in.ws_off) : x;
  T* next = pp.a.final_pass ? nullptr : reinterpret_cast<T*>(ws + pp.next_off);
  T* acc = reinterpret_cast<T*>(ws + pp.acc_off);
  int* has = reinterpret_cast<int*>(ws + pp.has_off);
  if (i1 - i0 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  PassArgs a = pp.a;
  a.item_base = i0;
  const unsigned grid = (unsigned)(i1 - i0);
  // runs shorter than 16 rows use smaller register blocks; one-lane passes
  // (contiguous runs, 16-byte aligned) load with vector accesses
  const bool contig = pp.in.row == 1 && (reinterpret_cast<uintptr_t>(in_base) & 15) == 0 &&
                      (pp.in.seg * (int64_t)sizeof(T)) % 16 == 0;
#define CR_LANE(UU, CC)                                                                   \
  CR_LAUNCH(kKLanePass, s,                                                                \
            (lane_pass_kernel<T, UU, CC><<<grid, kThreads, 0, s>>>(                       \
                in_base, pp.in.seg, pp.in.row, pp.in.lane, next, acc, has, out, init, a)))
  if (pp.a.P >= 16) {
    if (contig) CR_LANE(16, true);
    else CR_LANE(16, false);
  } else {
    CR_LANE(4, false);
  }
#undef CR_LANE
  return cudaGetLastError();
}

template <class T>
cudaError_t run_reduce(const ReducePlan& plan, const T* x, T* out, T init, char* ws,
                       cudaStream_t s) {
  if (plan.passes.empty()) {
    if (plan.batch > 0)
      CR_LAUNCH(kKWriteInit, s,
                write_init_kernel<T><<<(unsigned)((plan.batch + 255) / 256), 256, 0, s>>>(
                    out, plan.batch, init));
    return cudaGetLastError();
  }
  if (plan.rows_lv && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
    const int64_t blocks = (plan.batch + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
#define CR_ROWS(LVV)                                                                       \
  CR_LAUNCH(kKRowReduce, s,                                                                \
            (row_reduce_kernel<T, LVV><<<(unsigned)blocks, 256, 0, s>>>(x, out, plan.batch, \
                                                                      plan.rows_P,         \
                                                                      plan.rows_bs, init)))
    if (plan.rows_lv == 6) CR_ROWS(6);
    else if (plan.rows_lv == 11) CR_ROWS(11);
    else if (plan.rows_lv == 16) CR_ROWS(16);
    else CR_ROWS(21);
#undef CR_ROWS
    return cudaGetLastError();
  }
  for (const PassPlan& pp : plan.passes) {
    const cudaError_t e = launch_pass<T>(pp, x, out, init, ws, s, 0, pp.grid);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <class T>
cudaError_t run_reduce_host(const ReducePlan& plan, const T* x_host, T* x_dev, T* out, T init,
                            char* ws, cudaStream_t s, int64_t n) {
  cudaError_t e;
  const bool chunked = plan.batch == 1 && !plan.rows_lv && !plan.passes.empty() &&
                       !plan.passes[0].a.final_pass && plan.passes[0].a.C >= 16;
  if (!chunked) {  // one copy, then the passes
    if (n > 0 && (e = cudaMemcpyAsync(x_dev, x_host, (size_t)n * sizeof(T),
                                      cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return e;
    return run_reduce<T>(plan, x_dev, out, init, ws, s);
  }
  // The first pass's leaf items reduce chunks of T rows of L consecutive
  // elements each, independently: the chunks are copied in (up to 32) groups on the
  // copy stream and each group's leaf items run once it has arrived; the
  // tail items, which read the rows after the last chunk, and the later
  // passes follow the last copy.
  const PassPlan& p0 = plan.passes[0];
  const int64_t C = p0.a.C, tiles = p0.a.tiles, per_chunk = p0.a.T * p0.a.L;
  const int groups = C < 32 ? (int)C : 32;
  std::lock_guard<std::mutex> lock(host_pipe_mutex());
  HostPipe* pipe = host_pipe();
  if (pipe == nullptr) return cudaErrorInvalidDevice;
  HostPipe& hp = *pipe;
  if ((e = hp.ensure(groups + 1)) != cudaSuccess) return e;
  if ((e = cudaEventRecord(hp.start, s)) != cudaSuccess) return e;  // after the caller's work
  if ((e = cudaStreamWaitEvent(hp.in, hp.start, 0)) != cudaSuccess) return e;
  for (int g = 0; g <= groups; ++g) {
    const int64_t e0 = g < groups ? (C * g / groups) * per_chunk : C * per_chunk;
    const int64_t e1 = g < groups ? (C * (g + 1) / groups) * per_chunk : n;
    if (e1 > e0 && (e = cudaMemcpyAsync(x_dev + e0, x_host + e0, (size_t)(e1 - e0) * sizeof(T),
                                        cudaMemcpyHostToDevice, hp.in)) != cudaSuccess)
      return e;
    if ((e = cudaEventRecord(hp.ev_in[g], hp.in)) != cudaSuccess) return e;
  }
  for (int g = 0; g <= groups; ++g) {
    if ((e = cudaStreamWaitEvent(s, hp.ev_in[g], 0)) != cudaSuccess) return e;
    const int64_t i0 = g < groups ? (C * g / groups) * tiles : C * tiles;
    const int64_t i1 = g < groups ? (C * (g + 1) / groups) * tiles : p0.grid;
    if ((e = launch_pass<T>(p0, x_dev, out, init, ws, s, i0, i1)) != cudaSuccess) return e;
  }
  for (size_t k = 1; k < plan.passes.size(); ++k) {
    const PassPlan& pp = plan.passes[k];
    if ((e = launch_pass<T>(pp, x_dev, out, init, ws, s, 0, pp.grid)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template cudaError_t run_reduce<double>(const ReducePlan&, const double*, double*, double,
                                        char*, cudaStream_t);
template cudaError_t run_reduce<float>(const ReducePlan&, const float*, float*, float, char*,
                                       cudaStream_t);
template cudaError_t run_reduce_host<double>(const ReducePlan&, const double*, double*, double*,
                                             double, char*, cudaStream_t, int64_t);
template cudaError_t run_reduce_host<float>(const ReducePlan&, const float*, float*, float*,
                                            float, char*, cudaStream_t, int64_t);

}  // namespace cr
