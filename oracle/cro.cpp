// Oracle for the canonical reduction and the canonical scan policies.
//
// TEST INFRASTRUCTURE ONLY. This is a plain, slow, single-threaded CPU
// evaluator of the named expressions. Only tests/, __graft_entry__.smoke()
// and bench.py's cpu_baseline / reference leg may load, call or run it. The
// CUDA library never includes, links or calls anything here, and nothing here
// includes or calls the CUDA library.
//
// Source of the definitions: "Canonical Parallel Reduction and Scan"
// (github README andyD123/canonical-reduce):
//   * P4016R0, Key Design Points: the input is split across L interleaved
//     lanes by i mod L; each lane is reduced by the iterative pairwise
//     (shift-reduce) tree; the lane results are combined by the same tree
//     rule; init is combined once after the tree as op(init, R).
//   * P4229R0, Summary and Key Design Points: named expression policies
//     left_fold, pairwise, iterated_pairwise and block_dyadic<B>; a scan
//     returns the prefix observations of the named expression and a reduce
//     returns its root; consistency means
//     inclusive_scan<E>(xs)[i] == reduce<E>(xs[0..i+1)).
//
// Readings where the page is silent (each one stated here is the one the CUDA
// library implements too):
//   * tree(): operands are pushed left to right; whenever the two topmost
//     partial trees cover equally many operands they are replaced by
//     op(lower, upper); at the end the remaining partial trees are folded
//     from the top down, op(below, above).
//   * empty lanes (n < L) are omitted, not filled with an identity.
//   * pairwise scan: y[i] folds the maximal complete subtrees that cover
//     x[0..i] from the left; iterated_pairwise folds the same subtrees from
//     the right (it is tree(x[0..i])).
//   * block_dyadic<B> (reading A): iterated_pairwise inside each block of B
//     operands, blocks chained left to right by a running carry.
//   * block_dyadic_alt<B> (reading B, kept for comparison only): left fold
//     inside each block, tree() across the block results.
//   * exclusive scan and include_initial (the inclusive/exclusive duality of
//     the page "Vertical scan redesign: research notes", section B.2; init
//     placement of P4016R0): with y the inclusive scan, out[0] = init and
//     out[k] = op(init, y[k-1]); exclusive has n outputs, include_initial
//     n + 1.
//
// Arithmetic: op is IEEE-754 addition in the element type, round to nearest
// even; build with -ffp-contract=off and without fast-math (the page's
// cross-platform witness states that FP environment).

#include <cstdint>
#include <cstring>
#include <string>
#include <vector>

namespace {

// ---------------------------------------------------------------- operators
struct AddF64 {
  double operator()(double a, double b) const { return a + b; }
};
struct AddF32 {
  float operator()(float a, float b) const { return a + b; }
};
// A non-associative, non-commutative operator on integers modulo the
// Mersenne prime 2^61 - 1: op(a, b) = 3a + 5b + 1. Used only to check that
// the evaluation structure (which operand goes where) is the specified one.
struct ModP {
  static constexpr uint64_t P = (uint64_t(1) << 61) - 1;
  uint64_t operator()(uint64_t a, uint64_t b) const {
    return (3 * (a % P) + 5 * (b % P) + 1) % P;  // < 8 * 2^61, no overflow
  }
};
// Builds the expression text, so the parenthesisation itself can be read.
struct Sym {
  std::string operator()(const std::string& a, const std::string& b) const {
    return "(" + a + "+" + b + ")";
  }
};

// ------------------------------------------------------- the shift-reduce tree
// A stack of partial trees; size[k] counts the operands under val[k].
template <class V, class Op>
struct ShiftReduce {
  std::vector<V> val;
  std::vector<int64_t> size;

  void push(const V& v, const Op& op) {
    val.push_back(v);
    size.push_back(1);
    while (size.size() >= 2 && size[size.size() - 1] == size[size.size() - 2]) {
      V upper = val.back();
      int64_t s = size.back();
      val.pop_back();
      size.pop_back();
      V lower = val.back();
      val.pop_back();
      size.pop_back();
      val.push_back(op(lower, upper));
      size.push_back(2 * s);
    }
  }
  // The end of the shift-reduce: fold the stack from the top down,
  // val[0] op (val[1] op (... op val[top])). The stack is left unchanged so
  // that a scan can keep pushing.
  V collapse_from_top(const Op& op) const {
    V acc = val.back();
    for (int64_t k = (int64_t)val.size() - 2; k >= 0; --k) acc = op(val[k], acc);
    return acc;
  }
  // Left fold of the same partial trees: ((val[0] op val[1]) op ...) op val[top].
  V fold_from_bottom(const Op& op) const {
    V acc = val[0];
    for (size_t k = 1; k < val.size(); ++k) acc = op(acc, val[k]);
    return acc;
  }
};

// tree(v_0 .. v_{m-1}) for m >= 1 operands read at v[0], v[stride], ...
template <class V, class Op>
V tree(const V* v, int64_t m, int64_t stride, const Op& op) {
  ShiftReduce<V, Op> st;
  for (int64_t t = 0; t < m; ++t) st.push(v[t * stride], op);
  return st.collapse_from_top(op);
}

// ------------------------------------------------------ canonical reduction
// reduce(x, n, L, init) = op(init, tree(R_0 .. R_{m-1})), m = min(n, L),
// R_j = tree(x_j, x_{j+L}, x_{j+2L}, ...). n == 0 gives init.
template <class V, class Op>
V canonical_reduce(const V* x, int64_t n, int64_t stride, int64_t L, const V& init,
                   const Op& op) {
  if (n == 0) return init;
  const int64_t m = n < L ? n : L;
  ShiftReduce<V, Op> across;  // lane results, in lane order
  for (int64_t j = 0; j < m; ++j) {
    ShiftReduce<V, Op> lane;  // lane j holds the operands i with i mod L == j
    for (int64_t i = j; i < n; i += L) lane.push(x[i * stride], op);
    across.push(lane.collapse_from_top(op), op);
  }
  return op(init, across.collapse_from_top(op));
}

// ---------------------------------------------------------- scan policies
enum Policy {
  LEFT_FOLD = 0,
  PAIRWISE = 1,
  ITERATED_PAIRWISE = 2,
  BLOCK_DYADIC = 3,
  BLOCK_DYADIC_ALT = 4
};

// left_fold: y[0] = x[0], y[i] = op(y[i-1], x[i]).
template <class V, class Op>
void scan_left_fold(const V* x, int64_t xs, V* y, int64_t ys, int64_t n, const Op& op) {
  if (n == 0) return;
  V acc = x[0];
  y[0] = acc;
  for (int64_t i = 1; i < n; ++i) {
    acc = op(acc, x[i * xs]);
    y[i * ys] = acc;
  }
}

// iterated_pairwise: y[i] = tree(x[0..i]). The shift-reduce stack after the
// first i+1 pushes is exactly the state tree() reaches on that prefix, so its
// top-down fold is tree(x[0..i]).
template <class V, class Op>
void scan_iterated_pairwise(const V* x, int64_t xs, V* y, int64_t ys, int64_t n,
                            const Op& op) {
  ShiftReduce<V, Op> st;
  for (int64_t i = 0; i < n; ++i) {
    st.push(x[i * xs], op);
    y[i * ys] = st.collapse_from_top(op);
  }
}

// pairwise: the prefix observation of the one tree over all of x. The stack
// after i+1 pushes holds the maximal complete subtrees covering x[0..i];
// y[i] folds them from the left.
template <class V, class Op>
void scan_pairwise(const V* x, int64_t xs, V* y, int64_t ys, int64_t n, const Op& op) {
  ShiftReduce<V, Op> st;
  for (int64_t i = 0; i < n; ++i) {
    st.push(x[i * xs], op);
    y[i * ys] = st.fold_from_bottom(op);
  }
}

// block_dyadic<B>, reading A. Block k covers [kB, min(kB + B, n)).
// P(i) = tree(x[kB..i]); T_k = P(last of block k); C_0 = T_0,
// C_k = op(C_{k-1}, T_k); y[i] = P(i) in block 0, else op(C_{k-1}, P(i)).
template <class V, class Op>
void scan_block_dyadic(const V* x, int64_t xs, V* y, int64_t ys, int64_t n, int64_t B,
                       const Op& op) {
  V carry{};
  for (int64_t k0 = 0, k = 0; k0 < n; k0 += B, ++k) {
    const int64_t end = (k0 + B < n) ? k0 + B : n;
    ShiftReduce<V, Op> blk;
    for (int64_t i = k0; i < end; ++i) {
      blk.push(x[i * xs], op);
      const V p = blk.collapse_from_top(op);
      y[i * ys] = (k == 0) ? p : op(carry, p);
    }
    const V t = blk.collapse_from_top(op);
    carry = (k == 0) ? t : op(carry, t);
  }
}

// block_dyadic_alt<B>, reading B: F_k(i) = left fold of x[kB..i];
// y[i] = tree(T_0, ..., T_{k-1}, F_k(i)) with T_k the full-block folds.
template <class V, class Op>
void scan_block_dyadic_alt(const V* x, int64_t xs, V* y, int64_t ys, int64_t n, int64_t B,
                           const Op& op) {
  ShiftReduce<V, Op> totals;
  for (int64_t k0 = 0; k0 < n; k0 += B) {
    const int64_t end = (k0 + B < n) ? k0 + B : n;
    V f = x[k0 * xs];
    for (int64_t i = k0; i < end; ++i) {
      if (i > k0) f = op(f, x[i * xs]);
      ShiftReduce<V, Op> st = totals;  // tree over the prefix of block values
      st.push(f, op);
      y[i * ys] = st.collapse_from_top(op);
    }
    totals.push(f, op);
  }
}

template <class V, class Op>
int scan(const V* x, int64_t xs, V* y, int64_t ys, int64_t n, int policy, int64_t B,
         const Op& op) {
  switch (policy) {
    case LEFT_FOLD: scan_left_fold(x, xs, y, ys, n, op); return 0;
    case PAIRWISE: scan_pairwise(x, xs, y, ys, n, op); return 0;
    case ITERATED_PAIRWISE: scan_iterated_pairwise(x, xs, y, ys, n, op); return 0;
    case BLOCK_DYADIC:
      if (B < 1) return -1;
      scan_block_dyadic(x, xs, y, ys, n, B, op);
      return 0;
    case BLOCK_DYADIC_ALT:
      if (B < 1) return -1;
      scan_block_dyadic_alt(x, xs, y, ys, n, B, op);
      return 0;
    default: return -1;
  }
}

// Exclusive scan (m = n outputs) or include_initial (m = n + 1 outputs):
// out[0] = init, out[k] = op(init, y[k-1]) for 1 <= k < m, where y is the
// inclusive scan of the policy. init is combined once, as the left operand,
// after the expression, as the reduction combines it with its root.
template <class V, class Op>
int scan_with_init(const V* x, int64_t xs, V* out, int64_t os, int64_t n, int policy,
                   int64_t B, const V& init, bool include_initial, const Op& op) {
  std::vector<V> y((size_t)n);
  if (scan(x, xs, y.data(), 1, n, policy, B, op)) return -1;
  const int64_t m = include_initial ? n + 1 : n;
  if (m == 0) return 0;
  out[0] = init;
  for (int64_t k = 1; k < m; ++k) out[k * os] = op(init, y[(size_t)(k - 1)]);
  return 0;
}

// reduce<E>(x): the root of the named expression, evaluated directly from
// its definition (not from a scan), for n >= 1.
template <class V, class Op>
int reduce_policy(const V* x, int64_t xs, int64_t n, int policy, int64_t B, const Op& op,
                  V* out) {
  if (n < 1) return -1;
  switch (policy) {
    case LEFT_FOLD: {
      V acc = x[0];
      for (int64_t i = 1; i < n; ++i) acc = op(acc, x[i * xs]);
      *out = acc;
      return 0;
    }
    case PAIRWISE:
    case ITERATED_PAIRWISE:
      *out = tree(x, n, xs, op);
      return 0;
    case BLOCK_DYADIC: {  // C_0 = tree(block 0), C_k = op(C_{k-1}, tree(block k))
      if (B < 1) return -1;
      V c = tree(x, (B < n ? B : n), xs, op);
      for (int64_t k0 = B; k0 < n; k0 += B) {
        const int64_t len = (k0 + B < n) ? B : n - k0;
        c = op(c, tree(x + k0 * xs, len, xs, op));
      }
      *out = c;
      return 0;
    }
    case BLOCK_DYADIC_ALT: {  // tree over the left folds of the blocks
      if (B < 1) return -1;
      std::vector<V> folds;
      for (int64_t k0 = 0; k0 < n; k0 += B) {
        const int64_t end = (k0 + B < n) ? k0 + B : n;
        V f = x[k0 * xs];
        for (int64_t i = k0 + 1; i < end; ++i) f = op(f, x[i * xs]);
        folds.push_back(f);
      }
      *out = tree(folds.data(), (int64_t)folds.size(), 1, op);
      return 0;
    }
    default: return -1;
  }
}

std::vector<std::string> leaves(int64_t n) {
  std::vector<std::string> v;
  v.reserve(n);
  for (int64_t i = 0; i < n; ++i) v.push_back("x" + std::to_string(i));
  return v;
}

int64_t put_text(const std::string& s, char* buf, int64_t cap) {
  if (buf && cap > 0) {
    const int64_t k = (int64_t)s.size() < cap - 1 ? (int64_t)s.size() : cap - 1;
    std::memcpy(buf, s.data(), (size_t)k);
    buf[k] = '\0';
  }
  return (int64_t)s.size();
}

}  // namespace

// ================================================================ C exports
extern "C" {

// ---- the shift-reduce tree on its own
double cro_tree_f64(const double* v, int64_t m, int64_t stride) {
  return tree(v, m, stride, AddF64{});
}
float cro_tree_f32(const float* v, int64_t m, int64_t stride) {
  return tree(v, m, stride, AddF32{});
}

// ---- canonical reduction, one sequence (stride in elements)
double cro_reduce_f64(const double* x, int64_t n, int64_t stride, int64_t L, double init) {
  return canonical_reduce(x, n, stride, L, init, AddF64{});
}
float cro_reduce_f32(const float* x, int64_t n, int64_t stride, int64_t L, float init) {
  return canonical_reduce(x, n, stride, L, init, AddF32{});
}
uint64_t cro_reduce_modp(const uint64_t* x, int64_t n, int64_t L, uint64_t init) {
  return canonical_reduce(x, n, 1, L, init, ModP{});
}

// ---- canonical reduction, batch of sequences: sequence b, element i at
// x[b * batch_stride + i * elem_stride]; out[b] receives its result.
void cro_reduce_batched_f64(const double* x, double* out, int64_t batch, int64_t n,
                            int64_t elem_stride, int64_t batch_stride, int64_t L,
                            double init) {
  for (int64_t b = 0; b < batch; ++b)
    out[b] = canonical_reduce(x + b * batch_stride, n, elem_stride, L, init, AddF64{});
}
void cro_reduce_batched_f32(const float* x, float* out, int64_t batch, int64_t n,
                            int64_t elem_stride, int64_t batch_stride, int64_t L,
                            float init) {
  for (int64_t b = 0; b < batch; ++b)
    out[b] = canonical_reduce(x + b * batch_stride, n, elem_stride, L, init, AddF32{});
}

// ---- inclusive scans; policy codes: 0 left_fold, 1 pairwise,
// 2 iterated_pairwise, 3 block_dyadic<B>, 4 block_dyadic_alt<B>.
// Return 0, or -1 for an unknown policy or B < 1.
int cro_scan_f64(const double* x, int64_t xs, double* y, int64_t ys, int64_t n, int policy,
                 int64_t B) {
  return scan(x, xs, y, ys, n, policy, B, AddF64{});
}
int cro_scan_f32(const float* x, int64_t xs, float* y, int64_t ys, int64_t n, int policy,
                 int64_t B) {
  return scan(x, xs, y, ys, n, policy, B, AddF32{});
}
int cro_scan_modp(const uint64_t* x, uint64_t* y, int64_t n, int policy, int64_t B) {
  return scan(x, 1, y, 1, n, policy, B, ModP{});
}
// Batched scans: the output uses the input's strides.
int cro_scan_batched_f64(const double* x, double* y, int64_t batch, int64_t n,
                         int64_t elem_stride, int64_t batch_stride, int policy, int64_t B) {
  for (int64_t b = 0; b < batch; ++b) {
    const int rc = scan(x + b * batch_stride, elem_stride, y + b * batch_stride,
                        elem_stride, n, policy, B, AddF64{});
    if (rc) return rc;
  }
  return 0;
}
int cro_scan_batched_f32(const float* x, float* y, int64_t batch, int64_t n,
                         int64_t elem_stride, int64_t batch_stride, int policy, int64_t B) {
  for (int64_t b = 0; b < batch; ++b) {
    const int rc = scan(x + b * batch_stride, elem_stride, y + b * batch_stride,
                        elem_stride, n, policy, B, AddF32{});
    if (rc) return rc;
  }
  return 0;
}

// ---- exclusive scan (mode 0, n outputs) and include_initial (mode 1,
// n + 1 outputs), output element k at out[k * out_stride]; batched forms
// take the output's own strides (sequence b, element k at
// out[b * out_batch_stride + k * out_elem_stride]).
int cro_scan_ex_f64(const double* x, int64_t xs, double* out, int64_t os, int64_t n,
                    int policy, int64_t B, double init, int mode) {
  if (mode != 0 && mode != 1) return -1;
  return scan_with_init(x, xs, out, os, n, policy, B, init, mode == 1, AddF64{});
}
int cro_scan_ex_f32(const float* x, int64_t xs, float* out, int64_t os, int64_t n,
                    int policy, int64_t B, float init, int mode) {
  if (mode != 0 && mode != 1) return -1;
  return scan_with_init(x, xs, out, os, n, policy, B, init, mode == 1, AddF32{});
}
int cro_scan_ex_modp(const uint64_t* x, uint64_t* out, int64_t n, int policy, int64_t B,
                     uint64_t init, int mode) {
  if (mode != 0 && mode != 1) return -1;
  return scan_with_init(x, 1, out, 1, n, policy, B, init, mode == 1, ModP{});
}
int cro_scan_ex_batched_f64(const double* x, double* out, int64_t batch, int64_t n,
                            int64_t elem_stride, int64_t batch_stride,
                            int64_t out_elem_stride, int64_t out_batch_stride, int policy,
                            int64_t B, double init, int mode) {
  if (mode != 0 && mode != 1) return -1;
  for (int64_t b = 0; b < batch; ++b) {
    const int rc = scan_with_init(x + b * batch_stride, elem_stride, out + b * out_batch_stride,
                                  out_elem_stride, n, policy, B, init, mode == 1, AddF64{});
    if (rc) return rc;
  }
  return 0;
}
int cro_scan_ex_batched_f32(const float* x, float* out, int64_t batch, int64_t n,
                            int64_t elem_stride, int64_t batch_stride,
                            int64_t out_elem_stride, int64_t out_batch_stride, int policy,
                            int64_t B, float init, int mode) {
  if (mode != 0 && mode != 1) return -1;
  for (int64_t b = 0; b < batch; ++b) {
    const int rc = scan_with_init(x + b * batch_stride, elem_stride, out + b * out_batch_stride,
                                  out_elem_stride, n, policy, B, init, mode == 1, AddF32{});
    if (rc) return rc;
  }
  return 0;
}

// ---- reduce<E>, computed from the expression's own definition
int cro_reduce_policy_f64(const double* x, int64_t n, int policy, int64_t B, double* out) {
  return reduce_policy(x, 1, n, policy, B, AddF64{}, out);
}
int cro_reduce_policy_f32(const float* x, int64_t n, int policy, int64_t B, float* out) {
  return reduce_policy(x, 1, n, policy, B, AddF32{}, out);
}
int cro_reduce_policy_modp(const uint64_t* x, int64_t n, int policy, int64_t B,
                           uint64_t* out) {
  return reduce_policy(x, 1, n, policy, B, ModP{}, out);
}

// ---- symbolic forms: operands are named x0, x1, ...; init is named I.
// Each writes the expression text (NUL-terminated, truncated to cap) and
// returns its full length, or -1 on bad arguments.
int64_t cro_sym_tree(int64_t m, char* buf, int64_t cap) {
  if (m < 1) return -1;
  const auto v = leaves(m);
  return put_text(tree(v.data(), m, 1, Sym{}), buf, cap);
}
int64_t cro_sym_reduce(int64_t n, int64_t L, char* buf, int64_t cap) {
  if (n < 0 || L < 1) return -1;
  const auto v = leaves(n);
  return put_text(canonical_reduce(v.data(), n, 1, L, std::string("I"), Sym{}), buf, cap);
}
int64_t cro_sym_scan(int64_t n, int policy, int64_t B, int64_t i, char* buf, int64_t cap) {
  if (n < 1 || i < 0 || i >= n) return -1;
  const auto v = leaves(n);
  std::vector<std::string> y((size_t)n);
  if (scan(v.data(), 1, y.data(), 1, n, policy, B, Sym{})) return -1;
  return put_text(y[(size_t)i], buf, cap);
}
int64_t cro_sym_scan_ex(int64_t n, int policy, int64_t B, int mode, int64_t k, char* buf,
                        int64_t cap) {
  const int64_t m = (mode == 1) ? n + 1 : n;
  if (n < 0 || (mode != 0 && mode != 1) || k < 0 || k >= m) return -1;
  const auto v = leaves(n);
  std::vector<std::string> y((size_t)m);
  if (scan_with_init(v.data(), 1, y.data(), 1, n, policy, B, std::string("I"), mode == 1,
                     Sym{}))
    return -1;
  return put_text(y[(size_t)k], buf, cap);
}
int64_t cro_sym_reduce_policy(int64_t n, int policy, int64_t B, char* buf, int64_t cap) {
  const auto v = leaves(n);
  std::string out;
  if (reduce_policy(v.data(), 1, n, policy, B, Sym{}, &out)) return -1;
  return put_text(out, buf, cap);
}

}  // extern "C"
