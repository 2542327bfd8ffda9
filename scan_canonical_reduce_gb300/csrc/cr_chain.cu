// Exact parallel evaluation of a floating-point left fold
//     C_0 = T_0,   C_k = fl(C_{k-1} + T_k)   (round to nearest even)
// the carry chain of block_dyadic<B> (P4229R0 on "Canonical Parallel
// Reduction and Scan": blocks chained left to right) and the whole 1-D
// left_fold scan. The result is bit-identical to the serial chain.
//
// Why it can be parallel. Let u_e = 2^(e - p) be the unit in the last place
// of binade e (|v| in [2^e, 2^(e+1)), p = 52 or 23 fraction bits). If C_{k-1}
// is an integer multiple M of u_e and the exact sum s = C_{k-1} + T_k lies in
// binade e, then fl(s) = u_e * RNE(M + T_k/u_e). With T_k/u_e = q + f
// (q integer, 0 <= f < 1): fl(s)/u_e = A + d, A = M + q, d = [f > 1/2] or,
// for f exactly 1/2, [A odd] (ties to even). When the sum drops to a lower
// binade e' (u_e' = u_e / 2^j), C_{k-1} = (2^j M) u_e' is still a multiple
// of the new unit, so the step is M -> 2^j M + q + d in the new unit. Every
// such step is an integer map
//     M -> a M + b[parity(M)],     a = 2^j,
// and these maps compose associatively (first g, then h):
//     a = a_h a_g,  b[p] = a_h b_g[p] + b_h[p'],  p' = parity(a_g M + b_g[p]).
// Arithmetic is modulo 2^64: every true intermediate is below 2^54 in
// magnitude whenever the steps are valid, so the residues are the values.
// What cannot compose is a rise to a higher binade (the sum is rounded to a
// coarser unit: an exact division by 2^j with round-half-even) and a step
// whose binade is uncertain (a real add). These are "breaks", evaluated in
// order by one thread from integers only (real adds only when uncertain).
// A rise by d after the thread's own steps since its last break have dropped
// j >= d binades is the exception: 2^j M is then a multiple of 2^d, so the
// rounding no longer depends on M's low bits and the rise folds into the map
// (fold_rise). A chain that oscillates across binade boundaries rises mostly
// back into binades it just left, so most rises fold.
//
// Passes (tile = 4096 steps, 16 consecutive steps per thread):
//   1 tile sums and the largest |T| of each tile (coalesced);
//   2 tile offsets and a bound B >= max |P_k| (one block);
//   3 classify: the approximate prefix P~_k (in registers) and the binade
//     and sign of s_k from it, certain when the whole interval P~_k +- mu
//     (mu = K ulp(2B) bounds both |C_k - P_k| and |P~_k - P_k|) lies inside
//     one binade, decided on the bits with integers only; step types MAP
//     (same or lower binade, or a folded rise), UP (higher binade, integer
//     break), FP (uncertain: real add); each thread's composed map after its
//     last break, scanned across the tile;
//   5 segment bases (one block), 6 segment records: each break and the
//     composed map of the MAP steps that follow it in its tile; the steps
//     before a tile's first break are folded into the previous tile's last
//     segment by a small link pass, so the walk sees breaks only;
//   7 walk: the breaks in order, from integers; M entering every segment;
//   8 fill: every MAP step recomputed from its segment's entry value with an
//     exact 128-bit test that s_k lies in the predicted binade and sign;
//   9 if any test failed (or the segment buffer overflowed), the serial chain
//     recomputes everything on the device (no host sync).
// mu is a rigorous bound for binary64, where K ulp stays small against the
// values for chains of any practical length. Binary32 chains (24-bit
// rounding over K steps) are classified against an estimate of the binary32
// chain itself with a statistical margin instead (passes 1 to 4 below, see
// "binary32"); the checks of passes 8 and 9 are the same.
// Every add of the chain is therefore the real add or proven equal to it.
#include <atomic>
#include <cstdint>

#include "cr_chain.h"
#include "cr_chain_map.h"
#include "cr_device.cuh"
#include "cr_launch.h"

namespace cr {
namespace {

constexpr int kCT = 256;           // threads per tile
constexpr int kCE = 16;            // steps per thread
constexpr int kCTile = kCT * kCE;  // 4096 steps per tile
constexpr int kPublishBatches = 16;  // fused form: the walk's progress every 512 records

template <class T>
struct FP;
template <>
struct FP<double> {
  using U = uint64_t;
  static constexpr int P = 52, BIAS = 1023, EMIN = -1022, EMAX = 1023, W = 64;
  __device__ static U bits(double v) { return (U)__double_as_longlong(v); }
  __device__ static double from_bits(U b) { return __longlong_as_double((long long)b); }
};
template <>
struct FP<float> {
  using U = uint32_t;
  static constexpr int P = 23, BIAS = 127, EMIN = -126, EMAX = 127, W = 32;
  __device__ static U bits(float v) { return (U)__float_as_uint(v); }
  __device__ static float from_bits(U b) { return __uint_as_float(b); }
};

// ---- step meta word: type, certain, negative, f class, jump d, binade e
enum : uint32_t { kMap = 0, kUp = 1, kFp = 2, kStart = 3 };
enum : uint32_t { kFZero = 0, kFLow = 1, kFHalf = 2, kFHigh = 3 };
__device__ __forceinline__ uint32_t make_meta(uint32_t type, bool certain, bool neg,
                                              uint32_t fcls, int d, int e) {
  return type | (certain ? 4u : 0u) | (neg ? 8u : 0u) | (fcls << 4) | ((uint32_t)d << 6) |
         ((uint32_t)(e + 2048) << 12);
}
__device__ __forceinline__ uint32_t m_type(uint32_t m) { return m & 3u; }
__device__ __forceinline__ bool m_certain(uint32_t m) { return m & 4u; }
__device__ __forceinline__ bool m_neg(uint32_t m) { return m & 8u; }
__device__ __forceinline__ uint32_t m_fcls(uint32_t m) { return (m >> 4) & 3u; }
__device__ __forceinline__ int m_d(uint32_t m) { return (int)((m >> 6) & 63u); }
__device__ __forceinline__ int m_e(uint32_t m) { return (int)((m >> 12) & 0xFFFu) - 2048; }
// A rise folded into its run's map (type kMap; d is the rise, q and the f
// class split T in the old unit, as for kUp).
constexpr uint32_t kFolded = 1u << 24;
__device__ __forceinline__ bool m_folded(uint32_t m) { return (m & kFolded) != 0; }

// ---- integer maps M -> a M + b[parity(M)] (mod 2^64): cr_chain_map.h
__device__ __forceinline__ uint32_t delta(uint32_t fcls, uint64_t parity) {
  return fcls == kFHigh ? 1u : (fcls == kFHalf ? (uint32_t)(parity & 1) : 0u);
}
// A MAP step: M -> 2^d M + q + delta, delta from the parity of A = 2^d M + q.
__device__ __forceinline__ Map step_map(int d, int64_t q, uint32_t fcls) {
  const uint64_t uq = (uint64_t)q, a = d >= 64 ? 0 : (uint64_t(1) << d);
  if (d == 0) return Map{1, uq + delta(fcls, uq & 1), uq + delta(fcls, (uq & 1) ^ 1)};
  const uint64_t b = uq + delta(fcls, uq & 1);  // 2^d M is even
  return Map{a, b, b};
}

// ---- exact conversions between T values and (integer, binade) pairs
// unit of binade e as T (exact, possibly subnormal)
template <class T>
__device__ __forceinline__ T unit_of(int e) {
  using F = FP<T>;
  const int ue = e - F::P;
  typename F::U b;
  if (ue >= F::EMIN) b = (typename F::U)(ue + F::BIAS) << F::P;
  else b = (typename F::U)1 << (ue - (F::EMIN - F::P));
  return F::from_bits(b);
}
template <class T>
__device__ __forceinline__ T m_to_value(int64_t M, int e) {  // M * u_e, exact when valid
  return (T)M * unit_of<T>(e);
}
// value -> M with value = M u_e exactly; false if not an integer multiple or
// the multiple does not fit
template <class T>
__device__ __forceinline__ bool value_to_m(T v, int e, int64_t& M) {
  using F = FP<T>;
  const typename F::U b = F::bits(v);
  const int bexp = (int)((b >> F::P) & ((1u << (F::W - 1 - F::P)) - 1));
  uint64_t mant = (uint64_t)(b & ((typename F::U(1) << F::P) - 1));
  if (bexp == (1 << (F::W - 1 - F::P)) - 1) return false;  // inf / nan
  if (bexp == 0 && mant == 0) { M = 0; return true; }
  int ev;  // v = mant 2^(ev - P)
  if (bexp == 0) ev = F::EMIN;
  else { mant |= uint64_t(1) << F::P; ev = bexp - F::BIAS; }
  const int sh = ev - e;  // v / u_e = mant 2^sh
  uint64_t m;
  if (sh >= 0) {
    if (sh > 9) return false;
    m = mant << sh;
  } else {
    if (sh < -63) return false;
    if (mant & ((uint64_t(1) << (-sh)) - 1)) return false;
    m = mant >> (-sh);
  }
  const bool neg = (b >> (F::W - 1)) & 1;
  M = neg ? -(int64_t)m : (int64_t)m;
  return true;
}

// The same two conversions with the common case first, integers only: a
// value of binade e itself (M its significand), and an M of one binade
// (|M| in [2^P, 2^(P+1))) inside T's normal range; else the general forms.
template <class T>
__device__ __forceinline__ bool value_to_m_fast(T v, int e, int64_t& M) {
  using F = FP<T>;
  const typename F::U b = F::bits(v);
  const int bexp = (int)((b >> F::P) & ((1u << (F::W - 1 - F::P)) - 1));
  if (bexp != 0 && bexp == e + F::BIAS) {
    const int64_t m = (int64_t)((uint64_t)(b & ((typename F::U(1) << F::P) - 1)) |
                                (uint64_t(1) << F::P));
    M = (b >> (F::W - 1)) ? -m : m;
    return true;
  }
  return value_to_m<T>(v, e, M);
}
template <class T>
__device__ __forceinline__ T m_to_value_fast(int64_t M, int e) {
  using F = FP<T>;
  const uint64_t mag = M < 0 ? (uint64_t)(-M) : (uint64_t)M;
  if ((mag >> F::P) == 1 && e >= F::EMIN && e <= F::EMAX) {
    typename F::U b = ((typename F::U)(e + F::BIAS) << F::P) |
                      (typename F::U)(mag - (uint64_t(1) << F::P));
    if (M < 0) b |= (typename F::U)1 << (F::W - 1);
    return F::from_bits(b);
  }
  return m_to_value<T>(M, e);
}

// T / u_e = q + f, 0 <= f < 1, classified. False when q would not fit.
template <class T>
__device__ __forceinline__ bool split_unit(T t, int e, int64_t& q, uint32_t& fcls) {
  using F = FP<T>;
  const typename F::U b = F::bits(t);
  const int bexp = (int)((b >> F::P) & ((1u << (F::W - 1 - F::P)) - 1));
  uint64_t mant = (uint64_t)(b & ((typename F::U(1) << F::P) - 1));
  if (bexp == (1 << (F::W - 1 - F::P)) - 1) return false;  // inf / nan
  if (bexp == 0 && mant == 0) { q = 0; fcls = kFZero; return true; }
  int et;  // t = mant * 2^et
  if (bexp == 0) et = F::EMIN - F::P;
  else { mant |= uint64_t(1) << F::P; et = bexp - F::BIAS - F::P; }
  const bool neg = (b >> (F::W - 1)) & 1;
  const int sh = et - (e - F::P);  // t / u = mant * 2^sh
  if (sh >= 0) {
    if (sh > 62 - F::P - 1) return false;
    const int64_t v = (int64_t)(mant << sh);
    q = neg ? -v : v;
    fcls = kFZero;
    return true;
  }
  const int r = -sh;
  if (r >= 62) {  // 0 < |t/u| < 2^-9: floor is 0 or -1
    q = neg ? -1 : 0;
    fcls = neg ? kFHigh : kFLow;
    return true;
  }
  const uint64_t a = mant >> r, rem = mant & ((uint64_t(1) << r) - 1);
  const uint64_t half = uint64_t(1) << (r - 1);
  if (!neg) {
    q = (int64_t)a;
    fcls = rem == 0 ? kFZero : (rem < half ? kFLow : (rem == half ? kFHalf : kFHigh));
  } else if (rem == 0) {
    q = -(int64_t)a;
    fcls = kFZero;
  } else {  // -(a + rem/2^r) = -(a+1) + (1 - rem/2^r)
    q = -(int64_t)a - 1;
    fcls = rem > half ? kFLow : (rem == half ? kFHalf : kFHigh);
  }
  return true;
}

// s / u = A + f lies in the predicted binade and sign (exact integer test).
template <class T>
__device__ __forceinline__ bool in_binade(__int128 A, bool neg, uint32_t fcls) {
  constexpr int64_t LO = int64_t(1) << FP<T>::P, HI = int64_t(1) << (FP<T>::P + 1);
  if (!neg) return A >= LO && A <= HI - 1;
  const bool fz = fcls == kFZero;
  return (fz ? A <= -LO : A <= -LO - 1) && (fz ? A >= -HI + 1 : A >= -HI);
}

template <class T>
__device__ __forceinline__ bool in_binade64(int64_t A, bool neg, bool fz) {
  constexpr int64_t LO = int64_t(1) << FP<T>::P, HI = int64_t(1) << (FP<T>::P + 1);
  if (!neg) return A >= LO && A <= HI - 1;
  return (fz ? A <= -LO : A <= -LO - 1) && (fz ? A >= -HI + 1 : A >= -HI);
}

// A rise by d binades: M (old unit) -> RNE((M + q + f) / 2^d) in the new
// unit. s / u_new = hi + F with hi = floor(A / 2^d), F = (lo + f) / 2^d;
// round up when F > 1/2, or F == 1/2 and hi is odd. `ok` records whether the
// new sum really lies in the predicted binade and sign (kept off the path
// that computes M, which the walk's next step depends on).
template <class T>
__device__ __forceinline__ uint64_t up_step(uint64_t M, int64_t q, uint32_t fcls, int d,
                                            bool neg, bool& ok) {
  const int64_t A = (int64_t)(M + (uint64_t)q);  // |M| <= 2^54, |q| < 2^62
  const int64_t hi = A >> d;         // floor
  const uint64_t lo = (uint64_t)A & ((uint64_t(1) << d) - 1);
  const uint64_t half = uint64_t(1) << (d - 1);
  const bool fpos = fcls != kFZero;
  const bool rup = lo > half || (lo == half && (fpos || (hi & 1)));
  ok = ok && in_binade64<T>(hi, neg, lo == 0 && !fpos);
  return (uint64_t)(hi + (rup ? 1 : 0));
}

// ---------------------------------------------------------------- runs
// N consecutive elements of a thread's run: 16-byte vector accesses when
// whole and aligned, bounded scalar ones at the tail.
template <class E, int N>
__device__ __forceinline__ void load_run(const E* p, int64_t cnt, E (&v)[N]) {
  constexpr int PER = 16 / sizeof(E);
  if (cnt >= N && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int k = 0; k < N / PER; ++k) {
      const uint4 d = q[k];
#pragma unroll
      for (int j = 0; j < PER; ++j) v[k * PER + j] = reinterpret_cast<const E*>(&d)[j];
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < N; ++e) v[e] = (e < cnt) ? p[e] : E(0);
}
template <class E, int N>
__device__ __forceinline__ void store_run(E* p, int64_t cnt, const E (&v)[N]) {
  constexpr int PER = 16 / sizeof(E);
  if (cnt >= N && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
    uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
    for (int k = 0; k < N / PER; ++k) {
      uint4 d;
#pragma unroll
      for (int j = 0; j < PER; ++j) reinterpret_cast<E*>(&d)[j] = v[k * PER + j];
      q[k] = d;
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < N; ++e)
    if (e < cnt) p[e] = v[e];
}

// ---------------------------------------------------------------- pass 1
// Binary64: per tile, the sum and the largest |T| (compared as bit
// patterns, no floating-point work) of its steps, which feed the offsets and
// the bound of pass 2; and each thread's exclusive prefix within the tile
// over the run of kCE steps the classification gives it, summed exactly as
// the classification would, which starts from the stored value.
__device__ __forceinline__ double block_excl_sum(double v, double* sh_w);
template <class T>
__global__ void __launch_bounds__(kCT) chain_tile_sum_kernel(const T* src, int64_t K,
                                                             double* tsum, double* tmax,
                                                             double* thr_start) {
  __shared__ double sh_w[kCT / 32];
  __shared__ uint64_t sh_m[kCT / 32];
  const unsigned full = 0xffffffffu;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int64_t k0 = (int64_t)blockIdx.x * kCTile + (int64_t)t * kCE;
  const int64_t n = k0 < K ? (K - k0 < kCE ? K - k0 : kCE) : 0;
  T tv[kCE];
  load_run(src + (k0 < K ? k0 : 0), n, tv);
  double sum = 0.0;
  uint64_t mx = 0;
#pragma unroll
  for (int i = 0; i < kCE; ++i) {  // zero past the end
    const double v = (double)tv[i];
    sum += v;
    const uint64_t a = (uint64_t)__double_as_longlong(v) & 0x7FFFFFFFFFFFFFFFull;
    mx = a > mx ? a : mx;
  }
  const double excl = block_excl_sum(sum, sh_w);
  thr_start[(int64_t)blockIdx.x * kCT + t] = excl;
  if (t == kCT - 1) tsum[blockIdx.x] = excl + sum;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t o = __shfl_down_sync(full, mx, off);
    mx = o > mx ? o : mx;
  }
  if (lane == 0) sh_m[w] = mx;
  __syncthreads();
  if (t == 0) {
    uint64_t M = 0;
    for (int i = 0; i < kCT / 32; ++i) M = sh_m[i] > M ? sh_m[i] : M;
    tmax[blockIdx.x] = __longlong_as_double((long long)M);  // NaN patterns stay NaN
  }
}

// ---------------------------------------------------------------- pass 2 / 5
// One block of 1024 threads; thread t owns the contiguous chunk
// [t per, (t + 1) per): its sum, an exclusive scan of the sums across the
// block (warp shuffles, then the warp totals), then its outputs.
template <class V>
__device__ __forceinline__ V block1024_excl(V v, V* sh_w, V& total) {
  const unsigned full = 0xffffffffu;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  V incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const V o = __shfl_up_sync(full, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) sh_w[w] = incl;
  __syncthreads();
  if (w == 0) {
    const V x = sh_w[lane];
    V xi = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const V o = __shfl_up_sync(full, xi, off);
      if (lane >= off) xi += o;
    }
    sh_w[lane] = xi - x;  // exclusive warp offsets
    if (lane == 31) sh_w[32] = xi;
  }
  __syncthreads();
  total = sh_w[32];
  const V r = sh_w[w] + incl - v;
  __syncthreads();
  return r;
}

template <class V>
__global__ void __launch_bounds__(1024) exclusive_scan_1block(const V* in, V* out, int64_t n,
                                                              V* total) {
  __shared__ V sh_w[33];
  const int t = threadIdx.x;
  const int64_t per = (n + 1023) / 1024;
  const int64_t a = t * per, b = a + per < n ? a + per : n;
  V s = V(0);
  for (int64_t i = a; i < b; ++i) s += in[i];
  V tot;
  V run = block1024_excl(s, sh_w, tot);
  for (int64_t i = a; i < b; ++i) {
    const V v = in[i];
    out[i] = run;
    run += v;
  }
  if (t == 0 && total) *total = tot;
}

// Tile offsets (exclusive prefix of the tile sums) and the bound
// B = max over tiles of |offset| + 4096 max|T| >= every |P~_k| (one block).
__global__ void __launch_bounds__(1024) chain_offsets_kernel(const double* tsum,
                                                             const double* tmax, int64_t n,
                                                             double* toff, double* bound) {
  __shared__ double sh_w[33];
  __shared__ double sh_b[32];
  const unsigned full = 0xffffffffu;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int64_t per = (n + 1023) / 1024;
  const int64_t a = t * per, b = a + per < n ? a + per : n;
  double s = 0.0;
  for (int64_t i = a; i < b; ++i) s += tsum[i];
  double tot;
  double run = block1024_excl(s, sh_w, tot);
  double bm = 0.0;
  for (int64_t i = a; i < b; ++i) {
    toff[i] = run;
    double bb = fabs(run) + (double)kCTile * tmax[i];
    if (!(bb <= 1.7e308)) bb = 1.7e308;  // non-finite: every step uncertain
    bm = fmax(bm, bb);
    run += tsum[i];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) bm = fmax(bm, __shfl_down_sync(full, bm, off));
  if (lane == 0) sh_b[w] = bm;
  __syncthreads();
  if (t == 0) {
    double m = 0.0;
    for (int i = 0; i < 32; ++i) m = fmax(m, sh_b[i]);
    *bound = m * (1.0 + 0x1p-40);  // covers the rounding of the bound itself
  }
}

// ---------------------------------------------------------------- pass 3
// mu = Kmu 2^emu as an integer and a power of two, from the bound of pass 2.
struct MuInt {
  int64_t K;
  int em;
  int all_uncertain;
};
template <class T>
__device__ __forceinline__ MuInt mu_from_bound(double bound, int64_t K) {
  const double m2 = 2.0 * bound;
  if (!(m2 < 1e300)) return MuInt{0, 0, 1};
  if (m2 <= 1e-290) return MuInt{1, -930, 0};
  const int e = (int)((FP<double>::bits(m2) >> 52) & 0x7FF) - 1023;
  return MuInt{K, e - FP<T>::P, 0};
}

// The binade e and sign of s from p = P~, certain when [|p| - mu,
// |p| + mu + ulp_T(e)) lies inside [2^e, 2^(e+1)) (and e is well inside T's
// normal range). On the bits of p: |p| = (2^52 + f) 2^(e-52), and with
// mu' = mu / 2^(e-52) = Kmu 2^s the test is f >= ceil(mu') and
// 2^52 - f - ulp_T / 2^(e-52) > floor(mu'): integers only.
template <class T>
__device__ __forceinline__ void classify(double p, const MuInt& mu, bool& certain, bool& neg,
                                         int& e) {
  constexpr int kEMin = FP<T>::EMIN + 2 > -960 ? FP<T>::EMIN + 2 : -960;
  constexpr int kEMax = FP<T>::EMAX - 2 < 996 ? FP<T>::EMAX - 2 : 996;
  const uint64_t b = FP<double>::bits(p);
  neg = (b >> 63) != 0;
  certain = false;
  e = 0;
  if (mu.all_uncertain) return;
  const int ef = (int)((b >> 52) & 0x7FF);
  const int ee = ef - 1023;
  if (ef == 0x7FF || ee < kEMin || ee > kEMax) return;  // also zero and subnormals
  const int64_t f = (int64_t)(b & ((uint64_t(1) << 52) - 1));
  const int sft = mu.em + 52 - ee;
  int64_t t1, t2;  // ceil(mu'), floor(mu')
  if (sft >= 0) {
    if (sft >= 52 || (mu.K >> (52 - sft)) != 0) return;  // mu' = Kmu 2^sft >= 2^52 > f
    t1 = t2 = mu.K << sft;
  } else if (-sft >= 62) {
    t2 = 0;
    t1 = mu.K > 0 ? 1 : 0;
  } else {
    const int r = -sft;
    t2 = mu.K >> r;
    t1 = t2 + ((mu.K & ((int64_t(1) << r) - 1)) != 0 ? 1 : 0);
  }
  constexpr int64_t c = int64_t(1) << (52 - FP<T>::P);  // ulp_T(e) / 2^(e-52)
  if (f < t1 || (int64_t(1) << 52) - f - c <= t2) return;
  certain = true;
  e = ee;
}

struct Summ {  // composition after the last break of a thread's steps
  Map map;
  int brk;
};
__device__ __forceinline__ Summ combine(const Summ& l, const Summ& r) {
  return r.brk ? Summ{r.map, l.brk + r.brk} : Summ{compose(l.map, r.map), l.brk};
}

// Exclusive segmented scan of the threads' summaries across the tile.
__device__ __forceinline__ Summ block_summ_scan(Summ me, Summ* sh) {
  const int t = threadIdx.x;
  sh[t] = me;
  __syncthreads();
  for (int off = 1; off < kCT; off <<= 1) {  // inclusive
    Summ a = sh[t];
    if (t >= off) a = combine(sh[t - off], a);
    __syncthreads();
    sh[t] = a;
    __syncthreads();
  }
  const Summ r = t > 0 ? sh[t - 1] : Summ{map_id(), 0};
  __syncthreads();
  return r;
}

// Exclusive sum of one double per thread across the block (warp shuffles).
__device__ __forceinline__ double block_excl_sum(double v, double* sh_w) {
  const unsigned full = 0xffffffffu;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  double incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(full, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) sh_w[w] = incl;
  __syncthreads();
  double base = 0.0;
  for (int i = 0; i < w; ++i) base += sh_w[i];
  __syncthreads();
  return base + incl - v;
}

// The type, integer offset and meta word of step k from its classification
// (certain c, sign ng, binade e) and the previous step's (pc, pe), and the
// thread's composed map after it (me; nbrk counts breaks).
template <class T>
__device__ __forceinline__ void step_record(int64_t k, T t, bool c, bool ng, int e, bool pc,
                                            int pe, Summ& me, int& nbrk, int64_t& q_out,
                                            uint32_t& m_out) {
  uint32_t type;
  int d = 0;
  int64_t q = 0;
  uint32_t f = 0;
  bool folded = false;
  if (k == 0) {
    type = kStart;
  } else if (!c || !pc) {
    type = kFp;
  } else if (e <= pe) {  // same or lower binade: a composable step
    d = pe - e;
    type = (d <= 63 && split_unit<T>(t, e, q, f)) ? kMap : kFp;
  } else {  // rise: T split in the old (finer) unit; a break unless the
            // run's map since its start or last break dropped far enough
    d = e - pe;
    type = (d <= 8 && split_unit<T>(t, pe, q, f)) ? kUp : kFp;
    if (type == kUp && rise_foldable(me.map, d)) {
      type = kMap;
      folded = true;
    }
  }
  if (type == kFp) {
    d = 0;
    q = 0;
  }
  m_out = make_meta(type, c, ng, f, d, e) | (folded ? kFolded : 0u);
  q_out = q;
  if (type != kMap) {
    me.map = map_id();
    me.brk += 1;
    nbrk += 1;
  } else {
    me.map = folded ? fold_rise(me.map, d, q, f != kFZero) : compose(me.map, step_map(d, q, f));
  }
}

template <class T>
__global__ void __launch_bounds__(kCT) chain_classify_kernel(
    const T* src, int64_t K, const double* toff, const double* thr_start, const double* bound,
    int64_t* qv, uint32_t* meta, int64_t* tile_nseg, Summ* thr_in) {
  __shared__ Summ sh[kCT];
  __shared__ int cnt[kCT / 32];
  const unsigned full = 0xffffffffu;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int64_t tile0 = (int64_t)blockIdx.x * kCTile;
  const int64_t k0 = tile0 + (int64_t)t * kCE;
  const int64_t n = k0 < K ? (K - k0 < kCE ? K - k0 : kCE) : 0;
  const MuInt mu = mu_from_bound<T>(*bound, K);
  T tv[kCE];
  load_run(src + (k0 < K ? k0 : 0), n, tv);
  // P~ just before k0 (the tile-sum pass's prefix of the threads before mine)
  double run = toff[blockIdx.x] + thr_start[(int64_t)blockIdx.x * kCT + t];
  bool pc = false, pneg = false;  // pc, pe: the previous step's certainty and binade
  int pe = 0;
  if (k0 > 0 && n > 0) classify<T>(run, mu, pc, pneg, pe);
  int nbrk = 0;
  Summ me{map_id(), 0};
  constexpr int H = kCE / 2;  // outputs written in two halves: fewer live registers
#pragma unroll
  for (int h = 0; h < 2; ++h) {
  int64_t q_out[H];
  uint32_t m_out[H];
#pragma unroll
  for (int j = 0; j < H; ++j) {
    const int i = h * H + j;
    q_out[j] = 0;
    m_out[j] = 0;
    if (i < n) {
      const int64_t k = k0 + i;
      run += (double)tv[i];
      bool c, ng;
      int e;
      classify<T>(run, mu, c, ng, e);
      step_record<T>(k, tv[i], c, ng, e, pc, pe, me, nbrk, q_out[j], m_out[j]);
      pc = c;
      pe = e;
    }
  }
  const int64_t nh = n - h * H;
  if (nh > 0) {
    store_run(qv + k0 + h * H, nh, q_out);
    store_run(meta + k0 + h * H, nh, m_out);
  }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) nbrk += __shfl_down_sync(full, nbrk, off);
  if (lane == 0) cnt[w] = nbrk;
  const Summ in = block_summ_scan(me, sh);  // synchronises: cnt visible
  thr_in[blockIdx.x * kCT + t] = in;
  if (t == 0) {  // one segment per break
    int total = 0;
    for (int i = 0; i < kCT / 32; ++i) total += cnt[i];
    tile_nseg[blockIdx.x] = total;
  }
}

// ---------------------------------------------------------------- binary32
// A binary32 chain rounds to 24 bits, so over K steps its value drifts from
// the exact prefix P_k by up to K ulp: a bound that rigorous leaves every
// step of a long chain uncertain. For binary32 the classification therefore
// compares against a better approximation of the chain itself and a
// statistical margin; the exact checks of the later passes (and the serial
// chain behind them) keep every result exact whatever the margin.
//
// The approximation is one Jacobi step from the exact prefix. Take the
// binades from P (e of P_k for the sum of step k, ep of P_{k-1} for the
// value before it). A step that stays in or drops to binade e adds T_k to a
// multiple of u_e = 2^(e-23), so its rounding error is RN(T_k / u_e) u_e -
// T_k, known from T_k's bits alone; then A_k = P_k + R_{k-1} with R the sum
// of these errors approximates the exact sum of step k far better than P_k.
// What stays unknown is the rounding of a tie (the chain value's parity
// decides: error +-u/2) and of a rise (the previous value's low bits decide:
// error within +-u/2 of the coarser unit). Counted as zero, they leave the
// approximation a random error with variance V_{k-1} = sum of u^2/4 per tie
// and u^2/12 per rise, and the margin of step k is kF32Sigmas sqrt(V_{k-1}).
// On random-walk chains (the benchmark's U[-1, 1) block totals and left
// folds, normal and power-of-two-scaled values) a host simulation of this
// estimate found the largest error at 3.8 standard deviations over 2^28
// steps. Chains whose rounding is biased for long stretches (positive values
// far below the chain's unit) can leave the estimate off by more; their
// checks then fail and the serial chain recomputes the result.
//
// P and R are kept as 128-bit fixed-point integers, value = I 2^-F, with F
// chosen from the chain's length K and largest |T| so that every prefix fits
// with 7 bits to spare: the sums are exact (each T and each estimated error
// is rounded to the unit once, adding at most K units over the chain, a
// rigorous part of the margin), every thread sees exactly the values its
// neighbours computed, and no binary64 arithmetic is needed (GB300 issues
// two binary64 operations a clock per SM, and integer ones at full rate).
constexpr double kF32Sigmas = 8.0;
using i128 = __int128;
using u128 = unsigned __int128;

// Index of the highest set bit of a nonzero value.
__device__ __forceinline__ int hibit128(u128 v) {
  const uint64_t hi = (uint64_t)(v >> 64);
  return hi ? 127 - __clzll((long long)hi) : 63 - __clzll((long long)(uint64_t)v);
}
__device__ __forceinline__ u128 abs128(i128 v) { return v < 0 ? (u128)(-v) : (u128)v; }

// The fixed-point scale F of a binary32 chain of K steps whose largest |T|
// has the bit pattern maxbits: |every prefix| <= K max|T| < 2^(120 - F).
// False when a T is not finite (every step is then left uncertain).
__device__ __forceinline__ bool fix_scale(uint32_t maxbits, int64_t K, int& F) {
  const int x = (int)((maxbits >> 23) & 0xFF);
  if (x == 0xFF) return false;
  const int emax = x == 0 ? -127 : x - 127;        // max|T| < 2^(emax + 1)
  const int eK = 64 - __clzll((long long)K);        // K < 2^eK
  F = 120 - eK - (emax + 1);
  return true;
}

// t 2^F rounded to the nearest integer (halves away from zero).
__device__ __forceinline__ i128 f32_to_fix(float t, int F) {
  const uint32_t b = __float_as_uint(t);
  const int x = (int)((b >> 23) & 0xFF);
  uint32_t m = b & 0x7FFFFFu;
  if (x == 0xFF || (x == 0 && m == 0)) return 0;
  int et;  // |t| = m 2^et
  if (x == 0) {
    et = -149;
  } else {
    m |= 0x800000u;
    et = x - 150;
  }
  const int sh = et + F;  // <= 96 by the choice of F
  u128 mag;
  if (sh >= 0) mag = (u128)m << sh;
  else if (sh <= -26) mag = 0;
  else mag = (u128)((m + (1u << (-sh - 1))) >> (-sh));
  return (b >> 31) ? -(i128)mag : (i128)mag;
}

// The binade e (|value| in [2^e, 2^(e+1))) of a nonzero fixed-point value.
__device__ __forceinline__ int fix_binade(i128 a, int F) { return hibit128(abs128(a)) - F; }

// Rounding estimate of one binary32 step (see above): sp ~ C_{k-1} and s ~
// the step's exact sum, in fixed point; t = T_k. r: the error RN(s) - s in
// fixed point when known (else 0); v: the variance added when it is not.
__device__ __forceinline__ void f32_round_est(i128 sp, i128 s, float t, int F, i128& r,
                                              double& v) {
  r = 0;
  v = 0.0;
  if (sp == 0 || s == 0) return;
  const int e = fix_binade(s, F), ep = fix_binade(sp, F);
  if (e > 127) return;                           // beyond binary32's range
  const int ue = e - 23 < -149 ? -149 : e - 23;  // binary32 unit of binade e
  if (e > ep) {                                  // a rise: u^2 / 12
    v = __longlong_as_double((long long)(2 * ue - 4 + 1023) << 52) * (4.0 / 3.0);
    return;
  }
  const uint32_t tb = __float_as_uint(t);
  const int tx = (int)((tb >> 23) & 0xFF);
  uint32_t m = tb & 0x7FFFFFu;
  if (tx == 0xFF || (tx == 0 && m == 0)) return;
  int et;  // |t| = m 2^et
  if (tx == 0) {
    et = -149;
  } else {
    m |= 0x800000u;
    et = tx - 150;
  }
  const int sh = ue - et;  // |t| / u = m / 2^sh
  if (sh <= 0) return;     // a multiple of u: added exactly
  uint32_t err;            // |RN(|t|) - |t|| / 2^et
  bool up;
  if (sh >= 25) {  // |t| < u / 2: rounds to zero
    err = m;
    up = false;
  } else {
    const uint32_t U = 1u << sh, rem = m & (U - 1u), half = U >> 1;
    if (rem == half) {  // a tie: u^2 / 4
      v = __longlong_as_double((long long)(2 * ue - 2 + 1023) << 52);
      return;
    }
    up = rem > half;
    err = up ? U - rem : rem;
  }
  const int fs = et + F;  // err 2^et in units of 2^-F
  u128 mag;
  if (fs >= 0) mag = (u128)err << fs;
  else if (fs <= -27) mag = 0;
  else mag = (u128)(((uint64_t)err + (1ull << (-fs - 1))) >> (-fs));
  r = (up != ((tb >> 31) != 0)) ? (i128)mag : -(i128)mag;
}

// The margin of a step in fixed-point units: kF32Sigmas sqrt(V) 2^F,
// rounded up, plus K + 16 units for the rounding of the fixed-point sums
// themselves. 2^126 (every step uncertain) when it does not fit.
__device__ __forceinline__ u128 fix_margin(double V, int F, int64_t K) {
  const u128 huge = (u128)1 << 126;
  if (F < -1000 || F > 1000) return huge;
  const double m = kF32Sigmas * sqrt(V > 0.0 ? V : 0.0) *
                   __longlong_as_double((long long)(F + 1023) << 52);
  const u128 rig = (u128)(uint64_t)K + 16u;
  if (!(m < 0x1p125)) return huge;
  if (m < 1.0) return rig + (m > 0.0 ? 1u : 0u);
  const uint64_t b = (uint64_t)__double_as_longlong(m);
  const int ex = (int)((b >> 52) & 0x7FF) - 1023;  // 0 <= ex < 125
  const uint64_t mant = (b & ((uint64_t(1) << 52) - 1)) | (uint64_t(1) << 52);
  const u128 q = ex >= 52 ? (u128)mant << (ex - 52) : (u128)((mant >> (52 - ex)) + 1);
  return q + rig;
}

// The binary32 binade e and sign of the exact sum from its fixed-point
// approximation a, certain when [|a| - mu, |a| + mu + ulp_32(e)) lies inside
// [2^e, 2^(e+1)) (and e well inside binary32's normal range), as classify()
// decides it for a binary64 approximation.
__device__ __forceinline__ void classify_fix(i128 a, u128 mu, int F, bool& certain, bool& neg,
                                             int& e) {
  neg = a < 0;
  certain = false;
  e = 0;
  const u128 m = abs128(a);
  if (m == 0) return;
  const int p = hibit128(m);
  const int ee = p - F;
  if (ee < FP<float>::EMIN + 2 || ee > FP<float>::EMAX - 2) return;
  const u128 lo = (u128)1 << p;
  const u128 ulp = p >= FP<float>::P ? ((u128)1 << (p - FP<float>::P)) : (u128)1;
  if (mu >= lo || m - lo < mu || m + mu + ulp >= 2 * lo) return;
  certain = true;
  e = ee;
}

// Sum of one 128-bit value per thread over the block (thread 0's result).
__device__ __forceinline__ i128 shfl_down128(i128 v, int off) {
  const unsigned full = 0xffffffffu;
  const uint64_t lo = __shfl_down_sync(full, (unsigned long long)(uint64_t)v, off);
  const uint64_t hi = __shfl_down_sync(full, (unsigned long long)(uint64_t)((u128)v >> 64), off);
  return (i128)(((u128)hi << 64) | lo);
}
__device__ __forceinline__ i128 shfl_up128(i128 v, int off) {
  const unsigned full = 0xffffffffu;
  const uint64_t lo = __shfl_up_sync(full, (unsigned long long)(uint64_t)v, off);
  const uint64_t hi = __shfl_up_sync(full, (unsigned long long)(uint64_t)((u128)v >> 64), off);
  return (i128)(((u128)hi << 64) | lo);
}

// Exclusive sum of one 128-bit value per thread across the block (exact).
__device__ __forceinline__ i128 block_excl_sum128(i128 v, i128* sh_w) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  i128 incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const i128 o = shfl_up128(incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) sh_w[w] = incl;
  __syncthreads();
  i128 base = 0;
  for (int i = 0; i < w; ++i) base += sh_w[i];
  __syncthreads();
  return base + incl - v;
}

// Total of one 128-bit value per thread across the block (thread 0).
__device__ __forceinline__ i128 block_sum128(i128 v, i128* sh_w) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += shfl_down128(v, off);
  if (lane == 0) sh_w[w] = v;
  __syncthreads();
  i128 tot = 0;
  if (t == 0)
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += sh_w[i];
  return tot;
}

// Pass 1 (binary32): the largest |T| of the chain, as a bit pattern (NaN
// patterns exceed infinity's: either makes the chain's values non-finite).
__global__ void __launch_bounds__(256) chain_absmax_kernel(const float* src, int64_t K,
                                                           unsigned* maxbits) {
  unsigned m = 0;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < K;
       i += (int64_t)gridDim.x * 256) {
    const unsigned b = __float_as_uint(src[i]) & 0x7FFFFFFFu;
    m = b > m ? b : m;
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0) atomicMax(maxbits, m);
}

// Pass 2 (binary32): per tile, the exact fixed-point sum of T.
__global__ void __launch_bounds__(kCT) chain_fixsum_kernel(const float* src, int64_t K,
                                                           const unsigned* maxbits,
                                                           i128* tsum) {
  __shared__ i128 sh_w[kCT / 32];
  const int t = threadIdx.x;
  const int64_t k0 = (int64_t)blockIdx.x * kCTile + (int64_t)t * kCE;
  const int64_t n = k0 < K ? (K - k0 < kCE ? K - k0 : kCE) : 0;
  int F = 0;
  if (!fix_scale(*maxbits, K, F)) {
    if (t == 0) tsum[blockIdx.x] = 0;
    return;
  }
  float tv[kCE];
  load_run(src + (k0 < K ? k0 : 0), n, tv);
  i128 sum = 0;
#pragma unroll
  for (int i = 0; i < kCE; ++i) sum += f32_to_fix(tv[i], F);  // zero past the end
  const i128 tot = block_sum128(sum, sh_w);
  if (t == 0) tsum[blockIdx.x] = tot;
}

// Exclusive scan of n 128-bit values in one block of 1024 threads (exact).
__global__ void __launch_bounds__(1024) exclusive_scan128_1block(const i128* in, i128* out,
                                                                 int64_t n) {
  __shared__ i128 sh_w[32];
  const int t = threadIdx.x;
  const int64_t per = (n + 1023) / 1024;
  const int64_t a = t * per, b = a + per < n ? a + per : n;
  i128 s = 0;
  for (int64_t i = a; i < b; ++i) s += in[i];
  i128 run = block_excl_sum128(s, sh_w);
  for (int64_t i = a; i < b; ++i) {
    const i128 v = in[i];
    out[i] = run;
    run += v;
  }
}

// Pass 3 (binary32): per tile, the sums of the estimated errors r (fixed
// point) and of their variances v, in the order the classification
// recomputes them. P_{k0-1} enters each thread from the exact tile offsets.
__global__ void __launch_bounds__(kCT) chain_round_sum_kernel(const float* src, int64_t K,
                                                              const unsigned* maxbits,
                                                              const i128* toff, i128* rsum,
                                                              double* vsum, i128* thr_s,
                                                              i128* thr_r, double* thr_v) {
  __shared__ i128 sh_w[kCT / 32];
  __shared__ double sh_v[kCT / 32];
  const int t = threadIdx.x;
  const int64_t k0 = (int64_t)blockIdx.x * kCTile + (int64_t)t * kCE;
  const int64_t n = k0 < K ? (K - k0 < kCE ? K - k0 : kCE) : 0;
  int F = 0;
  if (!fix_scale(*maxbits, K, F)) {  // not finite: the classification certifies nothing
    if (t == 0) {
      rsum[blockIdx.x] = 0;
      vsum[blockIdx.x] = 0.0;
    }
    return;
  }
  float tv[kCE];
  load_run(src + (k0 < K ? k0 : 0), n, tv);
  i128 tsum_me = 0;
#pragma unroll
  for (int i = 0; i < kCE; ++i) tsum_me += f32_to_fix(tv[i], F);
  i128 S = toff[blockIdx.x] + block_excl_sum128(tsum_me, sh_w);  // P_{k0-1}
  const int64_t gt = (int64_t)blockIdx.x * kCT + t;
  thr_s[gt] = S;
  i128 rs = 0;
  double vs = 0.0;
#pragma unroll
  for (int i = 0; i < kCE; ++i) {
    if (i < n) {
      const i128 sp = S;
      S += f32_to_fix(tv[i], F);
      if (k0 + i > 0) {
        i128 r;
        double v;
        f32_round_est(sp, S, tv[i], F, r, v);
        rs += r;
        vs += v;
      }
    }
  }
  // within the tile, the errors and variances of the threads before mine
  const i128 rx = block_excl_sum128(rs, sh_w);
  const double vx = block_excl_sum(vs, sh_v);
  thr_r[gt] = rx;
  thr_v[gt] = vx;
  if (t == kCT - 1) {
    rsum[blockIdx.x] = rx + rs;
    vsum[blockIdx.x] = vx + vs;
  }
}

// Pass 4 for binary32: as chain_classify_kernel, with A_k = P_k + R_{k-1}
// (fixed point) in place of P_k and a margin per step from V_{k-1}
// (recomputed when V changes: at ties and rises only).
__global__ void __launch_bounds__(kCT) chain_classify_f32_kernel(
    const float* src, int64_t K, const unsigned* maxbits, const i128* thr_s, const i128* thr_r,
    const double* thr_v, const i128* roff, const double* voff, int64_t* qv, uint32_t* meta,
    int64_t* tile_nseg, Summ* thr_in) {
  __shared__ Summ sh[kCT];
  __shared__ int cnt[kCT / 32];
  const unsigned full = 0xffffffffu;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int64_t tile0 = (int64_t)blockIdx.x * kCTile;
  const int64_t k0 = tile0 + (int64_t)t * kCE;
  const int64_t n = k0 < K ? (K - k0 < kCE ? K - k0 : kCE) : 0;
  int F = 0;
  const bool finite = fix_scale(*maxbits, K, F);
  float tv[kCE];
  load_run(src + (k0 < K ? k0 : 0), n, tv);
  const int64_t gt = (int64_t)blockIdx.x * kCT + t;
  i128 S = thr_s[gt];                      // P_{k0-1}
  i128 R = roff[blockIdx.x] + thr_r[gt];   // R_{k0-1}
  double V = voff[blockIdx.x] + thr_v[gt]; // V_{k0-1}
  const u128 all = (u128)1 << 126;  // no step certain
  bool pc = false, pneg = false;  // the previous step's classification, made
  int pe = 0;                     // exactly as its own thread made it
  if (k0 > 0 && n > 0) {
    const float tp = src[k0 - 1];
    i128 rp = 0;
    double vp = 0.0;
    const i128 sp2 = S - f32_to_fix(tp, F);  // P_{k0-2}
    if (k0 - 1 > 0) f32_round_est(sp2, S, tp, F, rp, vp);
    const u128 mp = finite ? fix_margin(V - vp, F, K) : all;
    classify_fix(S + (R - rp), mp, F, pc, pneg, pe);
  }
  u128 mu = finite ? fix_margin(V, F, K) : all;
  int nbrk = 0;
  Summ me{map_id(), 0};
  constexpr int H = kCE / 2;  // outputs written in two halves: fewer live registers
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    int64_t q_out[H];
    uint32_t m_out[H];
#pragma unroll
    for (int j = 0; j < H; ++j) {
      const int i = h * H + j;
      q_out[j] = 0;
      m_out[j] = 0;
      if (i < n) {
        const int64_t k = k0 + i;
        const i128 sp = S;
        S += f32_to_fix(tv[i], F);
        bool c, ng;
        int e;
        classify_fix(S + R, mu, F, c, ng, e);
        step_record<float>(k, tv[i], c, ng, e, pc, pe, me, nbrk, q_out[j], m_out[j]);
        pc = c;
        pe = e;
        if (k > 0) {  // this step's error, for the steps after it
          i128 r;
          double v;
          f32_round_est(sp, S, tv[i], F, r, v);
          R += r;
          if (v != 0.0) {
            V += v;
            if (finite) mu = fix_margin(V, F, K);
          }
        }
      }
    }
    const int64_t nh = n - h * H;
    if (nh > 0) {
      store_run(qv + k0 + h * H, nh, q_out);
      store_run(meta + k0 + h * H, nh, m_out);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) nbrk += __shfl_down_sync(full, nbrk, off);
  if (lane == 0) cnt[w] = nbrk;
  const Summ in = block_summ_scan(me, sh);  // synchronises: cnt visible
  thr_in[blockIdx.x * kCT + t] = in;
  if (t == 0) {  // one segment per break
    int total = 0;
    for (int i = 0; i < kCT / 32; ++i) total += cnt[i];
    tile_nseg[blockIdx.x] = total;
  }
}

// ---------------------------------------------------------------- pass 6

// Segment record: a break (or a tile start inside a run) and the composed
// map of the MAP steps after it, up to the next break or the tile end.
struct SegRec {
  int64_t start;
  Map map;
  int64_t q;        // up: T split in the old unit
  uint64_t tbits;   // start or fp break: the bit pattern of T at the start step
  uint32_t meta;    // meta word of the start step (type kMap marks a continuation)
  int32_t e_prev;   // fp break: binade of the previous step (if certain)
  int32_t prev_certain;
  int32_t nsteps;   // MAP steps in the map
};

// The steps of a tile before its first break (all of them if it has none)
// form no record of their own: their composed map goes to lead[tile] (and
// whether there are any to lead_steps), and the link pass folds it into the
// previous tile's last segment.
template <class T>
__global__ void __launch_bounds__(kCT) chain_segments_kernel(
    const T* src, const int64_t* qv, const uint32_t* meta, int64_t K, const int64_t* seg_base,
    const int64_t* tile_nseg, const Summ* thr_in, SegRec* segs, int64_t seg_cap, Map* lead,
    int* lead_steps, int* fail) {
  // MAP step counts of the records this tile opens (at most one a step),
  // summed here and stored once: no record needs clearing beforehand
  __shared__ int s_steps[kCTile];
  const int t = threadIdx.x;
  const int64_t nrec = tile_nseg[blockIdx.x];
  for (int64_t i = t; i < nrec && i < kCTile; i += kCT) s_steps[i] = 0;
  __syncthreads();
  const int64_t tile0 = (int64_t)blockIdx.x * kCTile;
  const int64_t k0 = tile0 + (int64_t)t * kCE;
  const int64_t n = k0 < K ? (K - k0 < kCE ? K - k0 : kCE) : 0;
  const Summ in = thr_in[blockIdx.x * kCT + t];
  int64_t qr[kCE];
  uint32_t mr[kCE];
  load_run(qv + (k0 < K ? k0 : 0), n, qr);
  load_run(meta + (k0 < K ? k0 : 0), n, mr);
  int64_t ord = in.brk - 1;  // segment open at my first step (-1: the leading run)
  // The open segment's map is in.map then my steps (before my first break),
  // or my steps since my last break. My steps are composed on their own, as
  // the classify pass composed them: a folded rise folds into that map.
  Map local = map_id();
  bool own = false;  // one of my breaks opened the segment
  int steps = 0;  // MAP steps of the open segment seen by this thread
  const int64_t base = seg_base[blockIdx.x];
#pragma unroll
  for (int i = 0; i < kCE; ++i) {
    if (i >= n) break;
    const int64_t k = k0 + i;
    const uint32_t m = mr[i];
    if (m_type(m) != kMap) {
      const Map cur = own ? local : compose(in.map, local);
      if (ord >= 0 && base + ord < seg_cap) {  // close the open segment
        segs[base + ord].map = cur;
        if (steps) atomicAdd(&s_steps[ord], steps);
      } else if (ord < 0) {  // the tile's leading run ends here
        lead[blockIdx.x] = cur;
        if (steps) atomicAdd(&lead_steps[blockIdx.x], steps);
      }
      ord += 1;
      local = map_id();
      own = true;
      steps = 0;
      if (base + ord < seg_cap) {
        SegRec& r = segs[base + ord];
        r.start = k;
        r.meta = m;
        r.q = qr[i];
        r.tbits = (uint64_t)FP<T>::bits(src[k]);
        const uint32_t pm = i > 0 ? mr[i > 0 ? i - 1 : 0] : meta[k > 0 ? k - 1 : 0];
        r.e_prev = m_e(pm);
        r.prev_certain = (k > 0 && m_certain(pm)) ? 1 : 0;
      } else {
        atomicExch(fail, 2);
      }
    } else {
      local = m_folded(m) ? fold_rise(local, m_d(m), qr[i], m_fcls(m) != kFZero)
                          : compose(local, step_map(m_d(m), qr[i], m_fcls(m)));
      steps += 1;
    }
  }
  // my trailing MAP steps belong to the segment still open; the thread
  // holding the tile's last step closes it
  const Map cur = own ? local : compose(in.map, local);
  const int64_t last = (tile0 + kCTile < K ? tile0 + kCTile : K) - 1;
  const bool closer = k0 <= last && last < k0 + kCE;
  if (ord >= 0 && base + ord < seg_cap) {
    if (steps) atomicAdd(&s_steps[ord], steps);
    if (closer) segs[base + ord].map = cur;
  } else if (ord < 0 && n > 0) {  // no break in the tile up to here
    if (steps) atomicAdd(&lead_steps[blockIdx.x], steps);
    if (closer) lead[blockIdx.x] = cur;
  }
  __syncthreads();
  for (int64_t i = t; i < nrec && i < kCTile; i += kCT)
    if (base + i < seg_cap) segs[base + i].nsteps = s_steps[i];
}

// Link pass (one block): a segmented scan over the tiles. State after tile
// u: the last segment r that starts at or before it and the composed map
// from r's start to the end of u. A tile with breaks resets it to (its last
// segment, that segment's map); a tile without composes its leading run on.
// Then entry[u] = the state entering tile u (the fill pass starts u's
// leading run from it), and the segment r whose chain tile u (with breaks)
// ends gets the map up to u's first break: the walk sees breaks only.
struct LinkSt {
  Map map;
  int64_t r;
  int steps;
  int reset;
};
__device__ __forceinline__ LinkSt link_combine(const LinkSt& a, const LinkSt& b) {
  if (b.reset) return b;
  return LinkSt{compose(a.map, b.map), a.r, a.steps + b.steps, a.reset};
}

// Segment maps are read (scan phases) before any is written (last phase, after
// a barrier); a tile's lead slots, touched by one thread only, hold the new
// map in between.
__global__ void __launch_bounds__(1024) chain_link_kernel(const int64_t* tile_nseg,
                                                          const int64_t* seg_base,
                                                          int64_t ntiles, SegRec* segs,
                                                          int64_t seg_cap, Map* lead,
                                                          int* lead_steps, Map* entry,
                                                          int64_t* entry_rec) {
  __shared__ LinkSt sh[1024];
  __shared__ LinkSt last_st;
  const int t = threadIdx.x;
  const int64_t per = (ntiles + 1023) / 1024;
  const int64_t a = t * per, b = a + per < ntiles ? a + per : ntiles;
  auto elem = [&](int64_t u) -> LinkSt {
    const int64_t nb = tile_nseg[u];
    if (nb > 0) {
      const int64_t r = seg_base[u] + nb - 1;
      if (r >= seg_cap) return LinkSt{map_id(), -1, 0, 1};  // overflow: the walk fails
      return LinkSt{segs[r].map, r, segs[r].nsteps, 1};
    }
    return LinkSt{lead[u], -1, lead_steps[u], 0};
  };
  LinkSt agg{map_id(), -1, 0, 0};
  for (int64_t u = a; u < b; ++u) agg = link_combine(agg, elem(u));
  sh[t] = agg;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive
    LinkSt v = sh[t];
    if (t >= off) v = link_combine(sh[t - off], v);
    __syncthreads();
    sh[t] = v;
    __syncthreads();
  }
  LinkSt st = t > 0 ? sh[t - 1] : LinkSt{map_id(), -1, 0, 0};
  for (int64_t u = a; u < b; ++u) {
    entry[u] = st.map;
    entry_rec[u] = st.r;
    const LinkSt e = elem(u);
    if (e.reset) {  // the chain of segment st.r ends at u's first break
      lead[u] = compose(st.map, lead[u]);
      lead_steps[u] = st.steps + lead_steps[u];
    }
    st = link_combine(st, e);
  }
  if (t == 1023) last_st = sh[1023];
  __syncthreads();
  for (int64_t u = a; u < b; ++u) {
    const int64_t r = entry_rec[u];
    if (tile_nseg[u] > 0 && r >= 0 && r < seg_cap) {
      segs[r].map = lead[u];
      segs[r].nsteps = lead_steps[u];
    }
  }
  if (t == 0 && last_st.r >= 0 && last_st.r < seg_cap) {  // the last chain runs to the end
    segs[last_st.r].map = last_st.map;
    segs[last_st.r].nsteps = last_st.steps;
  }
}

// ---------------------------------------------------------------- pass 7
// The walk carries A = M + q, the integer to be rounded at the next break,
// instead of M: the next record's q is folded into this record's map
// offsets, which takes one 64-bit add off the sequential path. A rise by d
// binades rounds A / 2^d half to even in one step,
//   M1 = (A + 2^(d-1) - 1 + x) >> d,   x = fpos | (bit d of A),
// which rounds up exactly when the remainder exceeds half, or equals it and
// either the exact sum lies above A (fpos) or the quotient is odd.
struct alignas(16) Hot {
  uint64_t b0;      // the segment map's offset for an even M, plus the next
                    // record's q when that record is a rise
  int64_t db;       // the offset for an odd M minus b0
  uint32_t ctrl;    // d (4 bits) | sh (6) << 4 | zero map << 10 | fpos << 11 | neg << 12 |
                    // type (2) << 13 | steps << 15
  int32_t c;        // 2^(d-1) - 1 for a rise (d <= 8), 0 otherwise
  uint32_t pad[2];
};
__device__ __forceinline__ bool is_fast(uint32_t meta) { return m_type(meta) <= kUp; }
__device__ __forceinline__ Hot make_hot(const SegRec& r, int64_t q_next) {
  Hot h;
  const uint32_t m = r.meta, type = m_type(m);
  const int d = type == kUp ? m_d(m) : 0;  // a rise spans at most 8 binades
  h.c = d > 0 ? (1 << (d - 1)) - 1 : 0;
  h.b0 = r.map.b0 + (uint64_t)q_next;
  h.db = (int64_t)(r.map.b1 - r.map.b0);
  const bool zero = r.map.a == 0;  // the map multiplies by 2^64 = 0 mod 2^64
  const uint32_t shift = zero ? 0u : (uint32_t)(__ffsll((long long)r.map.a) - 1);
  h.ctrl = (uint32_t)d | (shift << 4) | (zero ? 1u << 10 : 0u) |
           ((m_fcls(m) != kFZero) ? 1u << 11 : 0u) | (m_neg(m) ? 1u << 12 : 0u) |
           (type << 13) | (r.nsteps > 0 ? 1u << 15 : 0u);
  h.pad[0] = h.pad[1] = 0;
  return h;
}
__device__ __forceinline__ uint32_t hot_type(const Hot& h) { return (h.ctrl >> 13) & 3u; }
__device__ __forceinline__ bool hot_steps(const Hot& h) { return (h.ctrl >> 15) & 1u; }

// The map of a record applied to M1, plus the next record's q:
// (M1 2^sh (or 0 for a zero map)) + b0 + (M1 odd ? db : 0).
__device__ __forceinline__ int64_t hot_map(const Hot& h, int64_t M1) {
  const uint32_t ctl = h.ctrl;
  const uint64_t amask = (ctl >> 10) & 1u ? 0ull : ~0ull;
  const uint64_t odd = 0ull - ((uint64_t)M1 & 1ull);
  return (int64_t)((((uint64_t)M1 << ((ctl >> 4) & 63u)) & amask) + h.b0 +
                   (odd & (uint64_t)h.db));
}

// One rise from A: writes m_in, returns the next A. (Whether the rise really
// lands in its predicted binade is checked afterwards, in parallel, by
// chain_verify_kernel, which recomputes A from the previous record.)
template <class T>
__device__ __forceinline__ int64_t walk_fast(const Hot& h, int64_t A, int64_t* m_in_j,
                                             bool& cval) {
  const uint32_t ctl = h.ctrl;
  const int d = (int)(ctl & 15u);  // 1..8: bit d of A lies in its low word
  const uint32_t x = (((uint32_t)A >> d) | (ctl >> 11)) & 1u;
  const int64_t M1 = (A + (int64_t)(h.c + (int32_t)x)) >> d;
  *m_in_j = M1;
  cval = false;  // a rise leaves no real-add value current
  return hot_map(h, M1);
}

// Breaks in order, in one thread. The whole warp converts the next 32
// records to compact form while lane 0 runs the current 32 from shared
// memory; batches with no start or uncertain step run an unrolled loop of
// the integer path alone.
// dst == nullptr: the chain's outputs are not wanted (a reduction); with
// final_out, lane 0 also writes C_{K-1}, taken from the last segment's map
// (e_last: binade of the last step) or from the last real add.
// Run by one warp (lanes 0..31 of the calling block). With progress
// non-null, lane 0 publishes the number of records done every kPublishBatches
// batches and after the last (after a fence, so that their m_in and the
// start and uncertain values in dst are visible first; the fence waits for
// the walk's stores, hence not after every batch).
template <class T>
__device__ __forceinline__ void walk_body(const T* src, T* dst, const SegRec* segs,
                                          const int64_t* nseg_total, int64_t seg_cap,
                                          int64_t* m_in, int* fail, const uint32_t* meta,
                                          int64_t K, T* final_out,
                                          unsigned long long* progress) {
  __shared__ Hot hot[2][32];
  __shared__ T tv_s[2][32];          // each record's T
  __shared__ uint32_t meta_s[2][32];  // each record's meta word
  __shared__ uint32_t ep_s[2][32];    // binade of the step before + 2048 | certain << 16
  __shared__ int64_t st_s[2][32];     // each record's step
  __shared__ unsigned plain_s[2];    // records that are a real add and nothing else
  __shared__ int cold_batch[2];
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x;
  const int64_t nseg = *nseg_total;
  if (*fail || nseg > seg_cap) {
    if (lane == 0) atomicExch(fail, 2);
    return;
  }
  SegRec cur{}, nxt{};
  if (lane < nseg) cur = segs[lane];
  if (32 + lane < nseg) nxt = segs[32 + lane];
  // A = M + q of the next record: M = 0 before the first (in practice a start)
  int64_t A = __shfl_sync(full, (lane == 0 && nseg > 0 && m_type(cur.meta) == kUp) ? cur.q : 0, 0);
  T C = T(0);
  bool cval = false;  // C holds the current chain value
  bool bad = false;
  for (int64_t b0 = 0, it = 0; b0 < nseg; b0 += 32, ++it) {
    const int slot = (int)(it & 1);
    // q of the record after mine (lane 31: the next batch's first record)
    const int64_t q_mine = (b0 + lane < nseg && m_type(cur.meta) == kUp) ? cur.q : 0;
    const int64_t q_nb = (b0 + 32 < nseg && m_type(nxt.meta) == kUp) ? nxt.q : 0;
    int64_t q_next = __shfl_down_sync(full, q_mine, 1);
    const int64_t q_nb0 = __shfl_sync(full, q_nb, 0);
    if (lane == 31) q_next = q_nb0;
    hot[slot][lane] = make_hot(cur, q_next);
    tv_s[slot][lane] = FP<T>::from_bits((typename FP<T>::U)cur.tbits);
    meta_s[slot][lane] = cur.meta;
    ep_s[slot][lane] = (uint32_t)(cur.e_prev + 2048) | (cur.prev_certain ? 1u << 16 : 0u);
    st_s[slot][lane] = cur.start;
    const bool is_cold = b0 + lane < nseg && !is_fast(cur.meta);
    const unsigned any_cold = __ballot_sync(full, is_cold);
    // A real-add record followed directly (no MAP steps) by another: its
    // value is all the walk needs to compute (the next record adds to it;
    // nothing reads its integer form), so runs of them take a short loop.
    const bool me_fp = b0 + lane < nseg && m_type(cur.meta) == kFp;
    const bool nb_fp = b0 + 32 < nseg && m_type(nxt.meta) == kFp;
    bool next_fp = __shfl_down_sync(full, me_fp, 1);
    const bool nb_fp0 = __shfl_sync(full, nb_fp, 0);
    if (lane == 31) next_fp = nb_fp0;
    const unsigned plain = __ballot_sync(full, me_fp && cur.nsteps == 0 && next_fp);
    if (lane == 0) {
      cold_batch[slot] = any_cold != 0;
      plain_s[slot] = plain;
    }
    __syncwarp();
    cur = nxt;
    const int64_t nb = b0 + 64 + lane;
    if (nb < nseg) nxt = segs[nb];
    if (lane == 0) {
      const int cnt = (int)(nseg - b0 < 32 ? nseg - b0 : 32);
      bool ok = true;
      if (!cold_batch[slot]) {
        if (cnt == 32) {  // the next 4 records are loaded while 4 are walked
          Hot cur[4], nxt[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) cur[u] = hot[slot][u];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            if (g < 7) {
#pragma unroll
              for (int u = 0; u < 4; ++u) nxt[u] = hot[slot][(g + 1) * 4 + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) A = walk_fast<T>(cur[u], A, m_in + b0 + g * 4 + u, cval);
            if (g < 7) {
#pragma unroll
              for (int u = 0; u < 4; ++u) cur[u] = nxt[u];
            }
          }
        } else {
          for (int j = 0; j < cnt; ++j) A = walk_fast<T>(hot[slot][j], A, m_in + b0 + j, cval);
        }
      } else {
        // one record at a time, the next record's fields loaded meanwhile
        const unsigned plain = plain_s[slot];
        Hot h = hot[slot][0];
        uint32_t mw = meta_s[slot][0], ew = ep_s[slot][0];
        T tv = tv_s[slot][0];
        int64_t st = st_s[slot][0];
        for (int j = 0; j < cnt; ++j) {
          const int jn = j + 1 < cnt ? j + 1 : j;
          const Hot hn = hot[slot][jn];
          const uint32_t mwn = meta_s[slot][jn], ewn = ep_s[slot][jn];
          const T tvn = tv_s[slot][jn];
          const int64_t stn = st_s[slot][jn];
          const uint32_t type = hot_type(h);
          if (cval && ((plain >> j) & 1u)) {  // a real add, nothing else needed
            C = add_rn(C, tv);
            if (dst != nullptr) dst[st] = C;
          } else if (type <= kUp) {
            A = walk_fast<T>(h, A, m_in + b0 + j, cval);
          } else {
            // start or uncertain step: the real add. The previous record
            // folded no q into A for this one, so A is the entering M.
            if (type == kStart) {
              C = tv;
            } else {
              if (!cval) {
                ok = ok && (ew >> 16);
                C = m_to_value_fast<T>(A, (int)(ew & 0xFFFFu) - 2048);
              }
              C = add_rn(C, tv);
            }
            if (dst != nullptr) dst[st] = C;
            cval = true;
            int64_t M1 = A;
            if (m_certain(mw)) {
              int64_t Mi = 0;
              ok = ok && value_to_m_fast<T>(C, m_e(mw), Mi);
              M1 = Mi;
            }
            m_in[b0 + j] = M1;
            A = hot_map(h, M1);
            cval = cval && !hot_steps(h);
          }
          h = hn;
          mw = mwn;
          ew = ewn;
          tv = tvn;
          st = stn;
        }
      }
      bad = bad || !ok;
      if (bad) atomicExch(fail, 1);
      if (progress != nullptr && ((it + 1) % kPublishBatches == 0 || b0 + 32 >= nseg)) {
        __threadfence();  // m_in and dst before the count that releases them
        atomicExch(progress, (unsigned long long)(b0 + cnt));
      }
    }
    __syncwarp();
  }
  if (lane == 0 && final_out != nullptr && !bad)  // A = M after the last segment's map
    *final_out = cval ? C : m_to_value<T>(A, m_e(meta[K - 1]));
}

template <class T>
__global__ void __launch_bounds__(32) chain_walk_kernel(const T* src, T* dst, const SegRec* segs,
                                                        const int64_t* nseg_total,
                                                        int64_t seg_cap, int64_t* m_in,
                                                        int* fail, const uint32_t* meta,
                                                        int64_t K, T* final_out) {
  walk_body<T>(src, dst, segs, nseg_total, seg_cap, m_in, fail, meta, K, final_out, nullptr);
}

// Every rise of the walk, checked in parallel: A = (previous record's map
// applied to its M) + q must round into the predicted binade and sign
// (integer comparisons on hi = floor(A / 2^d)). A failure sends the chain
// to the serial fallback.
template <class T>
__device__ __forceinline__ void verify_record(const SegRec* segs, const int64_t* m_in, int64_t j,
                                              int* fail) {
  const uint32_t m = segs[j].meta;
  if (j == 0 || m_type(m) != kUp) return;
  const Map g = segs[j - 1].map;
  const int64_t A = (int64_t)apply(g, (uint64_t)__ldcg(m_in + j - 1)) + segs[j].q;
  const int d = m_d(m);
  const int64_t hi = A >> d;
  const uint64_t lo = (uint64_t)A & ((uint64_t(1) << d) - 1);
  const bool fpos = m_fcls(m) != kFZero;
  if (!in_binade64<T>(hi, m_neg(m), lo == 0 && !fpos)) atomicExch(fail, 1);
}

template <class T>
__global__ void __launch_bounds__(256) chain_verify_kernel(const SegRec* segs,
                                                           const int64_t* nseg_total,
                                                           int64_t seg_cap, const int64_t* m_in,
                                                           int* fail) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nseg = *nseg_total;
  if (j >= nseg || j >= seg_cap || *fail) return;
  verify_record<T>(segs, m_in, j, fail);
}

// ---------------------------------------------------------------- pass 8
// M u_e as T from its bits, for M in [2^P, 2^(P+1)] in magnitude (a value of
// binade e, or 2^(e+1) after rounding up at the binade's top) with e well
// inside T's normal range, as every validated step has: integers only.
template <class T>
__device__ __forceinline__ T m_to_value_normal(int64_t M, int e) {
  using F = FP<T>;
  using U = typename F::U;
  const uint64_t mag = M < 0 ? (uint64_t)(-M) : (uint64_t)M;
  U b;
  if (mag >> (F::P + 1)) b = (U)(e + 1 + F::BIAS) << F::P;
  else b = ((U)(e + F::BIAS) << F::P) | (U)(mag - (uint64_t(1) << F::P));
  if (M < 0) b |= (U)1 << (F::W - 1);
  return F::from_bits(b);
}

// The 16 steps of thread t (of kCT) of chain tile c, from its segment's
// entry value, in two parts: fill_prep issues the loads that do not depend
// on the walk (in the fused form, before waiting for it), fill_finish reads
// the walk's results (all of them at once) and evaluates the steps.
struct FillPrep {
  int64_t qr[kCE];    // q of each step; a record step's m_in once read
  uint32_t mr[kCE];
  Map in_map, entry;
  int64_t seg;        // the record before the thread's first step
  int64_t entry_rec;  // no break before the thread: the record its run enters from
  int brk;
  int n;              // steps (0: none)
};

__device__ __forceinline__ void fill_prep(int64_t c, int t, const int64_t* qv,
                                          const uint32_t* meta, int64_t K,
                                          const int64_t* seg_base, const Summ* thr_in,
                                          const Map* entry, const int64_t* entry_rec,
                                          FillPrep& p) {
  const int64_t k0 = c * kCTile + (int64_t)t * kCE;
  p.n = 0;
  if (k0 >= K) return;
  p.n = (int)(K - k0 < kCE ? K - k0 : kCE);
  const Summ in = thr_in[c * kCT + t];
  p.in_map = in.map;
  p.brk = in.brk;
  p.seg = seg_base[c] + in.brk - 1;
  p.entry_rec = -1;
  if (c > 0) {  // the tile's leading run enters from an earlier tile
    p.entry_rec = entry_rec[c];
    p.entry = entry[c];
  }
  load_run(qv + k0, p.n, p.qr);
  load_run(meta + k0, p.n, p.mr);
}

template <class T>
__device__ __forceinline__ void fill_finish(int64_t c, int t, FillPrep& p, int64_t seg_cap,
                                            const int64_t* m_in, T* dst, int* fail) {
  if (p.n == 0) return;
  const int64_t k0 = c * kCTile + (int64_t)t * kCE;
  // the walk's results, read from L2 (__ldcg: in the fused form the walk
  // writes them during this launch), all loads issued together: the entry
  // record's M, each record step's M and the walk's start and uncertain
  // values
  uint64_t Me = 0;
  const bool from_seg = p.brk > 0 && p.seg < seg_cap;
  const bool from_entry = p.brk == 0 && c > 0 && p.entry_rec >= 0 && p.entry_rec < seg_cap;
  if (from_seg) Me = (uint64_t)__ldcg(m_in + p.seg);
  else if (from_entry) Me = (uint64_t)__ldcg(m_in + p.entry_rec);
  T out[kCE];
  {
    int64_t s = p.seg;
#pragma unroll
    for (int i = 0; i < kCE; ++i) {
      out[i] = T(0);
      const uint32_t type = m_type(p.mr[i]);
      if (i < p.n && type != kMap) {
        s += 1;
        if (s < seg_cap) {
          p.qr[i] = __ldcg(m_in + s);
          if (type != kUp && dst != nullptr) out[i] = __ldcg(dst + k0 + i);
        }
      }
    }
  }
  uint64_t M = 0;
  if (from_seg) M = apply(p.in_map, Me);
  else if (from_entry) M = apply(p.in_map, apply(p.entry, Me));
  bool ok = true;
  int64_t seg = p.seg;
#pragma unroll
  for (int i = 0; i < kCE; ++i) {
    if (i < p.n) {
      const uint32_t m = p.mr[i];
      const uint32_t type = m_type(m);
      if (type != kMap) {  // enter the next segment
        seg += 1;
        if (seg >= seg_cap) {
          ok = false;
        } else {
          M = (uint64_t)p.qr[i];
          // the walk wrote start and uncertain steps (read above); keep them
          if (type == kUp) out[i] = m_to_value_normal<T>((int64_t)M, m_e(m));
        }
        continue;
      }
      const int d = m_d(m);
      const uint32_t f = m_fcls(m);
      if (m_folded(m)) {  // a rise folded into its run's map: the rise itself
        M = up_step<T>(M, p.qr[i], f, d, m_neg(m), ok);
        out[i] = m_to_value_normal<T>((int64_t)M, m_e(m));
        continue;
      }
      int64_t A64;
      if (d <= 9) {  // |M 2^d| <= 2^63 / 2 and |q| < 2^62: no overflow
        A64 = (int64_t)(M << d) + p.qr[i];
        if (!in_binade64<T>(A64, m_neg(m), f == kFZero)) ok = false;
      } else {
        const __int128 A = (__int128)(int64_t)M * ((__int128)1 << d) + (__int128)p.qr[i];
        if (!in_binade<T>(A, m_neg(m), f)) ok = false;
        A64 = (int64_t)A;
      }
      M = (uint64_t)(A64 + (int64_t)delta(f, (uint64_t)A64 & 1));
      out[i] = m_to_value_normal<T>((int64_t)M, m_e(m));
    }
  }
  if (dst != nullptr) store_run(dst + k0, p.n, out);  // else: validation only
  if (!ok) atomicExch(fail, 1);
}

template <class T>
__global__ void __launch_bounds__(kCT) chain_fill_kernel(const int64_t* qv, const uint32_t* meta,
                                                         int64_t K, const int64_t* seg_base,
                                                         const Summ* thr_in, const Map* entry,
                                                         const int64_t* entry_rec,
                                                         int64_t seg_cap, const int64_t* m_in,
                                                         T* dst, int* fail) {
  if (*fail) return;
  FillPrep p;
  fill_prep(blockIdx.x, threadIdx.x, qv, meta, K, seg_base, thr_in, entry, entry_rec, p);
  fill_finish<T>(blockIdx.x, threadIdx.x, p, seg_cap, m_in, dst, fail);
}

// ---------------------------------------------------------------- pass 9
// The left fold in one warp, streamed: the warp moves the steps through
// shared memory in buffers of 1024 (coalesced loads and stores) while lane 0
// folds the current buffer; the next buffer's loads are in flight meanwhile.
// With only_if non-null it runs only when *only_if is set (the fallback of
// the parallel evaluation). A buffer is read before any of its results is
// stored, and the next buffer is read before this one's results are stored,
// so dst may equal src.
template <class T>
__global__ void __launch_bounds__(32) chain_serial_kernel(const T* src, T* dst, int64_t K,
                                                          const int* only_if, T* final_out) {
  constexpr int kBuf = 1024, kPer = kBuf / 32;
  __shared__ __align__(16) T buf[kBuf];
  const int lane = threadIdx.x;
  if (only_if != nullptr && *only_if == 0) return;
  // past the end the buffer holds -0.0, the exact identity of the add: the
  // last group's padding steps leave c (and so final_out) unchanged, a -0.0
  // included (+0.0 would turn it into +0.0)
  T nxt[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int64_t k = lane + 32 * i;
    nxt[i] = k < K ? src[k] : -T(0);
  }
  T c = T(0);
  for (int64_t base = 0; base < K; base += kBuf) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) buf[lane + 32 * i] = nxt[i];
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kPer; ++i) {  // the next buffer, in flight during the fold
      const int64_t k = base + kBuf + lane + 32 * i;
      nxt[i] = k < K ? src[k] : -T(0);
    }
    if (lane == 0) {  // 32 steps at a time through registers (16-byte smem moves)
      const int cnt = (int)(K - base < kBuf ? K - base : kBuf);
      constexpr int G = 32, PER = 16 / sizeof(T);
      for (int j0 = 0; j0 < cnt; j0 += G) {
        T v[G];
#pragma unroll
        for (int u = 0; u < G / PER; ++u) {
          const uint4 d = reinterpret_cast<const uint4*>(buf + j0)[u];
#pragma unroll
          for (int w = 0; w < PER; ++w) v[u * PER + w] = reinterpret_cast<const T*>(&d)[w];
        }
        c = (base == 0 && j0 == 0) ? v[0] : add_rn(c, v[0]);  // the chain starts at C_0 = T_0
        v[0] = c;
#pragma unroll
        for (int u = 1; u < G; ++u) {
          c = add_rn(c, v[u]);
          v[u] = c;
        }
#pragma unroll
        for (int u = 0; u < G / PER; ++u) {
          uint4 d;
#pragma unroll
          for (int w = 0; w < PER; ++w) reinterpret_cast<T*>(&d)[w] = v[u * PER + w];
          reinterpret_cast<uint4*>(buf + j0)[u] = d;
        }
      }
    }
    __syncwarp();
    if (dst != nullptr) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int64_t k = base + lane + 32 * i;
        if (k < K) dst[k] = buf[lane + 32 * i];
      }
    }
    __syncwarp();
  }
  if (lane == 0 && final_out != nullptr) *final_out = c;
}

// ---------------------------------------------------------------- fused
// The walk, verify and fill of the chain, fused with the fix-up of a block
// scan that waits for the chain's carries: out[i] = C_{k-1} op out[i] for
// the elements i of blocks k >= 1 (B = 2^logB elements a block). Launched
// cooperatively (every block resident), three roles:
//   block 0, first warp   the walk; publishes how many records are done;
//   blocks 1 .. F         fill tiles c = b - 1, b - 1 + F, ...: wait for the
//                         walk to pass the tile's records, check their rises,
//                         write the tile's carries (a whole block: short
//                         latency), raise the tile's flag;
//   the other blocks      every warp on its own: fix-up items w, w + W, ...
//                         (kFixItem elements each) in order, each after the
//                         flags of the (at most two) tiles holding its
//                         carries, streamed in sub-chunks whose elements and
//                         carries are loaded one sub-chunk ahead.
// Waits run walk <- fills <- fix-up only, so all of them end; each also
// gives up after kWaitLimitNs and sets fail. Any failure (validation,
// overflow, time limit) leaves out partly fixed: the caller's recovery
// passes, which run only when fail is set, recompute the local values, the
// carries (serially) and the fix-up. The fix-up warps need no block
// barrier, so the warps of an SM stay in different phases (loads, FP64
// adds, stores) as a plain streaming kernel's would.
// Fill blocks: at most 96 and a quarter of the resident blocks (48 and a
// third measured alike at B = 16; half of them starve the fix-up).
#ifndef CR_MAX_FILL_BLOCKS
#define CR_MAX_FILL_BLOCKS 96
#endif
constexpr int64_t kMaxFillBlocks = CR_MAX_FILL_BLOCKS;  // (an override changes the schedule only)
constexpr int kFillShareDiv = 4;
constexpr int kFixPer = 16;                    // elements a lane per sub-chunk
constexpr int64_t kFixSub = 32 * kFixPer;      // 512 elements a sub-chunk
constexpr int kFixSubs = 16;                   // sub-chunks an item
constexpr int64_t kFixItem = kFixSub * kFixSubs;  // 8192 elements a warp item
constexpr int kFailTimeout = 3;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second
constexpr uint32_t kWaitMaxSpins = 1u << 24;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One thread: waits until *v >= need (an acquire load: what was written
// before the matching release is visible after it), with a growing sleep.
// Returns false once fail is set, setting it itself at the limit.
template <class V>
__device__ bool wait_at_least(const V* v, unsigned long long need, int* fail) {
  if (ld_acquire(v) >= need) return true;
  const volatile int* vf = fail;
  const uint64_t t0 = global_ns();
  uint32_t spins = 0, ns = 32;
  for (;;) {
    if (*vf != 0) return false;
    if (++spins > kWaitMaxSpins || global_ns() - t0 > kWaitLimitNs) {
      atomicCAS(fail, 0, kFailTimeout);
      return false;
    }
    __nanosleep(ns);
    if (ns < 2048) ns *= 2;
    if (ld_acquire(v) >= need) return true;
  }
}

struct FusedArgs {
  const SegRec* segs;
  const int64_t* total;     // records
  int64_t seg_cap;
  int64_t* m_in;
  int* fail;
  const uint32_t* meta;
  const int64_t* qv;
  int64_t K;                // chain steps
  int64_t ntiles;
  const int64_t* seg_base;  // first record of each tile
  const int64_t* tile_nseg; // records of each tile
  const Summ* thr_in;
  const Map* entry;
  const int64_t* entry_rec;
  unsigned long long* progress;
  unsigned long long* next_item;  // fix-up items handed out so far
  unsigned* tile_done;
  int64_t n;                // fix-up: elements of out
  int logB;
  int64_t nfill;            // fill blocks
  int64_t nitems;           // fix-up items (kFixItem elements)
  int debug_fail;           // test hook: fail once the walk is half-way
};

// A fix-up sub-chunk of one warp: elements [i0, i0 + kFixSub) of out, a lane
// taking 2 runs of 8 (coalesced across the warp), with the carries they
// need: a run of 8 lies in one block for B >= 8 (NC = 1), in up to 4 for
// B = 2, 4 (NC = 4; carry q of a run is that of block (i0 >> logB) + q).
template <class T, int NC>
struct FixRegs {
  T v[kFixPer / 8][8];
  T c[kFixPer / 8][NC];
};

// The sub-chunk's elements (independent of the chain: may be loaded before
// the carries are ready).
template <class T, int NC>
__device__ __forceinline__ void fix_load_values(const T* out, int64_t i0s, int64_t n, int logB,
                                                int lane, FixRegs<T, NC>& r) {
  const int64_t Bk = int64_t(1) << logB;
#pragma unroll
  for (int g = 0; g < kFixPer / 8; ++g) {
    const int64_t i0 = i0s + (int64_t)g * 32 * 8 + (int64_t)lane * 8;
    const int64_t cnt = n - i0 < 0 ? 0 : (n - i0 < 8 ? n - i0 : 8);
    if (i0 + 8 > Bk) load_run(out + i0, cnt, r.v[g]);  // not all in block 0
  }
}

// Its carries (only once the tiles holding them are flagged).
template <class T, int NC>
__device__ __forceinline__ void fix_load_carries(const T* carries, int64_t i0s, int64_t n,
                                                 int logB, int lane, FixRegs<T, NC>& r) {
  const int64_t Bk = int64_t(1) << logB;
#pragma unroll
  for (int g = 0; g < kFixPer / 8; ++g) {
    const int64_t i0 = i0s + (int64_t)g * 32 * 8 + (int64_t)lane * 8;
    if (i0 >= n || i0 + 8 <= Bk) continue;
    const int64_t k0 = i0 >> logB, k1 = ((i0 + 8 < n ? i0 + 8 : n) - 1) >> logB;
#pragma unroll
    for (int q = 0; q < NC; ++q)
      if (k0 + q >= 1 && k0 + q <= k1) r.c[g][q] = __ldcg(carries + k0 + q - 1);
  }
}

template <class T, int NC>
__device__ __forceinline__ void fix_apply(T* out, int64_t i0s, int64_t n, int logB, int lane,
                                          FixRegs<T, NC>& r) {
  const int64_t Bk = int64_t(1) << logB;
#pragma unroll
  for (int g = 0; g < kFixPer / 8; ++g) {
    const int64_t i0 = i0s + (int64_t)g * 32 * 8 + (int64_t)lane * 8;
    if (i0 >= n || i0 + 8 <= Bk) continue;
    const int64_t cnt = n - i0 < 8 ? n - i0 : 8;
    if (NC == 1) {
#pragma unroll
      for (int e = 0; e < 8; ++e) r.v[g][e] = add_rn(r.c[g][0], r.v[g][e]);
      store_run(out + i0, cnt, r.v[g]);
    } else {
      const int64_t k0 = i0 >> logB;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int64_t i = i0 + e;
        const int q = (int)((i >> logB) - k0);
        T c = r.c[g][0];
#pragma unroll
        for (int u = 1; u < NC; ++u)
          if (q == u) c = r.c[g][u];
        if (e < cnt && i >= Bk) out[i] = add_rn(c, r.v[g][e]);
      }
    }
  }
}

// Fix-up items (kFixItem elements each) of one warp, taken in order from the
// shared counter until none is left: the fix-up warps from the start, the
// fill blocks' warps once their fills are done.
template <class T, int NC>
__device__ __forceinline__ void fix_items(T* out, const T* carries, const FusedArgs& f) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  for (;;) {
    unsigned long long jj = 0;
    if (lane == 0) jj = atomicAdd(f.next_item, 1ull);
    const int64_t j = (int64_t)__shfl_sync(full, jj, 0);
    if (j >= f.nitems) break;
    const int64_t lo = j * kFixItem;
    const int64_t end = lo + kFixItem < f.n ? lo + kFixItem : f.n;
    FixRegs<T, NC> a, b;
    fix_load_values<T, NC>(out, lo, end, f.logB, lane, a);  // ahead of the wait
    int go = 0;
    if (lane == 0) {
      // carries (lo >> logB) - 1 .. ((end - 1) >> logB) - 1 of its elements
      const int64_t klo = (lo >> f.logB) - 1, khi = ((end - 1) >> f.logB) - 1;
      go = khi >= 0;
      if (go) go = wait_at_least(f.tile_done + khi / kCTile, 1ull, f.fail);
      if (go && klo >= 0 && klo / kCTile != khi / kCTile)
        go = wait_at_least(f.tile_done + klo / kCTile, 1ull, f.fail);
    }
    go = __shfl_sync(full, go, 0);
    if (!go) continue;
    fix_load_carries<T, NC>(carries, lo, end, f.logB, lane, a);
#pragma unroll 1
    for (int s = 0; s < kFixSubs; ++s) {
      const int64_t i0 = lo + s * kFixSub;
      if (i0 >= end) break;
      const int64_t i1 = i0 + kFixSub;
      if (s + 1 < kFixSubs && i1 < end) {  // the next sub-chunk in flight meanwhile
        fix_load_values<T, NC>(out, i1, end, f.logB, lane, b);
        fix_load_carries<T, NC>(carries, i1, end, f.logB, lane, b);
      }
      fix_apply<T, NC>(out, i0, end, f.logB, lane, a);
      a = b;
    }
  }
}

// 2 blocks per SM (128 registers): an earlier, ticket-driven form of this
// pass took 2.4 ms at B = 16 with 2 blocks per SM and 4.1 ms with 1.
template <class T>
__global__ void __launch_bounds__(kCT, 2)
    chain_walk_fix_kernel(const T* src, T* dst, T* out, FusedArgs f) {
  if (blockIdx.x == 0) {
    if (threadIdx.x < 32) {
      walk_body<T>(src, dst, f.segs, f.total, f.seg_cap, f.m_in, f.fail, f.meta, f.K, nullptr,
                   f.progress);
    } else if (threadIdx.x == 32 && f.debug_fail) {
      const unsigned long long half = (unsigned long long)(*f.total / 2);
      if (wait_at_least(f.progress, half, f.fail)) atomicCAS(f.fail, 0, 1);
    }
    return;
  }
  const int t = threadIdx.x;
  if ((int64_t)blockIdx.x <= f.nfill) {  // a fill block
    __shared__ int s_go;
    for (int64_t c = blockIdx.x - 1; c < f.ntiles; c += f.nfill) {
      FillPrep prep;  // in flight during the wait
      fill_prep(c, t, f.qv, f.meta, f.K, f.seg_base, f.thr_in, f.entry, f.entry_rec, prep);
      if (t == 0)
        s_go = wait_at_least(f.progress, (unsigned long long)(f.seg_base[c] + f.tile_nseg[c]),
                             f.fail);
      __syncthreads();
      const int go = s_go;
      if (go) fill_finish<T>(c, t, prep, f.seg_cap, f.m_in, dst, f.fail);
      __threadfence();  // the tile's carries before its flag
      __syncthreads();  // (also: s_go read by every thread)
      if (t == 0) atomicExch(f.tile_done + c, 1u);
      if (go) {  // the check of the tile's rises, off the fix-up's path
        const int64_t r0 = f.seg_base[c], r1 = r0 + f.tile_nseg[c];
        for (int64_t r = r0 + t; r < r1 && r < f.seg_cap; r += kCT)
          verify_record<T>(f.segs, f.m_in, r, f.fail);
      }
    }
    // fills done: the block's warps join the fix-up
  }
  if (f.logB >= 3) fix_items<T, 1>(out, dst, f);
  else fix_items<T, 4>(out, dst, f);
}

// The fix-up again after a failure (grid-stride; nothing to do otherwise).
template <class T>
__global__ void __launch_bounds__(256) fixup_again_kernel(T* out, const T* carries, int64_t n,
                                                          int logB, const int* only_if) {
  if (*only_if == 0) return;
  const int64_t Bk = int64_t(1) << logB;
  for (int64_t i = Bk + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    out[i] = add_rn(carries[(i >> logB) - 1], out[i]);
}

size_t r256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

ChainPlan plan_chain(int64_t K, size_t esize) {
  const bool f32 = esize == 4;  // the binary32 classification's arrays
  ChainPlan p;
  p.K = K;
  p.ntiles = (K + kCTile - 1) / kCTile;
  p.seg_cap = K / 16 + p.ntiles + 64;  // denser breaks: the serial chain is as fast
  size_t off = 0;
  p.tsum_off = off; off += r256(p.ntiles * sizeof(double));
  p.toff_off = off; off += r256(p.ntiles * sizeof(double));
  p.tmax_off = off; off += r256(p.ntiles * sizeof(double));
  p.thr_off = off; off += r256(p.ntiles * kCT * sizeof(Summ));
  p.lead_off = off; off += r256(p.ntiles * sizeof(Map));
  p.leadsteps_off = off; off += r256(p.ntiles * sizeof(int));
  p.done_off = off; off += r256(p.ntiles * sizeof(unsigned));  // right after: one memset
  p.entry_off = off; off += r256(p.ntiles * sizeof(Map));
  p.entryrec_off = off; off += r256(p.ntiles * sizeof(int64_t));
  p.q_off = off; off += r256(K * sizeof(int64_t));
  p.meta_off = off; off += r256(K * sizeof(uint32_t));
  p.nseg_off = off; off += r256(p.ntiles * sizeof(int64_t));
  p.segbase_off = off; off += r256(p.ntiles * sizeof(int64_t));
  p.segs_off = off; off += r256(p.seg_cap * sizeof(SegRec));
  p.min_off = off; off += r256(p.seg_cap * sizeof(int64_t));
  // binary32: fixed-point tile sums of T and of the estimated errors (16
  // bytes each), their offsets, and the errors' variances
  const int64_t nf = f32 ? p.ntiles : 0, nt = f32 ? p.ntiles * kCT : 0;
  p.tfix_off = off; off += r256(nf * 16);
  p.tfoff_off = off; off += r256(nf * 16);
  p.rsum_off = off; off += r256(nf * 16);
  p.roff_off = off; off += r256(nf * 16);
  p.vsum_off = off; off += r256(nf * sizeof(double));
  p.voff_off = off; off += r256(nf * sizeof(double));
  // binary32: each thread's starting prefix, errors and variance (binary64:
  // the prefix alone, in the variance's slots)
  p.thrs_off = off; off += r256(nt * 16);
  p.thrr_off = off; off += r256(nt * 16);
  p.thrv_off = off; off += r256(p.ntiles * kCT * sizeof(double));
  // bound (8), total segments (8), fail (4), progress (8), binary32 max|T| (4)
  p.misc_off = off; off += 256;
  p.bytes = off;
  return p;
}

namespace {

// The chain's workspace, carved by the plan's offsets.
struct ChainWs {
  double *tsum, *toff, *tmax, *bound, *vsum, *voff;
  i128 *tfix, *tfoff, *rsum, *roff, *thr_s, *thr_r;
  double* thr_v;
  unsigned* maxbits;
  Summ* thr_in;
  Map *lead, *entry;
  int* lead_steps;
  unsigned* done;
  int64_t *entry_rec, *qv, *nseg, *segbase, *m_in, *total;
  uint32_t* meta;
  SegRec* segs;
  int* fail;
  unsigned long long* progress;
  unsigned long long* next_item;
  ChainWs(const ChainPlan& p, char* ws) {
    tsum = reinterpret_cast<double*>(ws + p.tsum_off);
    toff = reinterpret_cast<double*>(ws + p.toff_off);
    tmax = reinterpret_cast<double*>(ws + p.tmax_off);
    thr_in = reinterpret_cast<Summ*>(ws + p.thr_off);
    lead = reinterpret_cast<Map*>(ws + p.lead_off);
    lead_steps = reinterpret_cast<int*>(ws + p.leadsteps_off);
    done = reinterpret_cast<unsigned*>(ws + p.done_off);
    entry = reinterpret_cast<Map*>(ws + p.entry_off);
    entry_rec = reinterpret_cast<int64_t*>(ws + p.entryrec_off);
    qv = reinterpret_cast<int64_t*>(ws + p.q_off);
    meta = reinterpret_cast<uint32_t*>(ws + p.meta_off);
    nseg = reinterpret_cast<int64_t*>(ws + p.nseg_off);
    segbase = reinterpret_cast<int64_t*>(ws + p.segbase_off);
    segs = reinterpret_cast<SegRec*>(ws + p.segs_off);
    m_in = reinterpret_cast<int64_t*>(ws + p.min_off);
    tfix = reinterpret_cast<i128*>(ws + p.tfix_off);
    tfoff = reinterpret_cast<i128*>(ws + p.tfoff_off);
    rsum = reinterpret_cast<i128*>(ws + p.rsum_off);
    roff = reinterpret_cast<i128*>(ws + p.roff_off);
    vsum = reinterpret_cast<double*>(ws + p.vsum_off);
    voff = reinterpret_cast<double*>(ws + p.voff_off);
    maxbits = reinterpret_cast<unsigned*>(ws + p.misc_off + 32);
    thr_s = reinterpret_cast<i128*>(ws + p.thrs_off);
    thr_r = reinterpret_cast<i128*>(ws + p.thrr_off);
    thr_v = reinterpret_cast<double*>(ws + p.thrv_off);
    bound = reinterpret_cast<double*>(ws + p.misc_off);
    total = reinterpret_cast<int64_t*>(ws + p.misc_off + 8);
    fail = reinterpret_cast<int*>(ws + p.misc_off + 16);
    progress = reinterpret_cast<unsigned long long*>(ws + p.misc_off + 24);
    next_item = reinterpret_cast<unsigned long long*>(ws + p.misc_off + 40);
  }
};

// Passes 1 to 6: tile sums, offsets and bound, classification, record
// numbering, segments, links.
template <class T>
cudaError_t run_chain_front(const ChainPlan& p, const T* src, char* ws, const ChainWs& w,
                            cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(ws + p.misc_off, 0, 256, s);
  if (e != cudaSuccess) return e;
  // the lead step counts and the fused form's tile flags (adjacent)
  e = cudaMemsetAsync(w.lead_steps, 0, p.done_off + r256(p.ntiles * sizeof(unsigned)) -
                                           p.leadsteps_off, s);
  if (e != cudaSuccess) return e;
  if (p.ntiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned g = (unsigned)p.ntiles;
  if constexpr (sizeof(T) == 4) {  // binary32: classify against the estimated chain
    const int64_t ab = p.ntiles * 16 < 1216 ? p.ntiles * 16 : 1216;
    CR_LAUNCH(kKChainTileSum, s,
              chain_absmax_kernel<<<(unsigned)ab, 256, 0, s>>>(src, p.K, w.maxbits));
    CR_LAUNCH(kKChainTileSum, s,
              chain_fixsum_kernel<<<g, kCT, 0, s>>>(src, p.K, w.maxbits, w.tfix));
    CR_LAUNCH(kKChainOffsets, s,
              exclusive_scan128_1block<<<1, 1024, 0, s>>>(w.tfix, w.tfoff, p.ntiles));
    CR_LAUNCH(kKChainRoundSum, s,
              chain_round_sum_kernel<<<g, kCT, 0, s>>>(src, p.K, w.maxbits, w.tfoff, w.rsum,
                                                       w.vsum, w.thr_s, w.thr_r, w.thr_v));
    CR_LAUNCH(kKChainOffsets, s,
              exclusive_scan128_1block<<<1, 1024, 0, s>>>(w.rsum, w.roff, p.ntiles));
    CR_LAUNCH(kKChainOffsets, s,
              exclusive_scan_1block<double><<<1, 1024, 0, s>>>(w.vsum, w.voff, p.ntiles,
                                                               nullptr));
    CR_LAUNCH(kKChainClassify, s,
              chain_classify_f32_kernel<<<g, kCT, 0, s>>>(src, p.K, w.maxbits, w.thr_s,
                                                          w.thr_r, w.thr_v, w.roff, w.voff,
                                                          w.qv, w.meta, w.nseg, w.thr_in));
  } else {
    CR_LAUNCH(kKChainTileSum, s,
              chain_tile_sum_kernel<T><<<g, kCT, 0, s>>>(src, p.K, w.tsum, w.tmax, w.thr_v));
    CR_LAUNCH(kKChainOffsets, s,
              chain_offsets_kernel<<<1, 1024, 0, s>>>(w.tsum, w.tmax, p.ntiles, w.toff,
                                                      w.bound));
    CR_LAUNCH(kKChainClassify, s,
              chain_classify_kernel<T><<<g, kCT, 0, s>>>(src, p.K, w.toff, w.thr_v, w.bound,
                                                         w.qv, w.meta, w.nseg, w.thr_in));
  }
  CR_LAUNCH(kKChainOffsets, s,
            exclusive_scan_1block<int64_t><<<1, 1024, 0, s>>>(w.nseg, w.segbase, p.ntiles,
                                                              w.total));
  CR_LAUNCH(kKChainSegments, s,
            chain_segments_kernel<T><<<g, kCT, 0, s>>>(src, w.qv, w.meta, p.K, w.segbase,
                                                       w.nseg, w.thr_in, w.segs, p.seg_cap,
                                                       w.lead, w.lead_steps, w.fail));
  CR_LAUNCH(kKChainLink, s,
            chain_link_kernel<<<1, 1024, 0, s>>>(w.nseg, w.segbase, p.ntiles, w.segs, p.seg_cap,
                                                 w.lead, w.lead_steps, w.entry, w.entry_rec));
  return cudaGetLastError();
}

// Co-resident blocks of the fused kernel on this device (cached per device;
// threads that race to fill an entry store the same value).
template <class T>
int fused_grid_limit() {
  static std::atomic<int> cache[64];  // static storage: starts at zero
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int limit = cache[dev].load(std::memory_order_relaxed);
  if (limit == 0) {
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_walk_fix_kernel<T>, kCT,
                                                      0) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    limit = per_sm * sms;
    cache[dev].store(limit, std::memory_order_relaxed);
  }
  return limit;
}

}  // namespace

namespace {

// Passes 7 to 9 as separate launches: the walk, the check of its rises, the
// fill, and the serial chain that runs only when any of them failed.
template <class T>
cudaError_t run_chain_back(const ChainPlan& p, const T* src, T* dst, const ChainWs& w,
                           cudaStream_t s, T* final_out) {
  const unsigned g = (unsigned)p.ntiles;
  CR_LAUNCH(kKChainWalk, s,
            chain_walk_kernel<T><<<1, 32, 0, s>>>(src, dst, w.segs, w.total, p.seg_cap, w.m_in,
                                                  w.fail, w.meta, p.K, final_out));
  if ((p.seg_cap + 255) / 256 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  CR_LAUNCH(kKChainVerify, s,
            chain_verify_kernel<T><<<(unsigned)((p.seg_cap + 255) / 256), 256, 0, s>>>(
                w.segs, w.total, p.seg_cap, w.m_in, w.fail));
  CR_LAUNCH(kKChainFill, s,
            chain_fill_kernel<T><<<g, kCT, 0, s>>>(w.qv, w.meta, p.K, w.segbase, w.thr_in,
                                                   w.entry, w.entry_rec, p.seg_cap, w.m_in, dst,
                                                   w.fail));
  CR_LAUNCH(kKChainFallback, s,
            chain_serial_kernel<T><<<1, 32, 0, s>>>(src, dst, p.K, w.fail, final_out));
  return cudaGetLastError();
}

}  // namespace

template <class T>
cudaError_t run_chain(const ChainPlan& p, const T* src, T* dst, char* ws, cudaStream_t s,
                      T* final_out) {
  if (p.K <= 0) return cudaSuccess;
  const ChainWs w(p, ws);
  cudaError_t e = run_chain_front<T>(p, src, ws, w, s);
  if (e != cudaSuccess) return e;
  return run_chain_back<T>(p, src, dst, w, s, final_out);
}

template <class T>
cudaError_t run_chain_fixup(const ChainPlan& p, const T* src, T* dst, char* ws, T* out,
                            int64_t n, int logB, cudaStream_t s, const int** fail,
                            bool* fused, bool debug_fail, bool debug_refuse) {
  const ChainWs w(p, ws);
  *fail = w.fail;
  *fused = false;
  if (p.K <= 0 || p.K > (out != nullptr ? kMaxFusedChain : kMaxFusedChainAlone) ||
      (out != nullptr && (logB < 1 || logB > 40)))
    return cudaErrorInvalidValue;
  cudaError_t e = run_chain_front<T>(p, src, ws, w, s);
  if (e != cudaSuccess) return e;
  FusedArgs f{};
  f.segs = w.segs;
  f.total = w.total;
  f.seg_cap = p.seg_cap;
  f.m_in = w.m_in;
  f.fail = w.fail;
  f.meta = w.meta;
  f.qv = w.qv;
  f.K = p.K;
  f.ntiles = p.ntiles;
  f.seg_base = w.segbase;
  f.tile_nseg = w.nseg;
  f.thr_in = w.thr_in;
  f.entry = w.entry;
  f.entry_rec = w.entry_rec;
  f.progress = w.progress;
  f.next_item = w.next_item;
  f.tile_done = w.done;
  f.n = n;
  f.logB = logB;
  f.debug_fail = debug_fail ? 1 : 0;
  f.nitems = out != nullptr ? (n + kFixItem - 1) / kFixItem : 0;
  const int limit = fused_grid_limit<T>();
  // fill blocks: enough for the fills to keep pace with the walk, and at
  // least three quarters of the grid left for the fix-up
  f.nfill = p.ntiles < kMaxFillBlocks ? p.ntiles : kMaxFillBlocks;
  if (f.nfill > limit / kFillShareDiv) f.nfill = limit / kFillShareDiv;
  if (out == nullptr) f.nfill = p.ntiles < limit - 1 ? p.ntiles : limit - 1;  // all fill
  if (f.nfill >= 1 && !debug_refuse) {
    const int64_t fixers = (f.nitems + kCT / 32 - 1) / (kCT / 32);  // 8 warps a block
    const int64_t room = limit - 1 - f.nfill;
    const unsigned grid = (unsigned)(1 + f.nfill + (fixers < room ? fixers : room));
    void* args[] = {(void*)&src, (void*)&dst, (void*)&out, (void*)&f};
    CR_LAUNCH(kKChainWalkFix, s,
              e = cudaLaunchCooperativeKernel((const void*)chain_walk_fix_kernel<T>, dim3(grid),
                                              dim3(kCT), args, 0, s));
    if (e == cudaSuccess) {
      *fused = true;
      CR_LAUNCH(kKChainFallback, s,
                chain_serial_kernel<T><<<1, 32, 0, s>>>(src, dst, p.K, w.fail, nullptr));
      return cudaGetLastError();
    }
    // The cooperative launch was refused (fewer resident blocks than the
    // occupancy query promised: another context on the device, a smaller SM
    // partition). A refused launch enqueues nothing and its error is not
    // sticky: clear it and take the separate passes, whose result is the same.
    (void)cudaGetLastError();
  }
  return run_chain_back<T>(p, src, dst, w, s, nullptr);
}

template <class T>
cudaError_t run_fixup_again(T* out, const T* carries, int64_t n, int logB, const int* fail,
                            cudaStream_t s) {
  CR_LAUNCH(kKFixupAgain, s,
            fixup_again_kernel<T><<<1216, 256, 0, s>>>(out, carries, n, logB, fail));
  return cudaGetLastError();
}

template <class T>
cudaError_t run_serial_chain(const T* src, T* dst, int64_t K, cudaStream_t s, T* final_out) {
  if (K <= 0) return cudaSuccess;
  CR_LAUNCH(kKCarryChain, s,
            chain_serial_kernel<T><<<1, 32, 0, s>>>(src, dst, K, nullptr, final_out));
  return cudaGetLastError();
}

template cudaError_t run_serial_chain<double>(const double*, double*, int64_t, cudaStream_t,
                                              double*);
template cudaError_t run_serial_chain<float>(const float*, float*, int64_t, cudaStream_t,
                                             float*);
template cudaError_t run_chain<double>(const ChainPlan&, const double*, double*, char*,
                                       cudaStream_t, double*);
template cudaError_t run_chain_fixup<double>(const ChainPlan&, const double*, double*, char*,
                                             double*, int64_t, int, cudaStream_t, const int**,
                                             bool*, bool, bool);
template cudaError_t run_chain_fixup<float>(const ChainPlan&, const float*, float*, char*,
                                            float*, int64_t, int, cudaStream_t, const int**,
                                            bool*, bool, bool);
template cudaError_t run_fixup_again<double>(double*, const double*, int64_t, int, const int*,
                                             cudaStream_t);
template cudaError_t run_fixup_again<float>(float*, const float*, int64_t, int, const int*,
                                            cudaStream_t);
template cudaError_t run_chain<float>(const ChainPlan&, const float*, float*, char*,
                                      cudaStream_t, float*);

}  // namespace cr
