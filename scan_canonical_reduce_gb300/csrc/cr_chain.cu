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
//
// Passes (tile = 4096 steps, 16 per thread):
//   1 tile sums, 2 tile offsets (one block), 3 prefix P~_k and max|P~|;
//   4 classify: the binade and sign of s_k from P~_k, certain when the whole
//     interval P~_k +- mu (mu = K ulp(2 max|P~|) bounds both |C_k - P_k| and
//     |P~_k - P_k|) lies inside one binade; step types MAP (same or lower
//     binade), UP (higher binade, integer break), FP (uncertain: real add);
//   5 segment bases (one block), 6 segment records: each break (or tile
//     start) and the composed map of the MAP steps that follow it;
//   7 walk: the breaks in order, from integers; M entering every segment;
//   8 fill: every MAP step recomputed from its segment's entry value with an
//     exact 128-bit test that s_k lies in the predicted binade and sign;
//   9 if any test failed (or the segment buffer overflowed), the serial chain
//     recomputes everything on the device (no host sync).
// Every add of the chain is therefore the real add or proven equal to it.
#include <cstdint>

#include "cr_chain.h"
#include "cr_device.cuh"
#include "cr_launch.h"

namespace cr {
namespace {

constexpr int kCT = 256;           // threads per tile
constexpr int kCE = 16;            // steps per thread
constexpr int kCTile = kCT * kCE;  // 4096 steps per tile

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

// ---- integer maps M -> a M + b[parity(M)] (mod 2^64)
struct Map {
  uint64_t a, b0, b1;
};
__device__ __forceinline__ Map map_id() { return Map{1, 0, 0}; }
__device__ __forceinline__ uint64_t bsel(const Map& g, uint64_t p) { return p ? g.b1 : g.b0; }
__device__ __forceinline__ Map compose(const Map& g, const Map& h) {  // first g, then h
  const uint64_t p0 = (g.b0 & 1);                         // parity after g, from even M
  const uint64_t p1 = ((g.a & 1) ^ g.b1) & 1;            // parity after g, from odd M
  return Map{h.a * g.a, h.a * g.b0 + bsel(h, p0), h.a * g.b1 + bsel(h, p1)};
}
__device__ __forceinline__ uint64_t apply(const Map& g, uint64_t M) {
  return g.a * M + bsel(g, M & 1);
}
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
  const int64_t A = (int64_t)M + q;  // |M| <= 2^54, |q| < 2^62
  const int64_t hi = A >> d;         // floor
  const uint64_t lo = (uint64_t)A & ((uint64_t(1) << d) - 1);
  const uint64_t half = uint64_t(1) << (d - 1);
  const bool fpos = fcls != kFZero;
  const bool rup = lo > half || (lo == half && (fpos || (hi & 1)));
  ok = ok && in_binade64<T>(hi, neg, lo == 0 && !fpos);
  return (uint64_t)(hi + (rup ? 1 : 0));
}

// ---------------------------------------------------------------- pass 1
template <class T>
__global__ void __launch_bounds__(kCT) chain_tile_sum_kernel(const T* src, int64_t K,
                                                             double* tsum) {
  __shared__ double sh[kCT];
  const int t = threadIdx.x;
  const int64_t k0 = (int64_t)blockIdx.x * kCTile + (int64_t)t * kCE;
  double s = 0.0;
#pragma unroll
  for (int i = 0; i < kCE; ++i)
    if (k0 + i < K) s += (double)src[k0 + i];
  sh[t] = s;
  __syncthreads();
  for (int w = kCT / 2; w > 0; w >>= 1) {
    if (t < w) sh[t] += sh[t + w];
    __syncthreads();
  }
  if (t == 0) tsum[blockIdx.x] = sh[0];
}

// ---------------------------------------------------------------- pass 2 / 5
template <class V>
__global__ void __launch_bounds__(1024) exclusive_scan_1block(const V* in, V* out, int64_t n,
                                                              V* total) {
  __shared__ V sh[1024];
  __shared__ V carry;
  const int t = threadIdx.x;
  if (t == 0) carry = V(0);
  __syncthreads();
  for (int64_t base = 0; base < n; base += 1024) {
    const int64_t i = base + t;
    const V v = i < n ? in[i] : V(0);
    sh[t] = v;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const V a = t >= off ? sh[t - off] : V(0);
      __syncthreads();
      sh[t] += a;
      __syncthreads();
    }
    if (i < n) out[i] = carry + sh[t] - v;
    __syncthreads();
    if (t == 0) carry += sh[1023];
    __syncthreads();
  }
  if (t == 0 && total) *total = carry;
}

// ---------------------------------------------------------------- pass 3
template <class T>
__global__ void __launch_bounds__(kCT) chain_prefix_kernel(const T* src, int64_t K,
                                                           const double* toff, double* pre,
                                                           unsigned long long* maxabs) {
  __shared__ double sh[kCT];
  const int t = threadIdx.x;
  const int64_t k0 = (int64_t)blockIdx.x * kCTile + (int64_t)t * kCE;
  double v[kCE];
  double s = 0.0;
#pragma unroll
  for (int i = 0; i < kCE; ++i) {
    v[i] = (k0 + i < K) ? (double)src[k0 + i] : 0.0;
    s += v[i];
  }
  sh[t] = s;
  __syncthreads();
  for (int off = 1; off < kCT; off <<= 1) {  // inclusive scan of thread sums
    const double a = t >= off ? sh[t - off] : 0.0;
    __syncthreads();
    sh[t] += a;
    __syncthreads();
  }
  double run = toff[blockIdx.x] + (sh[t] - s);
  double mx = 0.0;
#pragma unroll
  for (int i = 0; i < kCE; ++i) {
    if (k0 + i < K) {
      run += v[i];
      pre[k0 + i] = run;
      mx = fmax(mx, fabs(run));
    }
  }
  if (!(mx <= 1.7e308)) mx = 1.7e308;  // non-finite: those steps are uncertain anyway
  __syncthreads();
  sh[t] = mx;
  __syncthreads();
  for (int w = kCT / 2; w > 0; w >>= 1) {
    if (t < w) sh[t] = fmax(sh[t], sh[t + w]);
    __syncthreads();
  }
  if (t == 0) atomicMax(maxabs, (unsigned long long)__double_as_longlong(sh[0]));
}

// ---------------------------------------------------------------- pass 4
// Binade exponent of a positive finite double from its bits.
__device__ __forceinline__ int dexp(double a) {
  return (int)((FP<double>::bits(a) >> 52) & 0x7FF) - 1023;
}
__device__ __forceinline__ double dpow2(int e) {  // 2^e, normal range
  return FP<double>::from_bits((uint64_t)(e + 1023) << 52);
}

template <class T>
__device__ __forceinline__ void classify(double p, double mu, bool& certain, bool& neg, int& e) {
  certain = false;
  neg = p < 0;
  e = 0;
  const double a = fabs(p);
  if (!(a <= 1e300)) return;  // non-finite
  if (a <= mu || a < 1e-290) return;  // sign, zero or the subnormal range uncertain
  const int ee = dexp(a);
  if (ee < FP<T>::EMIN + 2 || ee > FP<T>::EMAX - 2) return;
  const double lo = dpow2(ee), hi = dpow2(ee + 1), ulp = dpow2(ee - FP<T>::P);
  if (a - mu < lo || a + mu + ulp >= hi) return;  // interval crosses a binade edge
  certain = true;
  e = ee;
}

template <class T>
__global__ void __launch_bounds__(kCT) chain_classify_kernel(
    const T* src, int64_t K, const double* pre, const unsigned long long* maxabs, int64_t* qv,
    uint32_t* meta, int64_t* tile_nseg) {
  __shared__ int cnt[kCT];
  const int t = threadIdx.x;
  const int64_t k0 = (int64_t)blockIdx.x * kCTile + (int64_t)t * kCE;
  double mu;
  {
    const double m2 = 2.0 * __longlong_as_double((long long)*maxabs);
    mu = m2 > 1e-290 && m2 < 1e300 ? (double)K * dpow2(dexp(m2) - FP<T>::P) : 1e300;
    if (m2 <= 1e-290) mu = 1e-280;
  }
  int nbrk = 0;
  bool pc = false, pn = false;
  int pe = 0;
  if (k0 > 0 && k0 < K) classify<T>(pre[k0 - 1], mu, pc, pn, pe);
  for (int i = 0; i < kCE; ++i) {
    const int64_t k = k0 + i;
    if (k >= K) break;
    bool c, n;
    int e;
    classify<T>(pre[k], mu, c, n, e);
    uint32_t type;
    int d = 0;
    int64_t q = 0;
    uint32_t f = 0;
    const T tv = src[k];
    if (k == 0) {
      type = kStart;
    } else if (!c || !pc) {
      type = kFp;
    } else if (e <= pe) {  // same or lower binade: a composable step
      d = pe - e;
      type = (d <= 63 && split_unit<T>(tv, e, q, f)) ? kMap : kFp;
    } else {  // rise: integer break, T split in the old (finer) unit
      d = e - pe;
      type = (d <= 8 && split_unit<T>(tv, pe, q, f)) ? kUp : kFp;
    }
    if (type == kFp) d = 0;
    meta[k] = make_meta(type, c, n, f, d, e);
    qv[k] = q;
    nbrk += type != kMap ? 1 : 0;
    pc = c; pn = n; pe = e;
  }
  cnt[t] = nbrk;
  __syncthreads();
  for (int w = kCT / 2; w > 0; w >>= 1) {
    if (t < w) cnt[t] += cnt[t + w];
    __syncthreads();
  }
  if (t == 0) {  // one segment per break, plus one if the tile starts inside a run
    const int64_t first = (int64_t)blockIdx.x * kCTile;
    tile_nseg[blockIdx.x] = cnt[0] + (m_type(meta[first]) == kMap ? 1 : 0);
  }
}

// ---------------------------------------------------------------- pass 6
struct Summ {  // composition after the last break of a thread's steps
  Map map;
  int brk;
};
__device__ __forceinline__ Summ combine(const Summ& l, const Summ& r) {
  return r.brk ? Summ{r.map, l.brk + r.brk} : Summ{compose(l.map, r.map), l.brk};
}

// Segment record: a break (or a tile start inside a run) and the composed
// map of the MAP steps after it, up to the next break or the tile end.
struct SegRec {
  int64_t start;
  Map map;
  int64_t q;        // up: T split in the old unit
  double tval;      // start or fp break: T at the start step (exact in double)
  uint32_t meta;    // meta word of the start step (type kMap marks a continuation)
  int32_t e_prev;   // fp break: binade of the previous step (if certain)
  int32_t prev_certain;
  int32_t nsteps;   // MAP steps in the map
};

__device__ __forceinline__ void thread_scan(const int64_t* qv, const uint32_t* meta,
                                            int64_t k0, int64_t K, Summ& in_excl, Summ* sh) {
  Summ me{map_id(), 0};
  for (int i = 0; i < kCE; ++i) {
    const int64_t k = k0 + i;
    if (k >= K) break;
    const uint32_t m = meta[k];
    if (m_type(m) != kMap) {
      me.map = map_id();
      me.brk += 1;
    } else {
      me.map = compose(me.map, step_map(m_d(m), qv[k], m_fcls(m)));
    }
  }
  const int t = threadIdx.x;
  sh[t] = me;
  __syncthreads();
  for (int off = 1; off < kCT; off <<= 1) {  // inclusive segmented scan
    Summ a = sh[t];
    if (t >= off) a = combine(sh[t - off], a);
    __syncthreads();
    sh[t] = a;
    __syncthreads();
  }
  in_excl = t > 0 ? sh[t - 1] : Summ{map_id(), 0};
  __syncthreads();
}

template <class T>
__global__ void __launch_bounds__(kCT) chain_segments_kernel(
    const T* src, const int64_t* qv, const uint32_t* meta, int64_t K, const int64_t* seg_base,
    SegRec* segs, int64_t seg_cap, int* fail) {
  __shared__ Summ sh[kCT];
  const int t = threadIdx.x;
  const int64_t tile0 = (int64_t)blockIdx.x * kCTile;
  const int64_t k0 = tile0 + (int64_t)t * kCE;
  Summ in;
  thread_scan(qv, meta, k0, K, in, sh);
  const bool cont = m_type(meta[tile0]) == kMap;
  int64_t ord = (cont ? 1 : 0) + in.brk - 1;  // segment open at my first step
  Map cur = in.map;
  int steps = 0;  // MAP steps of the open segment seen by this thread
  const int64_t base = seg_base[blockIdx.x];
  if (t == 0 && cont) {
    if (base < seg_cap) {
      SegRec& r = segs[base];
      r.start = tile0;
      r.meta = meta[tile0];
      r.q = 0;
      r.e_prev = 0;
      r.prev_certain = 0;
    } else {
      atomicExch(fail, 2);
    }
  }
  for (int i = 0; i < kCE; ++i) {
    const int64_t k = k0 + i;
    if (k >= K) break;
    const uint32_t m = meta[k];
    if (m_type(m) != kMap) {
      if (ord >= 0 && base + ord < seg_cap) {  // close the open segment
        segs[base + ord].map = cur;
        if (steps) atomicAdd(&segs[base + ord].nsteps, steps);
      }
      ord += 1;
      cur = map_id();
      steps = 0;
      if (base + ord < seg_cap) {
        SegRec& r = segs[base + ord];
        r.start = k;
        r.meta = m;
        r.q = qv[k];
        r.tval = (double)src[k];
        const uint32_t pm = meta[k > 0 ? k - 1 : 0];
        r.e_prev = m_e(pm);
        r.prev_certain = (k > 0 && m_certain(pm)) ? 1 : 0;
      } else {
        atomicExch(fail, 2);
      }
    } else {
      cur = compose(cur, step_map(m_d(m), qv[k], m_fcls(m)));
      steps += 1;
    }
  }
  if (ord >= 0 && base + ord < seg_cap) {
    // my trailing MAP steps belong to the segment still open; the thread
    // holding the tile's last step closes it
    if (steps) atomicAdd(&segs[base + ord].nsteps, steps);
    const int64_t last = (tile0 + kCTile < K ? tile0 + kCTile : K) - 1;
    if (k0 <= last && last < k0 + kCE) segs[base + ord].map = cur;
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
  int64_t c;        // 2^(d-1) - 1 for a rise, 0 for a continuation
  uint64_t b0, b1;  // the segment map's offsets, plus the next record's q when
                    // that record is a rise or a continuation
  uint32_t ctrl;    // d (6 bits) | sh (7) << 6 | rise << 13 | fpos << 14 | neg << 15 |
                    // type (2) << 16 | steps << 18
  uint32_t pad;
};
__device__ __forceinline__ bool is_fast(uint32_t meta) { return m_type(meta) <= kUp; }
__device__ __forceinline__ Hot make_hot(const SegRec& r, int64_t q_next) {
  Hot h;
  const uint32_t m = r.meta, type = m_type(m);
  const bool up = type == kUp;
  const int d = up ? m_d(m) : 0;
  h.c = d > 0 ? (int64_t(1) << (d - 1)) - 1 : 0;
  h.b0 = r.map.b0 + (uint64_t)q_next;
  h.b1 = r.map.b1 + (uint64_t)q_next;
  const uint32_t shift = r.map.a == 0 ? 64u : (uint32_t)(__ffsll((long long)r.map.a) - 1);
  h.ctrl = (uint32_t)d | (shift << 6) | (d > 0 ? 1u << 13 : 0u) |
           ((m_fcls(m) != kFZero) ? 1u << 14 : 0u) | (m_neg(m) ? 1u << 15 : 0u) |
           (type << 16) | (r.nsteps > 0 ? 1u << 18 : 0u);
  h.pad = 0;
  return h;
}

// One break (rise or continuation) from A: writes m_in, returns the next A.
template <class T>
__device__ __forceinline__ int64_t walk_fast(const Hot& h, int64_t A, int64_t* m_in_j,
                                             uint32_t& okw, bool& cval) {
  const uint32_t c = h.ctrl;
  const int d = (int)(c & 63u);
  const uint32_t sh = (c >> 6) & 127u;
  const uint32_t rise = (c >> 13) & 1u, fpos = (c >> 14) & 1u;
  const int64_t hi = A >> d;
  const int64_t x = (int64_t)(((uint32_t)hi & rise) | (fpos & rise));
  const int64_t M1 = (A + h.c + x) >> d;
  *m_in_j = M1;
  // in-binade test of a rise, as integer comparisons on hi (off the chain)
  constexpr int64_t LO = int64_t(1) << FP<T>::P, HI = int64_t(1) << (FP<T>::P + 1);
  const uint64_t mask = (uint64_t(1) << d) - 1;  // d = 0: 0
  const uint32_t fz = (((uint64_t)A & mask) == 0) & (fpos ^ 1u);
  const uint32_t pos_ok = (hi >= LO) & (hi <= HI - 1);
  const uint32_t neg_ok = fz ? (hi <= -LO) & (hi >= -HI + 1) : (hi <= -LO - 1) & (hi >= -HI);
  const uint32_t in_ok = ((c >> 15) & 1u) ? neg_ok : pos_ok;
  okw &= rise ? in_ok : 1u;
  cval = cval & !rise & !((c >> 18) & 1u);
  const uint64_t aM = sh >= 64 ? 0 : ((uint64_t)M1 << sh);
  return (int64_t)(aM + ((M1 & 1) ? h.b1 : h.b0));
}

// Breaks in order, in one thread. The whole warp converts the next 32
// records to compact form while lane 0 runs the current 32 from shared
// memory; batches with no start or uncertain step run an unrolled loop of
// the integer path alone.
template <class T>
__global__ void __launch_bounds__(32) chain_walk_kernel(const T* src, T* dst, const SegRec* segs,
                                                        const int64_t* nseg_total,
                                                        int64_t seg_cap, int64_t* m_in,
                                                        int* fail) {
  __shared__ Hot hot[2][32];
  __shared__ SegRec cold[2][32];
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
    cold[slot][lane] = cur;
    const bool is_cold = b0 + lane < nseg && !is_fast(cur.meta);
    const unsigned any_cold = __ballot_sync(full, is_cold);
    if (lane == 0) cold_batch[slot] = any_cold != 0;
    __syncwarp();
    cur = nxt;
    const int64_t nb = b0 + 64 + lane;
    if (nb < nseg) nxt = segs[nb];
    if (lane == 0) {
      const int cnt = (int)(nseg - b0 < 32 ? nseg - b0 : 32);
      bool ok = true;
      uint32_t okw = 1u;
      if (!cold_batch[slot]) {
        if (cnt == 32) {
#pragma unroll 8
          for (int j = 0; j < 32; ++j)
            A = walk_fast<T>(hot[slot][j], A, m_in + b0 + j, okw, cval);
        } else {
          for (int j = 0; j < cnt; ++j)
            A = walk_fast<T>(hot[slot][j], A, m_in + b0 + j, okw, cval);
        }
      } else {
        for (int j = 0; j < cnt; ++j) {
          const Hot h = hot[slot][j];
          const uint32_t type = (h.ctrl >> 16) & 3u;
          if (type <= kUp) {
            A = walk_fast<T>(h, A, m_in + b0 + j, okw, cval);
            continue;
          }
          // start or uncertain step: the real add. The previous record folded
          // no q into A for this one, so A is the entering M.
          const SegRec& r = cold[slot][j];
          const uint32_t m = r.meta;
          if (type == kStart) {
            C = (T)r.tval;
          } else {
            if (!cval) {
              ok = ok && r.prev_certain;
              C = m_to_value<T>(A, r.e_prev);
            }
            C = add_rn(C, (T)r.tval);
          }
          dst[r.start] = C;
          cval = true;
          int64_t M1 = A;
          if (m_certain(m)) {
            int64_t Mi = 0;
            ok = ok && value_to_m<T>(C, m_e(m), Mi);
            M1 = Mi;
          }
          m_in[b0 + j] = M1;
          const uint32_t sh = (h.ctrl >> 6) & 127u;
          const uint64_t aM = sh >= 64 ? 0 : ((uint64_t)M1 << sh);
          A = (int64_t)(aM + ((M1 & 1) ? h.b1 : h.b0));
          cval = cval & !((h.ctrl >> 18) & 1u);
        }
      }
      bad = bad || !ok || !okw;
    }
    __syncwarp();
  }
  if (lane == 0 && bad) atomicExch(fail, 1);
}

// ---------------------------------------------------------------- pass 8
template <class T>
__global__ void __launch_bounds__(kCT) chain_fill_kernel(const int64_t* qv, const uint32_t* meta,
                                                         int64_t K, const int64_t* seg_base,
                                                         const SegRec* segs, int64_t seg_cap,
                                                         const int64_t* m_in, T* dst, int* fail) {
  __shared__ Summ sh[kCT];
  const int t = threadIdx.x;
  const int64_t tile0 = (int64_t)blockIdx.x * kCTile;
  const int64_t k0 = tile0 + (int64_t)t * kCE;
  Summ in;
  thread_scan(qv, meta, k0, K, in, sh);
  if (*fail) return;
  const bool cont = m_type(meta[tile0]) == kMap;
  int64_t seg = seg_base[blockIdx.x] + (cont ? 1 : 0) + in.brk - 1;
  uint64_t M = 0;
  if (k0 < K && seg >= 0 && seg < seg_cap) M = apply(in.map, (uint64_t)m_in[seg]);
  bool ok = true;
  for (int i = 0; i < kCE; ++i) {
    const int64_t k = k0 + i;
    if (k >= K) break;
    const uint32_t m = meta[k];
    const uint32_t type = m_type(m);
    if (type != kMap) {  // enter the next segment
      seg += 1;
      if (seg >= seg_cap) { ok = false; break; }
      M = (uint64_t)m_in[seg];
      if (type == kUp) dst[k] = m_to_value<T>((int64_t)M, m_e(m));  // walk wrote fp breaks
      continue;
    }
    const int d = m_d(m);
    const __int128 A = (__int128)(int64_t)M * ((__int128)1 << d) + (__int128)qv[k];
    const uint32_t f = m_fcls(m);
    if (!in_binade<T>(A, m_neg(m), f)) { ok = false; break; }
    const int64_t A64 = (int64_t)A;
    M = (uint64_t)(A64 + (int64_t)delta(f, (uint64_t)A64 & 1));
    dst[k] = m_to_value<T>((int64_t)M, m_e(m));
  }
  if (!ok) atomicExch(fail, 1);
}

// ---------------------------------------------------------------- pass 9
template <class T>
__global__ void chain_fallback_kernel(const T* src, T* dst, int64_t K, const int* fail) {
  if (threadIdx.x != 0 || blockIdx.x != 0 || *fail == 0) return;
  T c = src[0];
  dst[0] = c;
  for (int64_t k = 1; k < K; ++k) {
    c = add_rn(c, src[k]);
    dst[k] = c;
  }
}

size_t r256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

ChainPlan plan_chain(int64_t K) {
  ChainPlan p;
  p.K = K;
  p.ntiles = (K + kCTile - 1) / kCTile;
  p.seg_cap = K / 16 + p.ntiles + 64;  // denser breaks: the serial chain is as fast
  size_t off = 0;
  p.tsum_off = off; off += r256(p.ntiles * sizeof(double));
  p.toff_off = off; off += r256(p.ntiles * sizeof(double));
  p.pre_off = off; off += r256(K * sizeof(double));
  p.q_off = off; off += r256(K * sizeof(int64_t));
  p.meta_off = off; off += r256(K * sizeof(uint32_t));
  p.nseg_off = off; off += r256(p.ntiles * sizeof(int64_t));
  p.segbase_off = off; off += r256(p.ntiles * sizeof(int64_t));
  p.segs_off = off; off += r256(p.seg_cap * sizeof(SegRec));
  p.min_off = off; off += r256(p.seg_cap * sizeof(int64_t));
  p.misc_off = off; off += 256;  // maxabs (8), total segments (8), fail (4)
  p.bytes = off;
  return p;
}

template <class T>
cudaError_t run_chain(const ChainPlan& p, const T* src, T* dst, char* ws, cudaStream_t s) {
  if (p.K <= 0) return cudaSuccess;
  double* tsum = reinterpret_cast<double*>(ws + p.tsum_off);
  double* toff = reinterpret_cast<double*>(ws + p.toff_off);
  double* pre = reinterpret_cast<double*>(ws + p.pre_off);
  int64_t* qv = reinterpret_cast<int64_t*>(ws + p.q_off);
  uint32_t* meta = reinterpret_cast<uint32_t*>(ws + p.meta_off);
  int64_t* nseg = reinterpret_cast<int64_t*>(ws + p.nseg_off);
  int64_t* segbase = reinterpret_cast<int64_t*>(ws + p.segbase_off);
  SegRec* segs = reinterpret_cast<SegRec*>(ws + p.segs_off);
  int64_t* m_in = reinterpret_cast<int64_t*>(ws + p.min_off);
  unsigned long long* maxabs = reinterpret_cast<unsigned long long*>(ws + p.misc_off);
  int64_t* total = reinterpret_cast<int64_t*>(ws + p.misc_off + 8);
  int* fail = reinterpret_cast<int*>(ws + p.misc_off + 16);
  cudaError_t e = cudaMemsetAsync(ws + p.misc_off, 0, 256, s);
  if (e != cudaSuccess) return e;
  // per-segment MAP step counts are accumulated with atomics: clear them
  e = cudaMemsetAsync(segs, 0, (size_t)p.seg_cap * sizeof(SegRec), s);
  if (e != cudaSuccess) return e;
  if (p.ntiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned g = (unsigned)p.ntiles;
  CR_LAUNCH(kKChainTileSum, s, chain_tile_sum_kernel<T><<<g, kCT, 0, s>>>(src, p.K, tsum));
  CR_LAUNCH(kKChainOffsets, s,
            exclusive_scan_1block<double><<<1, 1024, 0, s>>>(tsum, toff, p.ntiles, nullptr));
  CR_LAUNCH(kKChainPrefix, s,
            chain_prefix_kernel<T><<<g, kCT, 0, s>>>(src, p.K, toff, pre, maxabs));
  CR_LAUNCH(kKChainClassify, s,
            chain_classify_kernel<T><<<g, kCT, 0, s>>>(src, p.K, pre, maxabs, qv, meta, nseg));
  CR_LAUNCH(kKChainOffsets, s,
            exclusive_scan_1block<int64_t><<<1, 1024, 0, s>>>(nseg, segbase, p.ntiles, total));
  CR_LAUNCH(kKChainSegments, s,
            chain_segments_kernel<T><<<g, kCT, 0, s>>>(src, qv, meta, p.K, segbase, segs,
                                                       p.seg_cap, fail));
  CR_LAUNCH(kKChainWalk, s,
            chain_walk_kernel<T><<<1, 32, 0, s>>>(src, dst, segs, total, p.seg_cap, m_in, fail));
  CR_LAUNCH(kKChainFill, s,
            chain_fill_kernel<T><<<g, kCT, 0, s>>>(qv, meta, p.K, segbase, segs, p.seg_cap, m_in,
                                                   dst, fail));
  CR_LAUNCH(kKChainFallback, s, chain_fallback_kernel<T><<<1, 32, 0, s>>>(src, dst, p.K, fail));
  return cudaGetLastError();
}

template cudaError_t run_chain<double>(const ChainPlan&, const double*, double*, char*,
                                       cudaStream_t);
template cudaError_t run_chain<float>(const ChainPlan&, const float*, float*, char*,
                                      cudaStream_t);

}  // namespace cr
