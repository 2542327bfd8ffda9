// Exact parallel evaluation of a floating-point left fold
//     C_0 = T_0,   C_k = fl(C_{k-1} + T_k)   (round to nearest even)
// the carry chain of block_dyadic<B> (P4229R0 on "Canonical Parallel
// Reduction and Scan": blocks chained left to right) and the whole 1-D
// left_fold scan. The result is bit-identical to the serial chain.
//
// Why it can be parallel. Let u = 2^(e - p) be the unit in the last place of
// binade e (|v| in [2^e, 2^(e+1)), p = 52 or 23 fraction bits). If C_{k-1}
// is an integer multiple M of u and the exact sum s = C_{k-1} + T_k lies in
// binade e, then fl(s) = u * RNE(M + T_k/u). With T_k/u = q + f (q integer,
// 0 <= f < 1): fl(s)/u = A + d, A = M + q, d = [f > 1/2] or, when f is
// exactly 1/2, [A odd] (ties to even). So inside a stretch of steps whose
// sums stay in one binade, every rounded add is an integer step
//     M -> M + b[parity(M)],   b[p] = q + d(f, p xor (q & 1)),
// and such maps compose associatively: (first g, then h)
//     b[p] = g.b[p] + h.b[(p + g.b[p]) & 1].
// The only sequential work left is where the binade changes ("breaks").
//
// Passes (tile = 2048 steps, 8 per thread):
//   1 tile sums of T             (approximate prefix, any order)
//   2 tile offsets               (one block)
//   3 prefix P~_k + max |P~|      (the chain stays within a proven margin
//                                  mu = K * ulp(2 max|P~|) of P~_k)
//   4 classify each step: binade and sign of s_k from P~_k when the whole
//     interval P~_k +- mu lies inside one binade; else "uncertain". A step
//     starts a new segment (break) when its class differs from the previous
//     step's or is uncertain. Non-break steps store (q_k, f class).
//   5 segment bases (one block), 6 segment maps (composition per segment),
//   7 walk (one thread): at each break C = fl(C + T_k) with a real add, then
//     M = C / u (checked integral), then the segment's composed map,
//   8 fill: every step recomputed from its segment's entry value with an
//     exact range check that s_k really lies in the predicted binade and
//     sign; C_k = M_k * u.
//   9 if any check failed (or segments overflowed their buffer), the plain
//     serial chain recomputes everything on the device (no host sync).
// Every fp add of the chain is therefore either the real add (breaks,
// fallback) or proven equal to it by integer arithmetic.
#include <cstdint>

#include "cr_chain.h"
#include "cr_device.cuh"
#include "cr_launch.h"

namespace cr {
namespace {

constexpr int kCT = 256;          // threads per tile
constexpr int kCE = 8;            // steps per thread
constexpr int kCTile = kCT * kCE; // 2048 steps per tile

template <class T>
struct FP;
template <>
struct FP<double> {
  using U = uint64_t;
  static constexpr int P = 52, BIAS = 1023, EMIN = -1022, EMAX = 1023;
  __device__ static U bits(double v) { return (U)__double_as_longlong(v); }
};
template <>
struct FP<float> {
  using U = uint32_t;
  static constexpr int P = 23, BIAS = 127, EMIN = -126, EMAX = 127;
  __device__ static U bits(float v) { return (U)__float_as_uint(v); }
};

// f classes of T/u - q
enum : uint32_t { kFZero = 0, kFLow = 1, kFHalf = 2, kFHigh = 3 };
// meta word of a step: bit0 break, bit1 certain, bit2 negative sign,
// bits 3-4 f class, bits 8..19 binade e + 2048
__device__ __forceinline__ uint32_t make_meta(bool brk, bool certain, bool neg, uint32_t fcls,
                                              int e) {
  return (brk ? 1u : 0u) | (certain ? 2u : 0u) | (neg ? 4u : 0u) | (fcls << 3) |
         ((uint32_t)(e + 2048) << 8);
}
__device__ __forceinline__ bool meta_break(uint32_t m) { return m & 1u; }
__device__ __forceinline__ bool meta_certain(uint32_t m) { return m & 2u; }
__device__ __forceinline__ bool meta_neg(uint32_t m) { return m & 4u; }
__device__ __forceinline__ uint32_t meta_fcls(uint32_t m) { return (m >> 3) & 3u; }
__device__ __forceinline__ int meta_e(uint32_t m) { return (int)((m >> 8) & 0xFFFu) - 2048; }

struct Map {  // M -> M + b[parity(M)] (two's complement, wraps like the hardware)
  uint64_t b0, b1;
};
__device__ __forceinline__ Map map_id() { return Map{0, 0}; }
__device__ __forceinline__ Map compose(Map g, Map h) {  // first g, then h
  const uint64_t g0 = g.b0, g1 = g.b1;
  return Map{g0 + ((g0 & 1) ? h.b1 : h.b0), g1 + (((1 + g1) & 1) ? h.b1 : h.b0)};
}
__device__ __forceinline__ uint64_t apply(Map g, uint64_t M) {
  return M + ((M & 1) ? g.b1 : g.b0);
}
__device__ __forceinline__ uint32_t delta(uint32_t fcls, uint64_t A) {
  return fcls == kFHigh ? 1u : (fcls == kFHalf ? (uint32_t)(A & 1) : 0u);
}
__device__ __forceinline__ Map step_map(int64_t q, uint32_t fcls) {
  const uint64_t uq = (uint64_t)q;
  // p = parity of the incoming M; A = M + q has parity p ^ (q & 1)
  return Map{uq + delta(fcls, uq & 1), uq + delta(fcls, (uq & 1) ^ 1)};
}

// T / 2^(e - P) = q + f, 0 <= f < 1, classified. Returns false when q would
// not fit (|T| far above the unit: never a valid in-binade step).
template <class T>
__device__ __forceinline__ bool split_unit(T t, int e, int64_t& q, uint32_t& fcls) {
  using F = FP<T>;
  const typename F::U b = F::bits(t);
  const int bexp = (int)((b >> F::P) & ((1u << (sizeof(T) * 8 - 1 - F::P)) - 1));
  uint64_t mant = (uint64_t)(b & ((typename F::U(1) << F::P) - 1));
  if (bexp == 0 && mant == 0) {
    q = 0;
    fcls = kFZero;
    return true;
  }
  int et;  // t = mant * 2^et
  if (bexp == 0) {
    et = F::EMIN - F::P;  // subnormal
  } else {
    mant |= uint64_t(1) << F::P;
    et = bexp - F::BIAS - F::P;
  }
  const bool neg = (b >> (sizeof(T) * 8 - 1)) & 1;
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

// s = M*u + T lies in the predicted binade and sign: exact integer test on
// A = M + q (see the header comment).
template <class T>
__device__ __forceinline__ bool in_binade(int64_t A, bool neg, uint32_t fcls) {
  constexpr int64_t LO = int64_t(1) << FP<T>::P, HI = int64_t(1) << (FP<T>::P + 1);
  if (!neg) return A >= LO && A <= HI - 1;
  const bool fz = fcls == kFZero;
  return (fz ? A <= -LO : A <= -LO - 1) && (fz ? A >= -HI + 1 : A >= -HI);
}

template <class T>
__device__ __forceinline__ T scale_pow2(int64_t M, int e) {  // M * 2^(e - P), exact
  return (T)ldexp((double)M, e - FP<T>::P);
}

// ---------------------------------------------------------------- pass 1
template <class T>
__global__ void __launch_bounds__(kCT) chain_tile_sum_kernel(const T* src, int64_t K,
                                                             double* tsum) {
  __shared__ double sh[kCT];
  const int t = threadIdx.x;
  const int64_t k0 = (int64_t)blockIdx.x * kCTile + (int64_t)t * kCE;
  double s = 0.0;
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

// ---------------------------------------------------------------- pass 2
// Exclusive prefix over the tile sums, and the segment bases (same shape).
__global__ void __launch_bounds__(1024) chain_offsets_kernel(const double* tsum, double* toff,
                                                             int64_t ntiles) {
  __shared__ double sh[1024];
  __shared__ double carry;
  const int t = threadIdx.x;
  if (t == 0) carry = 0.0;
  __syncthreads();
  for (int64_t base = 0; base < ntiles; base += 1024) {
    const int64_t i = base + t;
    const double v = i < ntiles ? tsum[i] : 0.0;
    sh[t] = v;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const double a = t >= off ? sh[t - off] : 0.0;
      __syncthreads();
      sh[t] += a;
      __syncthreads();
    }
    if (i < ntiles) toff[i] = carry + sh[t] - v;
    __syncthreads();
    if (t == 0) carry += sh[1023];
    __syncthreads();
  }
}

__global__ void __launch_bounds__(1024) chain_seg_base_kernel(const int* nseg, int64_t* base,
                                                              int64_t ntiles, int64_t* total) {
  __shared__ int64_t sh[1024];
  __shared__ int64_t carry;
  const int t = threadIdx.x;
  if (t == 0) carry = 0;
  __syncthreads();
  for (int64_t b0 = 0; b0 < ntiles; b0 += 1024) {
    const int64_t i = b0 + t;
    const int64_t v = i < ntiles ? nseg[i] : 0;
    sh[t] = v;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {
      const int64_t a = t >= off ? sh[t - off] : 0;
      __syncthreads();
      sh[t] += a;
      __syncthreads();
    }
    if (i < ntiles) base[i] = carry + sh[t] - v;
    __syncthreads();
    if (t == 0) carry += sh[1023];
    __syncthreads();
  }
  if (t == 0) *total = carry;
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
  for (int i = 0; i < kCE; ++i) {
    if (k0 + i < K) {
      run += v[i];
      pre[k0 + i] = run;
      mx = fmax(mx, fabs(run));
    }
  }
  if (!(mx <= 1.7e308)) mx = 1.7e308;  // non-finite: classify as uncertain later
  atomicMax(maxabs, (unsigned long long)__double_as_longlong(mx));
}

// ---------------------------------------------------------------- pass 4
// Class of the exact sum s_k from P~_k: (certain, negative, binade e).
template <class T>
__device__ __forceinline__ void classify(double p, double mu, bool& certain, bool& neg, int& e) {
  certain = false;
  neg = p < 0;
  e = 0;
  const double a = fabs(p);
  if (!(a <= 1e300)) return;  // non-finite
  if (a - mu <= 0.0) return;  // sign or zero uncertain
  const int ee = ilogb(a);
  if (ee < FP<T>::EMIN + 2 || ee > FP<T>::EMAX - 2) return;  // near subnormal / overflow
  const double lo = ldexp(1.0, ee), hi = ldexp(1.0, ee + 1);
  const double ulp = ldexp(1.0, ee - FP<T>::P);
  if (a - mu < lo || a + mu + ulp >= hi) return;  // interval crosses a binade edge
  certain = true;
  e = ee;
}

template <class T>
__global__ void __launch_bounds__(kCT) chain_classify_kernel(
    const T* src, int64_t K, const double* pre, const unsigned long long* maxabs, int64_t* qv,
    uint32_t* meta, int* tile_nseg) {
  __shared__ int cnt[kCT];
  const int t = threadIdx.x;
  const int64_t k0 = (int64_t)blockIdx.x * kCTile + (int64_t)t * kCE;
  // margin mu = K * ulp(2 max|P~|) bounds both |C_k - P_k| (K roundings of at
  // most half an ulp of |C| <= 2 max|P~|) and |P~_k - P_k|
  const double mx = __longlong_as_double((long long)*maxabs);
  double mu;
  {
    const double m2 = 2.0 * mx;
    const int em = m2 > 0 ? ilogb(m2) : -1074;
    mu = (double)K * ldexp(1.0, em - FP<T>::P);
    if (!(mu <= 1e300)) mu = 1e300;
  }
  int nbrk = 0;
  bool pc, pn;
  int pe;
  if (k0 == 0 || k0 > K) {
    pc = false; pn = false; pe = 0;
  } else {
    classify<T>(pre[k0 - 1], mu, pc, pn, pe);
  }
  for (int i = 0; i < kCE; ++i) {
    const int64_t k = k0 + i;
    if (k >= K) break;
    bool c, n;
    int e;
    classify<T>(pre[k], mu, c, n, e);
    bool brk = (k == 0) || !c || !pc || n != pn || e != pe;
    int64_t q = 0;
    uint32_t f = 0;
    if (!brk && !split_unit<T>(src[k], e, q, f)) brk = true;
    meta[k] = make_meta(brk, c, n, f, e);
    qv[k] = q;
    nbrk += brk ? 1 : 0;
    pc = c; pn = n; pe = e;
  }
  cnt[t] = nbrk;
  __syncthreads();
  for (int w = kCT / 2; w > 0; w >>= 1) {
    if (t < w) cnt[t] += cnt[t + w];
    __syncthreads();
  }
  if (t == 0) {
    // segments of this tile: one per break, plus one if the tile starts
    // inside a run (its first step is not a break)
    const int64_t first = (int64_t)blockIdx.x * kCTile;
    tile_nseg[blockIdx.x] = cnt[0] + (meta_break(meta[first]) ? 0 : 1);
  }
}

// ---------------------------------------------------------------- pass 6
// Per-thread summary for the in-tile segmented scan:
//   map: composition of the steps after the thread's last break (or all)
//   brk: number of breaks in the thread
struct Summ {
  Map map;
  int brk;
};
__device__ __forceinline__ Summ combine(Summ l, Summ r) {
  return r.brk ? Summ{r.map, l.brk + r.brk} : Summ{compose(l.map, r.map), l.brk};
}

// Segment record. A segment starts at a break (its first step is done with a
// real add) or at a tile start inside a run (continuation); `map` composes
// its remaining steps.
struct SegRec {
  int64_t start;
  Map map;
  int32_t e;
  int32_t flags;  // bit0 starts with a break, bit1 class certain
};

template <class T>
__device__ __forceinline__ void thread_scan(const int64_t* qv, const uint32_t* meta,
                                            int64_t k0, int64_t K, Summ& in_excl,
                                            Summ* sh) {
  Summ me{map_id(), 0};
  for (int i = 0; i < kCE; ++i) {
    const int64_t k = k0 + i;
    if (k >= K) break;
    const uint32_t m = meta[k];
    if (meta_break(m)) {
      me.map = map_id();
      me.brk += 1;
    } else {
      me.map = compose(me.map, step_map(qv[k], meta_fcls(m)));
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
    const int64_t* qv, const uint32_t* meta, int64_t K, const int64_t* seg_base,
    SegRec* segs, int64_t seg_cap, int* fail) {
  __shared__ Summ sh[kCT];
  const int t = threadIdx.x;
  const int64_t tile0 = (int64_t)blockIdx.x * kCTile;
  const int64_t k0 = tile0 + (int64_t)t * kCE;
  Summ in;
  thread_scan<T>(qv, meta, k0, K, in, sh);
  const bool cont = !meta_break(meta[tile0]);  // tile begins inside a run
  // segment ordinal (within the tile) of the segment open at my first step
  int64_t ord = (cont ? 1 : 0) + in.brk - 1;
  Map cur = in.map;
  const int64_t base = seg_base[blockIdx.x];
  if (t == 0 && cont) {
    if (base < seg_cap) {
      SegRec& r = segs[base];
      r.start = tile0;
      const uint32_t m = meta[tile0];
      r.e = meta_e(m);
      r.flags = meta_certain(m) ? 2 : 0;
    } else {
      atomicExch(fail, 2);
    }
  }
  for (int i = 0; i < kCE; ++i) {
    const int64_t k = k0 + i;
    if (k >= K) break;
    const uint32_t m = meta[k];
    if (meta_break(m)) {
      if (ord >= 0 && base + ord < seg_cap) segs[base + ord].map = cur;  // close
      ord += 1;
      cur = map_id();
      if (base + ord < seg_cap) {
        SegRec& r = segs[base + ord];
        r.start = k;
        r.e = meta_e(m);
        r.flags = 1 | (meta_certain(m) ? 2 : 0);
      } else {
        atomicExch(fail, 2);
      }
    } else {
      cur = compose(cur, step_map(qv[k], meta_fcls(m)));
    }
  }
  // the thread holding the tile's last step closes the open segment
  const int64_t last = (tile0 + kCTile < K ? tile0 + kCTile : K) - 1;
  if (k0 <= last && last < k0 + kCE && ord >= 0 && base + ord < seg_cap)
    segs[base + ord].map = cur;
}

// ---------------------------------------------------------------- pass 7
// One warp: all lanes load the next 32 segment records (and the break
// operands) while lane 0 runs the current 32 in order; records move to lane 0
// by shuffles, so the sequential part never waits on memory.
template <class T>
__global__ void chain_walk_kernel(const T* src, T* dst, const SegRec* segs,
                                  const int64_t* nseg_total, int64_t seg_cap, int64_t* m_in,
                                  int* fail) {
  if (blockIdx.x != 0) return;
  const int lane = threadIdx.x;
  const int64_t nseg = *nseg_total;
  if (*fail || nseg > seg_cap) {
    if (lane == 0) atomicExch(fail, 2);
    return;
  }
  T C = src[0];
  uint64_t M = 0;
  bool bad = false;
  // registers of the batch being loaded
  SegRec nr{};
  T nt = T(0);
  if (lane < nseg) {
    nr = segs[lane];
    nt = src[nr.start];
  }
  for (int64_t b0 = 0; b0 < nseg; b0 += 32) {
    const SegRec cr = nr;
    const T ct = nt;
    const int64_t nb = b0 + 32 + lane;
    if (nb < nseg) {  // prefetch the next batch
      nr = segs[nb];
      nt = src[nr.start];
    }
    const int cnt = (int)(nseg - b0 < 32 ? nseg - b0 : 32);
    for (int j = 0; j < cnt; ++j) {
      const int64_t start = __shfl_sync(0xffffffffu, cr.start, j);
      const uint64_t mb0 = __shfl_sync(0xffffffffu, cr.map.b0, j);
      const uint64_t mb1 = __shfl_sync(0xffffffffu, cr.map.b1, j);
      const int e = __shfl_sync(0xffffffffu, cr.e, j);
      const int flags = __shfl_sync(0xffffffffu, cr.flags, j);
      const T tv = __shfl_sync(0xffffffffu, ct, j);
      if (lane == 0 && !bad) {
        if (flags & 1) {  // break: the real add
          C = (start == 0) ? tv : add_rn(C, tv);
          dst[start] = C;
          if (flags & 2) {  // certain class: enter integer units of binade e
            const double v = ldexp((double)C, FP<T>::P - e);
            const double iv = trunc(v);
            if (!(iv == v) || !(fabs(v) <= ldexp(1.0, FP<T>::P + 1))) bad = true;
            M = (uint64_t)(int64_t)iv;
          }
        }
        m_in[b0 + j] = (int64_t)M;
        if (!bad && (flags & 2)) {
          M = apply(Map{mb0, mb1}, M);
          const int64_t Ms = (int64_t)M;
          if (Ms > (int64_t(1) << (FP<T>::P + 1)) || Ms < -(int64_t(1) << (FP<T>::P + 1)))
            bad = true;
          else
            C = scale_pow2<T>(Ms, e);
        }
      }
    }
  }
  if (lane == 0 && bad) atomicExch(fail, 1);
}

// ---------------------------------------------------------------- pass 8
template <class T>
__global__ void __launch_bounds__(kCT) chain_fill_kernel(const int64_t* qv, const uint32_t* meta,
                                                         int64_t K, const int64_t* seg_base,
                                                         const SegRec* segs, int64_t seg_cap,
                                                         const int64_t* m_in, T* dst,
                                                         int* fail) {
  __shared__ Summ sh[kCT];
  const int t = threadIdx.x;
  const int64_t tile0 = (int64_t)blockIdx.x * kCTile;
  const int64_t k0 = tile0 + (int64_t)t * kCE;
  Summ in;
  thread_scan<T>(qv, meta, k0, K, in, sh);
  if (*fail) return;
  const bool cont = !meta_break(meta[tile0]);
  int64_t seg = seg_base[blockIdx.x] + (cont ? 1 : 0) + in.brk - 1;
  uint64_t M = 0;
  int e = 0;
  bool live = false;  // M is meaningful (segment of certain class)
  if (k0 < K && seg >= 0 && seg < seg_cap) {
    const SegRec r = segs[seg];
    live = (r.flags & 2) != 0;
    e = r.e;
    M = apply(in.map, (uint64_t)m_in[seg]);
  }
  bool ok = true;
  for (int i = 0; i < kCE; ++i) {
    const int64_t k = k0 + i;
    if (k >= K) break;
    const uint32_t m = meta[k];
    if (meta_break(m)) {  // value written by the walk; enter the next segment
      seg += 1;
      if (seg >= seg_cap) { ok = false; break; }
      const SegRec r = segs[seg];
      live = (r.flags & 2) != 0;
      e = r.e;
      M = (uint64_t)m_in[seg];
      continue;
    }
    if (!live) { ok = false; break; }
    const int64_t A = (int64_t)M + qv[k];
    const uint32_t f = meta_fcls(m);
    if (!in_binade<T>(A, meta_neg(m), f)) { ok = false; break; }
    M = (uint64_t)(A + (int64_t)delta(f, (uint64_t)A));
    dst[k] = scale_pow2<T>((int64_t)M, e);
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
  p.nseg_off = off; off += r256(p.ntiles * sizeof(int));
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
  int* nseg = reinterpret_cast<int*>(ws + p.nseg_off);
  int64_t* segbase = reinterpret_cast<int64_t*>(ws + p.segbase_off);
  SegRec* segs = reinterpret_cast<SegRec*>(ws + p.segs_off);
  int64_t* m_in = reinterpret_cast<int64_t*>(ws + p.min_off);
  unsigned long long* maxabs = reinterpret_cast<unsigned long long*>(ws + p.misc_off);
  int64_t* total = reinterpret_cast<int64_t*>(ws + p.misc_off + 8);
  int* fail = reinterpret_cast<int*>(ws + p.misc_off + 16);
  cudaError_t e = cudaMemsetAsync(ws + p.misc_off, 0, 256, s);
  if (e != cudaSuccess) return e;
  if (p.ntiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned g = (unsigned)p.ntiles;
  CR_LAUNCH(kKChainTileSum, s, chain_tile_sum_kernel<T><<<g, kCT, 0, s>>>(src, p.K, tsum));
  CR_LAUNCH(kKChainOffsets, s, chain_offsets_kernel<<<1, 1024, 0, s>>>(tsum, toff, p.ntiles));
  CR_LAUNCH(kKChainPrefix, s,
            chain_prefix_kernel<T><<<g, kCT, 0, s>>>(src, p.K, toff, pre, maxabs));
  CR_LAUNCH(kKChainClassify, s,
            chain_classify_kernel<T><<<g, kCT, 0, s>>>(src, p.K, pre, maxabs, qv, meta, nseg));
  CR_LAUNCH(kKChainOffsets, s,
            chain_seg_base_kernel<<<1, 1024, 0, s>>>(nseg, segbase, p.ntiles, total));
  CR_LAUNCH(kKChainSegments, s,
            chain_segments_kernel<T><<<g, kCT, 0, s>>>(qv, meta, p.K, segbase, segs, p.seg_cap,
                                                       fail));
  CR_LAUNCH(kKChainWalk, s,
            chain_walk_kernel<T><<<1, 32, 0, s>>>(src, dst, segs, total, p.seg_cap, m_in,
                                                  fail));
  CR_LAUNCH(kKChainFill, s,
            chain_fill_kernel<T><<<g, kCT, 0, s>>>(qv, meta, p.K, segbase, segs, p.seg_cap,
                                                   m_in, dst, fail));
  CR_LAUNCH(kKChainFallback, s,
            chain_fallback_kernel<T><<<1, 32, 0, s>>>(src, dst, p.K, fail));
  return cudaGetLastError();
}

template cudaError_t run_chain<double>(const ChainPlan&, const double*, double*, char*,
                                       cudaStream_t);
template cudaError_t run_chain<float>(const ChainPlan&, const float*, float*, char*,
                                      cudaStream_t);

}  // namespace cr
