// Integer maps of the exact parallel carry chain (see cr_chain.cu): a step of
// the chain C_k = fl(C_{k-1} + T_k), with C in units of its binade, is a map
//     M -> a M + b[parity(M)]   (mod 2^64),  a = 2^j,
// and so is any composition of such steps. This header also compiles as
// plain C++ so that the map algebra can be checked on the host.
#ifndef CR_CHAIN_MAP_H_
#define CR_CHAIN_MAP_H_

#include <cstdint>

#if defined(__CUDACC__)
#define CR_MAP_FN __host__ __device__ __forceinline__
#else
#define CR_MAP_FN inline
#endif

namespace cr {

struct Map {
  uint64_t a, b0, b1;
};
CR_MAP_FN Map map_id() { return Map{1, 0, 0}; }
CR_MAP_FN uint64_t bsel(const Map& g, uint64_t p) { return p ? g.b1 : g.b0; }
CR_MAP_FN Map compose(const Map& g, const Map& h) {  // first g, then h
  const uint64_t p0 = (g.b0 & 1);                    // parity after g, from even M
  const uint64_t p1 = ((g.a & 1) ^ g.b1) & 1;        // parity after g, from odd M
  return Map{h.a * g.a, h.a * g.b0 + bsel(h, p0), h.a * g.b1 + bsel(h, p1)};
}
CR_MAP_FN uint64_t apply(const Map& g, uint64_t M) { return g.a * M + bsel(g, M & 1); }

// Index of the lowest set bit of a nonzero a.
CR_MAP_FN int low_bit(uint64_t a) {
#if defined(__CUDA_ARCH__)
  return __ffsll((long long)a) - 1;
#else
  return __builtin_ctzll(a);
#endif
}

// A rise by d binades after a map g = 2^j M + b[p] with d <= j: the rise
// rounds A = g(M) + q to the coarser unit, M1 = (A + 2^(d-1) - 1 + x) >> d
// with x = [f > 0] | bit d of A (half to even). 2^j M is a multiple of 2^d,
// so M1 = 2^(j-d) M + ((B + 2^(d-1) - 1 + x) >> d), B = b[p] + q, and bit d
// of A is bit d of B (plus M's parity when j = d): again a map of the same
// form. Exact when B is the true integer: along a valid chain |b[p]| <
// 2^53 + 2^(53+j) and |q| < 2^(53+d), so j <= kFoldMaxDrop keeps it in int64.
constexpr int kFoldMaxDrop = 7;
CR_MAP_FN bool rise_foldable(const Map& g, int d) {
  if (g.a == 0 || (g.a & (g.a - 1)) != 0) return false;
  const int j = low_bit(g.a);
  return d >= 1 && d <= j && j <= kFoldMaxDrop;
}
CR_MAP_FN Map fold_rise(const Map& g, int d, int64_t q, bool fpos) {
  const int j = low_bit(g.a);
  const uint64_t c = (uint64_t(1) << (d - 1)) - 1;
  uint64_t b[2];
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const uint64_t B = (p ? g.b1 : g.b0) + (uint64_t)q;
    const uint64_t bit = ((B >> d) ^ (j == d ? (uint64_t)p : 0ull)) & 1ull;
    const uint64_t x = fpos ? 1ull : bit;
    b[p] = (uint64_t)((int64_t)(B + c + x) >> d);
  }
  return Map{g.a >> d, b[0], b[1]};
}

}  // namespace cr

#endif  // CR_CHAIN_MAP_H_
