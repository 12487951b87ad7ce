// Row helpers shared by the row-streaming kernels (ts_sample.cu, ts_chain.cu): 16-byte
// vectors of logits or probabilities, composite-key tokens, warp sorts, scans and list
// reservations.
#pragma once

#include <stdint.h>

#include "ts_common.cuh"

namespace tsv {

template <typename E>
struct SVec;
template <>
struct SVec<float> {
  static constexpr int N = 4;
  static constexpr uint32_t kNegInfWord = 0xFF800000u;
  __device__ __forceinline__ static void unpack(const uint4& r, float* x) {
    x[0] = __uint_as_float(r.x);
    x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z);
    x[3] = __uint_as_float(r.w);
  }
  __device__ __forceinline__ static float vmax(const uint4& r) {
    return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                 fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
  }
  __device__ __forceinline__ static float vmin(const uint4& r) {
    return fminf(fminf(__uint_as_float(r.x), __uint_as_float(r.y)),
                 fminf(__uint_as_float(r.z), __uint_as_float(r.w)));
  }
  __device__ __forceinline__ static float at(const float* p, int64_t i) { return p[i]; }
  // element q (a run-time index) of a vector, by selects (no indexed register access)
  __device__ __forceinline__ static float elem(const uint4& r, int q) {
    const uint32_t w = q < 2 ? (q == 0 ? r.x : r.y) : (q == 2 ? r.z : r.w);
    return __uint_as_float(w);
  }
};
template <>
struct SVec<uint16_t> {
  static constexpr int N = 8;
  static constexpr uint32_t kNegInfWord = 0xFF80FF80u;
  __device__ __forceinline__ static void unpack(const uint4& r, float* x) {
    x[0] = __uint_as_float(r.x << 16);
    x[1] = __uint_as_float(r.x & 0xFFFF0000u);
    x[2] = __uint_as_float(r.y << 16);
    x[3] = __uint_as_float(r.y & 0xFFFF0000u);
    x[4] = __uint_as_float(r.z << 16);
    x[5] = __uint_as_float(r.z & 0xFFFF0000u);
    x[6] = __uint_as_float(r.w << 16);
    x[7] = __uint_as_float(r.w & 0xFFFF0000u);
  }
  __device__ __forceinline__ static uint32_t bmax2(uint32_t p, uint32_t q) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(p), "r"(q));
    return d;
  }
  __device__ __forceinline__ static float vmax(const uint4& r) {
    const uint32_t m = bmax2(bmax2(r.x, r.y), bmax2(r.z, r.w));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  __device__ __forceinline__ static uint32_t bmin2(uint32_t p, uint32_t q) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(p), "r"(q));
    return d;
  }
  __device__ __forceinline__ static float vmin(const uint4& r) {
    const uint32_t m = bmin2(bmin2(r.x, r.y), bmin2(r.z, r.w));
    return fminf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  __device__ __forceinline__ static float at(const uint16_t* p, int64_t i) {
    return bf16_bits_to_f32(p[i]);
  }
  // element q (a run-time index) of a vector, by selects (no indexed register access)
  __device__ __forceinline__ static float elem(const uint4& r, int q) {
    const uint32_t w = q < 4 ? (q < 2 ? r.x : r.y) : (q < 6 ? r.z : r.w);
    return __uint_as_float((q & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
};

// Appends this lane's candidates (bit u * N + q of m32: element q of vector rv[u], token
// c0 + (vbase + 32 u) N + q) to the list at pos .. as composite keys, one set bit at a
// time, so that a warp spends one step per candidate of its busiest lane rather than one
// per element slot. Entries at or past cap are dropped (the count still advances).
template <typename E, int NV>
__device__ __forceinline__ void append_candidates(uint32_t m32, const uint4 (&rv)[NV], int c0,
                                                  int vbase, uint32_t pos, uint64_t* list,
                                                  uint32_t cap) {
  constexpr int N = SVec<E>::N;
  while (m32) {
    const int b = __ffs(m32) - 1;
    m32 &= m32 - 1u;
    const int u = b / N, q = b % N;
    uint4 r = rv[0];
#pragma unroll
    for (int uu = 1; uu < NV; ++uu)
      if (u == uu) r = rv[uu];
    if (pos < cap)
      list[pos] = comp_key(fkey(SVec<E>::elem(r, q)), (uint32_t)(c0 + (vbase + u * 32) * N + q));
    ++pos;
  }
}

__device__ __forceinline__ uint32_t comp_token(uint64_t c) {
  return kIdxMax - (uint32_t)(c & kIdxMax);
}

// Warp reductions by butterfly: every lane ends with the same bits.
__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Ascending bitonic sort of the 32 E values of a warp, element e * 32 + lane in v[e].
template <int E>
__device__ __forceinline__ void warp_bitonic_asc(uint64_t (&v)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int kb = 2; kb <= 32 * E; kb <<= 1) {
#pragma unroll
    for (int jb = kb >> 1; jb > 0; jb >>= 1) {
      if (jb >= 32) {
        const int jj = jb >> 5;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (e & jj) continue;
          const bool up = ((e * 32 + lane) & kb) == 0;
          const uint64_t lo = v[e], hi = v[e ^ jj];
          if (up ? (lo > hi) : (lo < hi)) {
            v[e] = hi;
            v[e ^ jj] = lo;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const bool up = ((e * 32 + lane) & kb) == 0;
          const uint64_t pv = __shfl_xor_sync(0xffffffffu, v[e], jb);
          const bool lower = (lane & jb) == 0;
          v[e] = (lower == up) ? (v[e] < pv ? v[e] : pv) : (v[e] > pv ? v[e] : pv);
        }
      }
    }
  }
}

// Inclusive scan of the warp's 32 E values in element order (e * 32 + lane); returns the
// total.
template <int E>
__device__ __forceinline__ uint64_t warp_scan_incl(uint64_t (&v)[E]) {
  const int lane = threadIdx.x & 31;
  uint64_t carry = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    uint64_t x = v[e];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    v[e] = x + carry;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  return carry;
}

// Exclusive scan of a double over the consumer threads in thread order (a fixed order of

// Reserves n consecutive entries of a shared list for each lane of the (converged) warp
// with one atomic on the list's counter; returns the lane's first entry.
__device__ __forceinline__ uint32_t warp_reserve(uint32_t* counter, uint32_t n, int lane) {
  uint32_t incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
  uint32_t base = 0;
  if (lane == 31 && total) base = atomicAdd(counter, total);
  return __shfl_sync(0xffffffffu, base, 31) + incl - n;
}


// Exclusive scan of a double over the NW warps of the calling threads (the first NW*32 of
// the CTA, synchronised by Bar) in thread order: a fixed order of additions, so the result
// is reproducible. Writes the total; sc needs NW entries.
template <int NW, class Bar>
__device__ __forceinline__ double excl_scan_f64_t(double v, double* sc, double& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sc[w] = incl;
  Bar::sync();
  if (w == 0) {
    double t = lane < NW ? sc[lane] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < NW) sc[lane] = t;
  }
  Bar::sync();
  const double before = (w > 0) ? sc[w - 1] : 0.0;
  total = sc[NW - 1];
  Bar::sync();
  return before + (incl - v);
}

}  // namespace tsv
