// CTA-level selection helpers for the row-streaming and cluster-staged kernels: exact
// scans and radix selections over 64-bit composite keys (value descending, then token id
// ascending), with masses summed exactly as three 32-bit digit counters.
#pragma once

#include <stdint.h>

#include "ts_common.cuh"

namespace tsv {
namespace sel {


// Barrier policies: the whole CTA, or the 256 consumer threads of a warp-specialised CTA
// (named barrier 1; the producer warp never takes part).
struct BlockBar {
  __device__ __forceinline__ static void sync() { __syncthreads(); }
};
struct ConsumerBar {
  __device__ __forceinline__ static void sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
};

// Scratch a CTA needs for one selection at a time.
struct Scratch {
  uint32_t m3[3][256];  // per-bin mass as 14-, 14- and 13-bit digit sums
  uint32_t cnt[256];    // per-bin counts
  uint64_t scan[32];    // per-warp partials
  int32_t bin, bincnt;
  uint64_t above, aux, gmax;
};

// Exact accumulation of a weight below 2^42 with 32-bit shared-memory atomics (no
// overflow for fewer than 2^18 additions per counter).
__device__ __forceinline__ void add3(uint32_t* d0, uint32_t* d1, uint32_t* d2, uint64_t w) {
  const uint32_t lo = (uint32_t)w & 0x3FFFu, mid = (uint32_t)(w >> 14) & 0x3FFFu;
  const uint32_t hi = (uint32_t)(w >> 28);
  if (lo) atomicAdd(d0, lo);
  if (mid) atomicAdd(d1, mid);
  if (hi) atomicAdd(d2, hi);
}
__device__ __forceinline__ uint64_t get3(uint32_t a0, uint32_t a1, uint32_t a2) {
  return (uint64_t)a0 + ((uint64_t)a1 << 14) + ((uint64_t)a2 << 28);
}

// Exclusive scan of a u64 over the block, in thread order; writes the block total.
template <int NT, class Bar = BlockBar>
__device__ __forceinline__ uint64_t excl_scan(uint64_t v, Scratch& s, uint64_t& total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s.scan[w] = incl;
  Bar::sync();
  if (w == 0) {
    uint64_t t = lane < NW ? s.scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < NW) s.scan[lane] = t;
  }
  Bar::sync();
  const uint64_t before = (w > 0) ? s.scan[w - 1] : 0;
  total = s.scan[NW - 1];
  Bar::sync();
  return before + incl - v;
}

// Warp 0 finds, scanning bins 255 -> 0 with weights wt(bin) after `above`, the first
// nonempty bin whose inclusive weight reaches `target`; writes s.bin (-1 if none),
// s.above (the weight before that bin) and s.bincnt.
template <class WT>
__device__ __forceinline__ void find_bin(Scratch& s, uint64_t above, uint64_t target, WT wt) {
  const int lane = threadIdx.x;
  unsigned long long lw = 0;
  for (int q = 0; q < 8; ++q) lw += wt(255 - 8 * lane - q);
  unsigned long long incl = lw;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  unsigned long long acc = above + (incl - lw), acc_at = 0;
  int found = -1;
  for (int q = 0; q < 8; ++q) {
    const int bin = 255 - 8 * lane - q;
    const uint32_t c = s.cnt[bin];
    const unsigned long long w = wt(bin);
    if (c > 0 && acc + w >= target) {
      found = bin;
      acc_at = acc;
      break;
    }
    acc += w;
  }
  const unsigned m = __ballot_sync(0xffffffffu, found >= 0);
  if (m == 0) {
    if (lane == 0) s.bin = -1;
  } else if (lane == __ffs(m) - 1) {
    s.bin = found;
    s.above = acc_at;
    s.bincnt = (int32_t)s.cnt[found];
  }
}

// Radix selection over the items item(0..n) that are >= lo_key, in descending order:
// count mode finds the `target` largest, mass mode the shortest top set whose mass (wfn
// of each item) reaches `target`. Returns the smallest selected item, so an item is
// selected iff it is >= the result. group_max receives the largest item of the final
// digit group (the crossing item itself once the group holds one item); beyond is set
// if the target lies past the eligible total (then every eligible item is selected).
//
// kU: items a thread takes at a time, loaded before any of them is counted (items read
// from global memory then have kU loads in flight).
template <int NT, bool MASS, class Bar = BlockBar, int kU = 1, class Item, class WFn>
__device__ uint64_t radix(int n, Item item, uint64_t lo_key, uint64_t target, WFn wfn,
                          const int* shifts, int nsh, Scratch& s, uint64_t* group_max = nullptr,
                          bool* beyond = nullptr) {
  uint64_t prefix = 0, mask = 0, above = 0;
  const int tid = threadIdx.x;
  bool all = false;
  for (int di = 0; di < nsh; ++di) {
    const int sh = shifts[di];
    for (int i = tid; i < 256; i += NT) {
      s.m3[0][i] = 0;
      s.m3[1][i] = 0;
      s.m3[2][i] = 0;
      s.cnt[i] = 0;
    }
    Bar::sync();
    for (int i0 = tid * kU; i0 < n; i0 += NT * kU) {
      uint64_t v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) v[u] = (i0 + u < n) ? item(i0 + u) : 0ull;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (i0 + u < n && v[u] >= lo_key && (v[u] & mask) == prefix) {
          const int b = (int)((v[u] >> sh) & 255u);
          atomicAdd(&s.cnt[b], 1u);
          if (MASS) add3(&s.m3[0][b], &s.m3[1][b], &s.m3[2][b], wfn(v[u]));
        }
      }
    }
    Bar::sync();
    if (tid < 32) {
      if (MASS)
        find_bin(s, above, target, [&](int b) { return get3(s.m3[0][b], s.m3[1][b], s.m3[2][b]); });
      else
        find_bin(s, above, target, [&](int b) { return (unsigned long long)s.cnt[b]; });
    }
    Bar::sync();
    const int bin = s.bin;
    const uint64_t ab = s.above;
    const int bc = s.bincnt;
    Bar::sync();
    if (bin < 0) {
      all = true;
      break;
    }
    prefix |= (uint64_t)bin << sh;
    mask |= (uint64_t)255u << sh;
    above = ab;
    if (!MASS && above + (uint64_t)bc == target) break;
    if (MASS && bc == 1) break;
  }
  if (beyond) *beyond = all;
  unsigned long long mn = ~0ull, gx = 0;
  for (int i0 = tid * kU; i0 < n; i0 += NT * kU) {
    uint64_t vv[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) vv[u] = (i0 + u < n) ? item(i0 + u) : 0ull;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const uint64_t v = vv[u];
      if (i0 + u >= n || v < lo_key) continue;
      if ((all || (v & mask) >= prefix) && v < mn) mn = v;
      if (!all && (v & mask) == prefix && v > gx) gx = v;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, mn, off);
    mn = y < mn ? y : mn;
    const unsigned long long z = __shfl_xor_sync(0xffffffffu, gx, off);
    gx = z > gx ? z : gx;
  }
  if (tid == 0) {
    s.aux = ~0ull;
    s.gmax = 0;
  }
  Bar::sync();
  if ((tid & 31) == 0) {
    atomicMin(reinterpret_cast<unsigned long long*>(&s.aux), mn);
    atomicMax(reinterpret_cast<unsigned long long*>(&s.gmax), gx);
  }
  Bar::sync();
  const uint64_t r = s.aux;
  if (group_max) *group_max = s.gmax;
  Bar::sync();
  return r;
}

// AND and OR of the 32-bit values f(i) over i < n with pred(i), reduced over the block
// (kU items a thread at a time, as in radix).
template <int NT, class Bar, int kU = 1, class F>
__device__ __forceinline__ void block_and_or(int n, F f, Scratch& s, uint32_t& and_, uint32_t& or_) {
  constexpr int NW = NT / 32;
  uint32_t a = 0xFFFFFFFFu, o = 0u;
  for (int i0 = (int)threadIdx.x * kU; i0 < n; i0 += NT * kU) {
    uint32_t v[kU];
    bool ok[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) ok[u] = (i0 + u < n) && f(i0 + u, v[u]);
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (ok[u]) {
        a &= v[u];
        o |= v[u];
      }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a &= __shfl_xor_sync(0xffffffffu, a, off);
    o |= __shfl_xor_sync(0xffffffffu, o, off);
  }
  if ((threadIdx.x & 31) == 0) s.scan[threadIdx.x >> 5] = ((uint64_t)a << 32) | o;
  Bar::sync();
  a = 0xFFFFFFFFu;
  o = 0u;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    a &= (uint32_t)(s.scan[w] >> 32);
    o |= (uint32_t)s.scan[w];
  }
  Bar::sync();
  and_ = a;
  or_ = o;
}

// The largest C, made of the keys' common top bits and whole 8-bit digits below them down
// to bit `lowbit`, such that at least k of the items key(0..n) are >= C (0 if fewer than
// k items): a lower bound for the k-th largest. Digits start below the bits every key
// shares, so that clustered keys still spread over the bins.
template <int NT, class Bar = BlockBar, class Key>
__device__ uint32_t select_bound(int n, Key key, uint32_t k, int ndig, Scratch& s) {
  const int lowbit = 32 - 8 * ndig;
  const int tid = threadIdx.x;
  if (n < (int)k || k == 0) return 0u;
  uint32_t ka, ko;
  block_and_or<NT, Bar>(n, [&](int i, uint32_t& v) { v = key(i); return true; }, s, ka, ko);
  const uint32_t diff = ka ^ ko;
  const uint32_t lowmask = (lowbit >= 32) ? 0xFFFFFFFFu : ((1u << lowbit) - 1u);
  if ((diff & ~lowmask) == 0u) return ka & ~lowmask;  // every key the same above lowbit
  const int h = 31 - __clz(diff & ~lowmask);
  uint32_t mask = (h >= 31) ? 0u : ~((2u << h) - 1u);
  uint32_t prefix = ka & mask;
  uint64_t above = 0;
  int sh = h - 7;
  for (;;) {
    if (sh < lowbit) sh = lowbit;
    for (int i = tid; i < 256; i += NT) s.cnt[i] = 0;
    Bar::sync();
    for (int i = tid; i < n; i += NT) {
      const uint32_t v = key(i);
      if ((v & mask) == prefix) atomicAdd(&s.cnt[(v >> sh) & 255u], 1u);
    }
    Bar::sync();
    if (tid < 32) find_bin(s, above, k, [&](int b) { return (unsigned long long)s.cnt[b]; });
    Bar::sync();
    const int bin = s.bin;
    const uint64_t ab = s.above;
    Bar::sync();
    if (bin < 0) return prefix;  // fewer than k items in the group: keep it whole
    prefix |= (uint32_t)bin << sh;
    mask |= 255u << sh;
    above = ab;
    if (sh == lowbit) break;
    sh -= 8;
  }
  return prefix;
}

// radix() over composite keys (32-bit value key << 24 | 24-bit reversed id) whose value
// digits start below the bits that all eligible items share, down to value bit
// `lowvbit` (16 when the values are widened bf16, whose low key bits follow from the
// high ones), then the three id digits.
template <int NT, bool MASS, class Bar = BlockBar, int kU = 1, class Item, class WFn>
__device__ uint64_t radix_adaptive(int n, Item item, uint64_t lo_key, uint64_t target, WFn wfn,
                                   int lowvbit, Scratch& s, uint64_t* group_max = nullptr,
                                   bool* beyond = nullptr) {
  uint32_t ka, ko;
  block_and_or<NT, Bar, kU>(
      n,
      [&](int i, uint32_t& v) {
        const uint64_t c = item(i);
        v = (uint32_t)(c >> 24);
        return c >= lo_key;
      },
      s, ka, ko);
  int shifts[8];
  int ns = 0;
  const uint32_t lowmask = (1u << lowvbit) - 1u;
  const uint32_t diff = (ka ^ ko) & ~lowmask;
  if (ka <= ko && diff != 0u) {
    const int h = 31 - __clz(diff);
    for (int sh = h - 7;; sh -= 8) {
      shifts[ns++] = 24 + (sh < lowvbit ? lowvbit : sh);
      if (sh <= lowvbit) break;
    }
  }
  shifts[ns++] = 16;
  shifts[ns++] = 8;
  shifts[ns++] = 0;
  return radix<NT, MASS, Bar, kU>(n, item, lo_key, target, wfn, shifts, ns, s, group_max, beyond);
}

}  // namespace sel
}  // namespace tsv
