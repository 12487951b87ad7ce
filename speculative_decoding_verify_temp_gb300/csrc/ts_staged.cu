// Cluster-staged row kernels: one thread-block cluster per row. Each CTA of the cluster
// copies its slice of the row into shared memory with 1-D TMA bulk copies (one HBM read
// of the row); every later pass runs over shared memory, and the CTAs exchange partial
// results through distributed shared memory (DSMEM).
//
// Modes
//  kSoftmax  probs = softmax(x / T) per row (TokenSpeed flashinfer.py verify(): softmax)
//  kRenorm   top-k then top-p renorm of probability rows (verify(): fused_topk_topp_renorm)
//  kChain    target-only chain speculative sampling from logits with per-request T, top-k,
//            top-p (verify(): softmax + fused renorm + chain_speculative_sampling_target_only):
//            every row computes its filtered distribution p'', the accept test of its draft
//            (u_j < p''_j(x_j)) and, speculatively, its final draw (the residual p''_j without
//            x_j, or the bonus p''_D) with u_D; the last row of a request to finish writes
//            the chain.
//
// Order and thresholds. "Value descending, then token id ascending" is the order of 56-bit
// composite keys (an order-preserving image of the value above 2^24 - 1 - id). Top-k keeps
// the k largest composites and top-p a prefix of them, so every filter ends as one
// threshold: a token is kept iff its composite >= C. The thresholds are found without
// sorting the row:
//  - top-k: the k-th largest of the per-thread maxima (gathered over the cluster) bounds
//    the k-th largest element from below; one sweep compacts the few elements above the
//    bound, and every CTA sorts the gathered candidates (bitonic, in shared memory);
//  - top-p without top-k: a 512-bucket histogram of the weights (sixteenths of an octave
//    below the row maximum) locates the bucket where the ordered mass crosses top_p; only
//    that bucket's elements are compacted and sorted.
// If a candidate list would overflow, the row takes a general path: a cluster-wide radix
// selection over the staged slice (slower, same result).
//
// Exactness. Weights are fixed-point integers w = floor(e * 2^40) of the fp32 weight e =
// 2^(-(M - x) * log2(e) / T), so the masses that decide the thresholds are exact integer
// sums and the result is deterministic. The draw walks token ids in order: each thread
// owns a contiguous range, sums its weights in fp32 (a fixed order), and the thread
// totals, taken to fixed point, are combined exactly.
#include <stdint.h>

#include "ts_common.cuh"
#include "ts_internal.h"

namespace tsv {

static __device__ unsigned int g_staged_err;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunks = 4;
constexpr int kMaxCluster = 8;
constexpr uint32_t kWaitLimit = 1u << 26;
constexpr int64_t kSliceTarget = 50 * 1024;  // bytes of row per CTA we aim for
constexpr int64_t kSliceMax = 160 * 1024;    // bytes of row per CTA we accept
constexpr int kGatherCap = 4096;             // candidates of a row (held by CTA 0)
constexpr int kNBins = 512;                  // top-p weight buckets
constexpr float kBinScale = 16.f;            // buckets per octave
constexpr int kHistBins = 384;               // buckets over 24 octaves; the rest is the tail
static_assert(kNBins == kThreads, "the bucket scan gives one bucket to each thread");

struct RowCtl {
  // read by peer CTAs through DSMEM
  float p_max;
  int32_t p_am;
  float p_lm;
  float p_ls;
  uint64_t p_sum;
  uint32_t gcount;  // CTA 0: candidates appended by the cluster
  uint32_t lcnt;    // candidates collected by this CTA
  uint32_t lbase;   // their place in CTA 0's list
  int32_t p_tok;
  int32_t b_ok;     // written by CTA 0: the selection result
  int32_t b_pad;
  uint64_t b_C;
  uint64_t b_Zk;
  // radix mass histograms as three 32-bit digit sums (14, 14 and 13 bits of each
  // weight), double-buffered; the top-p buckets use them as [3][512]
  uint32_t m3[2][3][256];
  uint32_t cnt[2][256];
  // local
  unsigned long long tot_mass[256];
  uint32_t tot_cnt[256];
  uint64_t bar[kChunks];
  uint64_t scan[kWarps];
  float red_f[3][kWarps];
  int32_t red_i[kWarps];
  float M, S1;
  int32_t am;
  int32_t bin;
  int32_t bincnt;
  int32_t found;
  uint64_t above;
  uint64_t target;
  uint64_t Z;
  uint64_t C;
  uint64_t aux;
  int32_t tok;
  int32_t round;
  float uj, uD, vx;  // this row's coins and its draft token's value
};

// Exact accumulation of weights below 2^42 with 32-bit shared-memory atomics: the
// weight is split into 14-, 14- and 13-bit digits, each summed on its own counter
// (no overflow for fewer than 2^18 additions per counter).
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

template <typename E>
struct SV;
template <>
struct SV<float> {
  static constexpr int N = 4;  // elements per 16-byte vector
  __device__ __forceinline__ static float get(const float* s, int64_t i) { return s[i]; }
  __device__ __forceinline__ static float vmax(const float* s, int64_t i) {
    const float4 r = *reinterpret_cast<const float4*>(s + i);
    return fmaxf(fmaxf(r.x, r.y), fmaxf(r.z, r.w));
  }
  __device__ __forceinline__ static void vec(const float* s, int64_t i, float* x) {
    const float4 r = *reinterpret_cast<const float4*>(s + i);
    x[0] = r.x;
    x[1] = r.y;
    x[2] = r.z;
    x[3] = r.w;
  }
};
template <>
struct SV<uint16_t> {
  static constexpr int N = 8;
  __device__ __forceinline__ static float get(const uint16_t* s, int64_t i) {
    return bf16_bits_to_f32(s[i]);
  }
  // the largest of 8 bf16 values with packed bf16x2 maxima
  __device__ __forceinline__ static uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  __device__ __forceinline__ static float vmax(const uint16_t* s, int64_t i) {
    const uint4 r = *reinterpret_cast<const uint4*>(s + i);
    const uint32_t m = bmax2(bmax2(r.x, r.y), bmax2(r.z, r.w));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  __device__ __forceinline__ static void vec(const uint16_t* s, int64_t i, float* x) {
    const uint4 r = *reinterpret_cast<const uint4*>(s + i);
    x[0] = __uint_as_float(r.x << 16);
    x[1] = __uint_as_float(r.x & 0xFFFF0000u);
    x[2] = __uint_as_float(r.y << 16);
    x[3] = __uint_as_float(r.y & 0xFFFF0000u);
    x[4] = __uint_as_float(r.z << 16);
    x[5] = __uint_as_float(r.z & 0xFFFF0000u);
    x[6] = __uint_as_float(r.w << 16);
    x[7] = __uint_as_float(r.w & 0xFFFF0000u);
  }
};

// inverse of fkey
__device__ __forceinline__ float key_to_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ uint32_t comp_idx(uint64_t c) {
  return kIdxMax - (uint32_t)(c & kIdxMax);
}

struct RadixOut {
  uint64_t prefix, mask, above;
  int keep_all;
};

// Cluster-wide radix selection over 64-bit composite keys (the general path).
//   count mode: finds the group of the `target`-th largest key;
//   mass mode:  finds the element at which the mass, accumulated in descending key
//               order, first reaches `target` (or ceil(top_p * total) when top_p >= 0).
// An element is selected iff (key & mask) >= prefix. `sweep(f)` must call f(key, v) for
// every eligible element of this CTA; wfn(v) gives its weight (mass mode).
template <bool MASS, class Sweep, class WFn>
__device__ RadixOut cluster_radix(RowCtl* ctl, cg::cluster_group& cluster, uint32_t CL,
                                  Sweep sweep, WFn wfn, const int* shifts, int nsh,
                                  uint64_t target, float top_p) {
  RadixOut o{0, 0, 0, 0};
  const int tid = threadIdx.x;
  for (int di = 0; di < nsh; ++di) {
    const int sh = shifts[di];
    const int buf = ctl->round & 1;
    for (int i = tid; i < 256; i += kThreads) {
      ctl->m3[buf][0][i] = 0;
      ctl->m3[buf][1][i] = 0;
      ctl->m3[buf][2][i] = 0;
      ctl->cnt[buf][i] = 0;
    }
    __syncthreads();
    const uint64_t pre = o.prefix, msk = o.mask;
    sweep([&](uint64_t key, float v) {
      if ((key & msk) == pre) {
        const int bin = (int)((key >> sh) & 255u);
        atomicAdd(&ctl->cnt[buf][bin], 1u);
        if (MASS)
          add3(&ctl->m3[buf][0][bin], &ctl->m3[buf][1][bin], &ctl->m3[buf][2][bin], wfn(v));
      }
    });
    __syncthreads();
    cluster.sync();
    if (tid < 256) {
      unsigned long long tm = 0;
      uint32_t tc = 0;
      for (uint32_t c = 0; c < CL; ++c) {
        RowCtl* pc = cluster.map_shared_rank(ctl, c);
        tm += get3(pc->m3[buf][0][tid], pc->m3[buf][1][tid], pc->m3[buf][2][tid]);
        tc += pc->cnt[buf][tid];
      }
      ctl->tot_mass[tid] = tm;
      ctl->tot_cnt[tid] = tc;
    }
    __syncthreads();
    if (tid < 32) {
      const int lane = tid;
      if (di == 0 && MASS && top_p >= 0.f) {
        unsigned long long tot = 0;
        for (int k = lane; k < 256; k += 32) tot += ctl->tot_mass[k];
        tot = warp_sum_u64(tot);
        if (lane == 0) {
          const double want = ceil((double)top_p * (double)tot);
          ctl->target = (want > (double)tot) ? (uint64_t)tot + 1 : (uint64_t)want;
        }
        __syncwarp();
      }
      const uint64_t tgt = (MASS && top_p >= 0.f) ? ctl->target : target;
      // lane l owns bins 255-8l .. 248-8l (descending)
      unsigned long long lw = 0;
      for (int k = 0; k < 8; ++k) {
        const int bin = 255 - 8 * lane - k;
        lw += MASS ? ctl->tot_mass[bin] : (unsigned long long)ctl->tot_cnt[bin];
      }
      unsigned long long incl = lw;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      unsigned long long acc = o.above + (incl - lw);
      int found = -1;
      unsigned long long acc_at = 0;
      for (int k = 0; k < 8; ++k) {
        const int bin = 255 - 8 * lane - k;
        const uint32_t c = ctl->tot_cnt[bin];
        const unsigned long long wgt = MASS ? ctl->tot_mass[bin] : (unsigned long long)c;
        if (c > 0 && acc + wgt >= tgt) {
          found = bin;
          acc_at = acc;
          break;
        }
        acc += wgt;
      }
      const unsigned m = __ballot_sync(0xffffffffu, found >= 0);
      if (m == 0) {
        if (lane == 0) ctl->bin = -1;
      } else if (lane == __ffs(m) - 1) {
        ctl->bin = found;
        ctl->above = acc_at;
        ctl->bincnt = (int32_t)ctl->tot_cnt[found];
      }
      if (lane == 0) ctl->round = ctl->round + 1;
    }
    __syncthreads();
    const int bin = ctl->bin;
    const uint64_t tgt = (MASS && top_p >= 0.f) ? ctl->target : target;
    if (bin < 0) {  // the target lies beyond the total: everything eligible is selected
      o.keep_all = 1;
      break;
    }
    o.prefix |= (uint64_t)bin << sh;
    o.mask |= (uint64_t)255u << sh;
    o.above = ctl->above;
    const int bc = ctl->bincnt;
    __syncthreads();
    if (!MASS && o.above + (uint64_t)bc == tgt) break;
    if (MASS && bc == 1) break;
  }
  return o;
}

__device__ __forceinline__ bool selected(const RadixOut& o, uint64_t key) {
  return o.keep_all || (key & o.mask) >= o.prefix;
}

// Exclusive scan of a u64 over the block (fixed order); returns the exclusive prefix and
// writes the block total.
__device__ __forceinline__ uint64_t block_excl_scan_u64(uint64_t v, RowCtl* ctl, uint64_t& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ctl->scan[w] = incl;
  __syncthreads();
  if (w == 0) {
    uint64_t t = lane < kWarps ? ctl->scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kWarps) ctl->scan[lane] = t;
  }
  __syncthreads();
  const uint64_t before = (w > 0) ? ctl->scan[w - 1] : 0;
  total = ctl->scan[kWarps - 1];
  __syncthreads();
  return before + incl - v;
}

// The largest C made of whole top digits such that at least k of a[0..n) are >= C: a
// lower bound for the k-th largest, exact in the digits examined. CTA-local.
__device__ uint32_t cta_select_bound(const uint32_t* a, int n, uint32_t k, int ndig, RowCtl* ctl) {
  uint32_t prefix = 0, mask = 0, above = 0;
  const int tid = threadIdx.x;
  for (int di = 0; di < ndig; ++di) {
    const int sh = 24 - 8 * di;
    if (tid < 256) ctl->cnt[0][tid] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t v = a[i];
      if ((v & mask) == prefix) atomicAdd(&ctl->cnt[0][(v >> sh) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      const int lane = tid;
      uint32_t lw = 0;
      for (int q = 0; q < 8; ++q) lw += ctl->cnt[0][255 - 8 * lane - q];
      uint32_t incl = lw;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      uint32_t acc = above + (incl - lw);
      int found = -1;
      uint32_t acc_at = 0;
      for (int q = 0; q < 8; ++q) {
        const int bin = 255 - 8 * lane - q;
        const uint32_t c = ctl->cnt[0][bin];
        if (c > 0 && acc + c >= k) {
          found = bin;
          acc_at = acc;
          break;
        }
        acc += c;
      }
      const unsigned m = __ballot_sync(0xffffffffu, found >= 0);
      if (m == 0) {
        if (lane == 0) {  // fewer than k items remain: the bound keeps the whole group
          ctl->bin = 0;
          ctl->above = above;
        }
      } else if (lane == __ffs(m) - 1) {
        ctl->bin = found;
        ctl->above = acc_at;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)ctl->bin << sh;
    mask |= 255u << sh;
    above = (uint32_t)ctl->above;
    __syncthreads();
  }
  return prefix;
}

// CTA-local radix selection over the items of a[0..n) that are >= lo_key, in descending
// order: count mode finds the set of the `target` largest, mass mode the shortest top set
// whose mass (wfn of each item) reaches `target`. Returns the smallest item of that set,
// so an item is selected iff it is >= the result (all eligible items if the target lies
// beyond their total).
template <bool MASS, class WFn>
__device__ uint64_t cta_radix(const uint64_t* a, int n, uint64_t lo_key, uint64_t target, WFn wfn,
                              const int* shifts, int nsh, RowCtl* ctl, uint64_t* group_max = nullptr,
                              bool* beyond = nullptr) {
  uint64_t prefix = 0, mask = 0, above = 0;
  const int tid = threadIdx.x;
  bool all = false;
  for (int di = 0; di < nsh; ++di) {
    const int sh = shifts[di];
    if (tid < 256) {
      ctl->m3[0][0][tid] = 0;
      ctl->m3[0][1][tid] = 0;
      ctl->m3[0][2][tid] = 0;
      ctl->cnt[0][tid] = 0;
    }
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint64_t v = a[i];
      if (v >= lo_key && (v & mask) == prefix) {
        const int b = (int)((v >> sh) & 255u);
        atomicAdd(&ctl->cnt[0][b], 1u);
        if (MASS) add3(&ctl->m3[0][0][b], &ctl->m3[0][1][b], &ctl->m3[0][2][b], wfn(v));
      }
    }
    __syncthreads();
    if (tid < 32) {
      const int lane = tid;
      unsigned long long lw = 0;
      for (int q = 0; q < 8; ++q) {
        const int bin = 255 - 8 * lane - q;
        lw += MASS ? get3(ctl->m3[0][0][bin], ctl->m3[0][1][bin], ctl->m3[0][2][bin])
                   : (unsigned long long)ctl->cnt[0][bin];
      }
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
        const uint32_t c = ctl->cnt[0][bin];
        const unsigned long long wgt =
            MASS ? get3(ctl->m3[0][0][bin], ctl->m3[0][1][bin], ctl->m3[0][2][bin])
                 : (unsigned long long)c;
        if (c > 0 && acc + wgt >= target) {
          found = bin;
          acc_at = acc;
          break;
        }
        acc += wgt;
      }
      const unsigned m = __ballot_sync(0xffffffffu, found >= 0);
      if (m == 0) {
        if (lane == 0) ctl->bin = -1;
      } else if (lane == __ffs(m) - 1) {
        ctl->bin = found;
        ctl->above = acc_at;
        ctl->bincnt = (int32_t)ctl->cnt[0][found];
      }
    }
    __syncthreads();
    const int bin = ctl->bin;
    const uint64_t ab = ctl->above;
    const int bc = ctl->bincnt;
    __syncthreads();
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
  // the smallest selected item, and the largest item of the final group
  unsigned long long mn = ~0ull, gx = 0;
  for (int i = tid; i < n; i += kThreads) {
    const uint64_t v = a[i];
    if (v >= lo_key && (all || (v & mask) >= prefix) && v < mn) mn = v;
    if (v >= lo_key && !all && (v & mask) == prefix && v > gx) gx = v;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, mn, off);
    mn = y < mn ? y : mn;
    const unsigned long long z = __shfl_xor_sync(0xffffffffu, gx, off);
    gx = z > gx ? z : gx;
  }
  if (tid == 0) {
    ctl->aux = ~0ull;
    ctl->Z = 0;
  }
  __syncthreads();
  if ((tid & 31) == 0) {
    atomicMin(reinterpret_cast<unsigned long long*>(&ctl->aux), mn);
    atomicMax(reinterpret_cast<unsigned long long*>(&ctl->Z), gx);
  }
  __syncthreads();
  const uint64_t r = ctl->aux;
  if (group_max) *group_max = ctl->Z;
  __syncthreads();
  return r;
}

__device__ __forceinline__ int next_pow2(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

template <typename E>
__global__ void __launch_bounds__(kThreads, 2) k_staged(StagedArgs a, int64_t slice_n, int vec) {
  extern __shared__ __align__(128) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t crank = cluster.block_rank();
  const uint32_t CL = cluster.num_blocks();
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x / CL;
  constexpr int NV = SV<E>::N;
  E* sv = reinterpret_cast<E*>(smem);
  const int64_t sv_bytes = (slice_n * (int64_t)sizeof(E) + 127) & ~(int64_t)127;
  RowCtl* ctl = reinterpret_cast<RowCtl*>(smem + sv_bytes);
  uint64_t* gbuf =
      reinterpret_cast<uint64_t*>(smem + sv_bytes + ((sizeof(RowCtl) + 127) & ~(size_t)127));
  uint32_t* tmk = reinterpret_cast<uint32_t*>(gbuf + kGatherCap);  // this CTA's thread maxima
  uint32_t* tmall = tmk + kThreads;                                  // the cluster's
  const int64_t lo = (int64_t)crank * slice_n;
  const int64_t n = max((int64_t)0, min(slice_n, a.V - lo));
  const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;

  // the request's temperature, its draft at this row, and the coins: read before the
  // slice lands, so their latency hides under the copy
  const int64_t req = (a.mode == kChain) ? row / a.R : row;
  const int32_t j = (a.mode == kChain) ? (int32_t)(row % a.R) : 0;
  float T = 1.f;
  if (a.mode != kRenorm && a.temperature) T = a.temperature[req];
  if (a.mode == kChain && a.skip_greedy && !(T >= kGreedyT)) return;  // a streaming pass has it
  const int32_t D = a.D;
  const int32_t x = (a.mode == kChain && j < D) ? a.draft_tokens[req * D + j] : -1;
  const bool xvalid = x >= 0 && (int64_t)x < a.V;
  if (a.mode == kChain) {
    if (tid == 0) {
      const uint64_t seed = a.seed ? (uint64_t)a.seed[req] : 0;
      const uint64_t off = a.offset ? (uint64_t)a.offset[req] : 0;
      ctl->uj = (j < D) ? (a.uniforms ? a.uniforms[req * a.R + j] : verify_coin(seed, off, (uint32_t)j))
                        : 0.f;
      ctl->uD = a.uniforms ? a.uniforms[req * a.R + D] : verify_coin(seed, off, (uint32_t)D);
      ctl->tok = -1;
    }
    if (tid == 32) {
      ctl->vx = !xvalid ? 0.f
                        : (sizeof(E) == 2 ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(xr)[x])
                                          : reinterpret_cast<const float*>(xr)[x]);
    }
  }

  // ---- 1. stage the slice ----------------------------------------------------------
  if (tid == 0) {
    ctl->round = 0;
    ctl->gcount = 0;
    ctl->lcnt = 0;
  }
  for (int i = tid; i < 3 * kNBins; i += kThreads) (&ctl->m3[0][0][0])[i] = 0;
  if (vec) {
    const int64_t bulk = (n * (int64_t)sizeof(E)) & ~(int64_t)15;
    const int64_t cb = ((bulk / kChunks) + 15) & ~(int64_t)15;
    if (tid == 0) {
      for (int c = 0; c < kChunks; ++c) mbar_init(&ctl->bar[c], 1);
      fence_mbar_init();
      for (int c = 0; c < kChunks; ++c) {
        const int64_t off = min(bulk, c * cb);
        const int64_t len = min(bulk, off + cb) - off;
        mbar_arrive_expect_tx(&ctl->bar[c], (uint32_t)len);
        if (len > 0)
          bulk_g2s(reinterpret_cast<unsigned char*>(sv) + off,
                   reinterpret_cast<const unsigned char*>(xr + lo) + off, (uint32_t)len,
                   &ctl->bar[c]);
      }
    }
    const int64_t tail0 = bulk / (int64_t)sizeof(E);
    for (int64_t i = tail0 + tid; i < n; i += kThreads) sv[i] = xr[lo + i];
    __syncthreads();
    for (int c = 0; c < kChunks; ++c) {
      uint32_t it = 0;
      while (!mbar_try_wait(&ctl->bar[c], 0)) {
        if (++it > kWaitLimit) {
          atomicOr(&g_staged_err, 1u);
          break;
        }
      }
    }
  } else {
    for (int64_t i = tid; i < n; i += kThreads) sv[i] = xr[lo + i];
  }
  // pad the slice to whole vectors with -inf (never kept, zero weight)
  const int64_t nvec = (n + NV - 1) / NV;
  if (tid < NV) {
    const int64_t i = n + tid;
    if (i < nvec * NV) {
      if (sizeof(E) == 2) reinterpret_cast<uint16_t*>(sv)[i] = 0xFF80u;
      else reinterpret_cast<float*>(sv)[i] = -INFINITY;
    }
  }
  __syncthreads();

  // ---- 2. row maximum, argmax (lowest id), thread maxima, temperature-1 log-sum-exp ----
  const bool want_lse = (a.mode == kChain) && a.logprobs != nullptr;
  float bv = -INFINITY, lm = -INFINITY, ls = 0.f, lc = 0.f;
  int32_t bi = INT32_MAX;
  for (int64_t vi = tid; vi < nvec; vi += kThreads) {
    const float vm = SV<E>::vmax(sv, vi * NV);
    if (vm > bv || bi == INT32_MAX) {
      float x[NV];
      SV<E>::vec(sv, vi * NV, x);
      for (int q = 0; q < NV; ++q)
        if (x[q] == vm) {
          bi = (int32_t)(lo + vi * NV + q);
          break;
        }
      bv = vm;
    }
    if (want_lse && vm > -INFINITY) {
      float x[NV];
      SV<E>::vec(sv, vi * NV, x);
      const float nm = fmaxf(lm, vm);
      const float f = ex2((lm - nm) * kLog2e);
      ls *= f;
      lc *= f;
      lm = nm;
      float vs = 0.f;
#pragma unroll
      for (int q = 0; q < NV; ++q) vs += ex2((x[q] - nm) * kLog2e);
      kahan_add(ls, lc, vs);
    }
  }
  ls += lc;
  // a padding element can be a thread's maximum only if the thread holds nothing else
  if (bi != INT32_MAX && (int64_t)bi >= lo + n) bi = INT32_MAX;
  // this thread's largest value as an order key (0 = the thread holds no element)
  tmk[tid] = (bi == INT32_MAX) ? 0u : fkey(bv);
  {
    float v = bv, m = lm, s = ls;
    int32_t i = bi;
    warp_argmax(v, i);
    warp_lse(m, s);
    const int lane = tid & 31, w = tid >> 5;
    if (lane == 0) {
      ctl->red_f[0][w] = v;
      ctl->red_f[1][w] = m;
      ctl->red_f[2][w] = s;
      ctl->red_i[w] = i;
    }
    __syncthreads();
    if (w == 0) {
      v = lane < kWarps ? ctl->red_f[0][lane] : -INFINITY;
      m = lane < kWarps ? ctl->red_f[1][lane] : -INFINITY;
      s = lane < kWarps ? ctl->red_f[2][lane] : 0.f;
      i = lane < kWarps ? ctl->red_i[lane] : INT32_MAX;
      warp_argmax(v, i);
      warp_lse(m, s);
      if (lane == 0) {
        ctl->p_max = v;
        ctl->p_am = i;
        ctl->p_lm = m;
        ctl->p_ls = s;
      }
    }
  }
  cluster.sync();  // (1) partial statistics and thread maxima are visible
  if (tid < 32) {
    const int lane = tid;
    float v = -INFINITY, m = -INFINITY, s = 0.f;
    int32_t i = INT32_MAX;
    if ((uint32_t)lane < CL) {
      RowCtl* pc = cluster.map_shared_rank(ctl, (uint32_t)lane);
      v = pc->p_max;
      i = pc->p_am;
      m = pc->p_lm;
      s = pc->p_ls;
    }
    warp_argmax(v, i);
    warp_lse(m, s);
    if (lane == 0) {
      ctl->M = v;
      ctl->am = (i == INT32_MAX) ? 0 : i;
      ctl->S1 = s;
    }
  }
  __syncthreads();
  const float M = ctl->M;
  const int32_t am = ctl->am;

  // ---- 3. knobs ------------------------------------------------------------------------
  float tp = 1.f;
  int32_t k = 0;
  if (a.mode != kSoftmax) {
    if (a.top_k) k = a.top_k[req];
    if (a.top_p) tp = a.top_p[req];
  }
  const bool is_logits = (a.mode != kRenorm);
  const bool greedy = is_logits && !(T >= kGreedyT);
  const bool tk = !greedy && k > 0 && (int64_t)k < a.V;
  const bool tpa = !greedy && tp < 1.f;
  const float sl2 = is_logits ? __fdiv_rn(kLog2e, T) : 0.f;
  const uint32_t pmax_bits = __float_as_uint(fmaxf(M, 0.f));
  const bool bf16 = sizeof(E) == 2;

  // The weight of a value: e = 2^(-(M - x) log2(e)/T) (logits) or the value (probabilities).
  auto dfn = [&](float v) -> float { return (M - v) * sl2; };
  auto efn = [&](float v) -> float {
    return is_logits ? ex2(-dfn(v)) : fminf(fmaxf(v, 0.f), 1.f);
  };
  auto wfn = [&](float v) -> uint64_t { return fixw(efn(v)); };
  // the top-p bucket of a value, 0 = heaviest (sixteenths of an octave below the maximum)
  auto bin512 = [&](float v) -> int {
    if (is_logits) {
      const float t = __fadd_rd(fminf(dfn(v) * kBinScale, 1.0e6f), 8388608.f);
      return (int)min(__float_as_uint(t) - 0x4B000000u, (uint32_t)(kNBins - 1));
    }
    const uint32_t vb = __float_as_uint(fmaxf(v, 0.f));
    return (vb == 0u) ? (kNBins - 1) : (int)min((pmax_bits - vb) >> 19, (uint32_t)(kNBins - 1));
  };

  // Decided below, identically in every CTA of the cluster. fast: a token is kept iff its
  // composite >= C (C = 0 keeps everything), and Zk is the exact mass of the kept set
  // when a selection found it.
  bool fast = true;
  uint64_t C = 0;
  uint64_t Zk = 0;

  // Every CTA appends its candidates to CTA 0's list; after a cluster barrier CTA 0 sorts
  // them, finds the threshold and writes it to every CTA; a second barrier publishes it.
  // Candidates are first collected in this CTA (in the space of the gathered thread
  // maxima, free by then), then copied to CTA 0 in one block after one reservation.
  uint32_t* g0count = cluster.map_shared_rank(&ctl->gcount, 0);
  uint64_t* g0buf = cluster.map_shared_rank(gbuf, 0);
  uint64_t* llist = reinterpret_cast<uint64_t*>(tmall);
  constexpr int kLocalCap = kMaxCluster * kThreads / 2;
  auto append = [&](uint64_t cp) {
    const uint32_t pos = atomicAdd(&ctl->lcnt, 1u);
    if (pos < (uint32_t)kLocalCap) llist[pos] = cp;
  };
  auto ship = [&]() {  // after a __syncthreads that follows the appends
    if (tid == 0) {
      const uint32_t nl = ctl->lcnt;
      // an overflowing list reserves past the capacity, so CTA 0 sees the overflow
      ctl->lbase = atomicAdd(g0count, nl > (uint32_t)kLocalCap ? (uint32_t)kGatherCap + 1u : nl);
    }
    __syncthreads();
    const uint32_t nl = min(ctl->lcnt, (uint32_t)kLocalCap), base = ctl->lbase;
    for (uint32_t i = tid; i < nl; i += kThreads)
      if (base + i < (uint32_t)kGatherCap) g0buf[base + i] = llist[i];
  };
  // topk: the k largest candidates, then top-p inside them; else the candidates are one
  // weight bucket whose ordered mass starts at `base` and must reach P
  const int cs_f[7] = {48, 40, 32, 24, 16, 8, 0};
  const int cs_h[5] = {48, 40, 16, 8, 0};
  const int* cs = bf16 ? cs_h : cs_f;
  const int ncs = bf16 ? 5 : 7;
  auto wcomp = [&](uint64_t c) -> uint64_t { return wfn(key_to_f32((uint32_t)(c >> kIdxBits))); };
  // the exact mass of the candidates >= c0
  auto mass_from = [&](int cnt, uint64_t c0) -> uint64_t {
    uint64_t s = 0;
    for (int i = tid; i < cnt; i += kThreads)
      if (gbuf[i] >= c0) s += wcomp(gbuf[i]);
    uint64_t tot;
    (void)block_excl_scan_u64(s, ctl, tot);
    return tot;
  };
  // CTA 0: the threshold and the kept mass from its candidate list
  auto select_local = [&](bool topk, uint64_t base, uint64_t P, bool& ok, uint64_t& Cb,
                          uint64_t& Zb) {
      const uint32_t total = ctl->gcount;
      ok = total <= (uint32_t)kGatherCap && total > 0 && (!topk || total >= (uint32_t)k);
      Cb = 0;
      Zb = 0;
      if (ok) {
        const int cnt = (int)total;
        if (topk) {
          Cb = cta_radix<false>(gbuf, cnt, 0, (uint64_t)k, wcomp, cs, ncs, ctl);
          Zb = mass_from(cnt, Cb);
          if (tpa) {
            const double want = ceil((double)tp * (double)Zb);
            const uint64_t Pk = (want > (double)Zb) ? Zb : (uint64_t)want;
            Cb = cta_radix<true>(gbuf, cnt, Cb, Pk, wcomp, cs, ncs, ctl);
            Zb = mass_from(cnt, Cb);
          }
        } else {
          Cb = cta_radix<true>(gbuf, cnt, 0, P - base, wcomp, cs, ncs, ctl);
          Zb = base + mass_from(cnt, Cb);
        }
      }
  };
  auto select_and_broadcast = [&](bool topk, uint64_t base, uint64_t P) {
    if (crank == 0) {
      bool ok;
      uint64_t Cb, Zb;
      select_local(topk, base, P, ok, Cb, Zb);
      if (tid < (int)CL) {
        RowCtl* pc = cluster.map_shared_rank(ctl, (uint32_t)tid);
        pc->b_ok = ok ? 1 : 0;
        pc->b_C = Cb;
        pc->b_Zk = Zb;
      }
    }
    cluster.sync();  // the selection result is visible
    fast = ctl->b_ok != 0;
    C = ctl->b_C;
    Zk = ctl->b_Zk;
  };

  if (!greedy && a.mode != kSoftmax && (tk || tpa)) {
    if (tk && (int64_t)k <= (int64_t)CL * kThreads) {
      // ---- 4a. top-k: bound from the gathered thread maxima, compaction, selection -----
      for (int i = tid; i < (int)CL * kThreads; i += kThreads)
        tmall[i] = cluster.map_shared_rank(tmk, (uint32_t)(i / kThreads))[i % kThreads];
      __syncthreads();
      const uint32_t tkey = cta_select_bound(tmall, (int)CL * kThreads, (uint32_t)k, bf16 ? 2 : 4, ctl);
      for (int64_t vi = tid; vi < nvec; vi += kThreads) {
        if (fkey(SV<E>::vmax(sv, vi * NV)) < tkey) continue;
        float xv[NV];
        SV<E>::vec(sv, vi * NV, xv);
        for (int q = 0; q < NV; ++q) {
          const int64_t li = vi * NV + q;
          if (li >= n) break;
          const uint32_t kq = fkey(xv[q]);
          if (kq >= tkey) append(comp_key(kq, (uint32_t)(lo + li)));
        }
      }
      __syncthreads();
      ship();
      __syncthreads();
      cluster.sync();  // (2) the candidates are in CTA 0
      if (a.mode == kChain) {
        // CTA 0 selects and draws alone; the other CTAs are done (nothing reads their
        // shared memory any more) unless the list overflowed
        const uint32_t total0 = *g0count;
        if (!(total0 > 0 && total0 <= (uint32_t)kGatherCap && total0 >= (uint32_t)k)) {
          fast = false;
        } else if (crank != 0) {
          return;
        } else {
          bool ok;
          select_local(true, 0, 0, ok, C, Zk);
        }
      } else {
        select_and_broadcast(true, 0, 0);  // (3)
      }
    } else if (!tk) {
      // ---- 4b. top-p over the whole row: bucket histogram, then the crossing bucket ------
      uint64_t tail = 0;
      uint32_t* h3 = &ctl->m3[0][0][0];  // [3][kNBins]
      for (int64_t vi = tid; vi < nvec; vi += kThreads) {
        float xv[NV];
        SV<E>::vec(sv, vi * NV, xv);
#pragma unroll
        for (int q = 0; q < NV; ++q) {
          const uint64_t w = wfn(xv[q]);
          if (w == 0) continue;
          const int b = bin512(xv[q]);
          if (b < kHistBins) add3(h3 + b, h3 + kNBins + b, h3 + 2 * kNBins + b, w);
          else tail += w;  // lighter than 2^-24 of the maximum: the tail bucket
        }
      }
      tail = warp_sum_u64(tail);
      if ((tid & 31) == 0 && tail)
        add3(h3 + kNBins - 1, h3 + 2 * kNBins - 1, h3 + 3 * kNBins - 1, tail);
      __syncthreads();
      cluster.sync();  // (2) bucket histograms are visible
      // every CTA: the cluster histogram (one bucket per thread), the total, the crossing
      uint64_t hb = 0;
      for (uint32_t c = 0; c < CL; ++c) {
        const uint32_t* ph = cluster.map_shared_rank(&ctl->m3[0][0][0], c);
        hb += get3(ph[tid], ph[kNBins + tid], ph[2 * kNBins + tid]);
      }
      uint64_t Zt;
      const uint64_t ex = block_excl_scan_u64(hb, ctl, Zt);  // heaviest bucket first
      const double want = ceil((double)tp * (double)Zt);
      const uint64_t P = (want > (double)Zt) ? Zt : (uint64_t)want;
      if (tid == 0) ctl->bin = (P == 0) ? -2 : -1;
      __syncthreads();
      if (P > 0 && hb > 0 && ex < P && ex + hb >= P) {
        ctl->bin = tid;
        ctl->above = ex;
      }
      __syncthreads();
      const int bstar = ctl->bin;
      const uint64_t acc0 = (bstar >= 0) ? ctl->above : 0;
      if (bstar == -2) {
        // top_p <= 0 keeps the argmax alone
        const float vam = (sizeof(E) == 2) ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(xr)[am])
                                           : reinterpret_cast<const float*>(xr)[am];
        C = comp_key(fkey(vam), (uint32_t)am);
        Zk = wfn(vam);
        cluster.sync();  // (3) every branch here passes the same barriers
        cluster.sync();  // (4)
      } else if (bstar < 0 || bstar >= kHistBins) {
        fast = false;  // the crossing lies in the tail bucket: general path
        cluster.sync();  // (3)
        cluster.sync();  // (4)
      } else {
        for (int64_t vi = tid; vi < nvec; vi += kThreads) {
          if (bin512(SV<E>::vmax(sv, vi * NV)) > bstar) continue;  // even its heaviest is lighter
          float xv[NV];
          SV<E>::vec(sv, vi * NV, xv);
          for (int q = 0; q < NV; ++q) {
            const int64_t li = vi * NV + q;
            if (li >= n) break;
            if (bin512(xv[q]) != bstar || wfn(xv[q]) == 0) continue;
            append(comp_key(fkey(xv[q]), (uint32_t)(lo + li)));
          }
        }
        __syncthreads();
        ship();
        __syncthreads();
        cluster.sync();  // (3) the candidates are in CTA 0
        select_and_broadcast(false, acc0, P);  // (4)
      }
    } else {
      fast = false;  // k larger than the thread-maxima bound can serve
    }
  }

  // ---- 5. general path (rare): cluster-wide radix selection over the staged slice -------
  RadixOut KT{0, 0, 0, 1}, KK{0, 0, 0, 1}, PP{0, 0, 0, 1};
  auto binkey = [&](float v) -> uint64_t {
    uint32_t b;
    if (is_logits) {
      b = (uint32_t)fminf(dfn(v) * 8.f, 255.f);
    } else {
      const uint32_t vb = __float_as_uint(fmaxf(v, 0.f));
      b = (vb == 0u) ? 255u : min(255u, (pmax_bits - vb) >> 20);
    }
    return (uint64_t)(255u - b) << 56;
  };
  if (!fast) {
    const int gk_f[7] = {48, 40, 32, 24, 16, 8, 0};
    const int gk_h[5] = {48, 40, 16, 8, 0};
    const int gp_f[8] = {56, 48, 40, 32, 24, 16, 8, 0};
    const int gp_h[6] = {56, 48, 40, 16, 8, 0};
    auto slice_sweep = [&](auto&& f) {
      for (int64_t i = tid; i < n; i += kThreads) {
        const float v = SV<E>::get(sv, i);
        f(comp_key(fkey(v), (uint32_t)(lo + i)), v);
      }
    };
    if (tk) {
      if ((int64_t)k <= (int64_t)CL * kThreads) {
        // thread maxima as (value, lowest id) composites: a bound on the k-th element
        const uint64_t tm = (tmk[tid] == 0u) ? 0ull : comp_key(tmk[tid], (uint32_t)bi);
        KT = cluster_radix<false>(
            ctl, cluster, CL,
            [&](auto&& f) {
              if (tm) f(tm, 0.f);
            },
            [](float) { return (uint64_t)1; }, bf16 ? gk_h : gk_f, bf16 ? 5 : 7, (uint64_t)k,
            -1.f);
      }
      KK = cluster_radix<false>(
          ctl, cluster, CL,
          [&](auto&& f) {
            slice_sweep([&](uint64_t key, float v) {
              if (selected(KT, key)) f(key, v);
            });
          },
          [](float) { return (uint64_t)1; }, bf16 ? gk_h : gk_f, bf16 ? 5 : 7, (uint64_t)k, -1.f);
    }
    if (tpa) {
      PP = cluster_radix<true>(
          ctl, cluster, CL,
          [&](auto&& f) {
            slice_sweep([&](uint64_t key, float v) {
              if (!tk || (selected(KT, key) && selected(KK, key))) f(binkey(v) | key, v);
            });
          },
          wfn, bf16 ? gp_h : gp_f, bf16 ? 6 : 8, 0, tp);
    }
  }
  // the kept predicate on a composite (and its value, for the general path's buckets)
  auto kept = [&](uint64_t key, float v) -> bool {
    if (fast) return key >= C;
    if (tk && !(selected(KT, key) && selected(KK, key))) return false;
    if (tpa && !selected(PP, binkey(v) | key)) return false;
    return true;
  };

  // ---- 6a. softmax and renorm outputs -----------------------------------------------------
  if (a.mode == kSoftmax || a.mode == kRenorm) {
    uint64_t Z = Zk;
    const bool have_z = fast && (tk || tpa) && Zk > 0;
    if (!have_z) {
      // the mass of the kept set by a sweep; thread sums of at most a few hundred
      // weights <= 1 stay below 2^49 in fixed point
      float s = 0.f;
      if (!greedy) {
        for (int64_t vi = tid; vi < nvec; vi += kThreads) {
          float xv[NV];
          SV<E>::vec(sv, vi * NV, xv);
#pragma unroll
          for (int q = 0; q < NV; ++q) {
            const int64_t li = vi * NV + q;
            if (a.mode == kSoftmax || kept(comp_key(fkey(xv[q]), (uint32_t)(lo + li)), xv[q]))
              s += efn(xv[q]);
          }
        }
      }
      uint64_t tot;
      (void)block_excl_scan_u64(fixw(s), ctl, tot);
      if (tid == 0) ctl->p_sum = tot;
      cluster.sync();
      Z = 0;
      for (uint32_t c = 0; c < CL; ++c) Z += cluster.map_shared_rank(ctl, c)->p_sum;
    }
    const float scale = (Z > 0) ? __fdiv_rn(kFx, __ull2float_rn(Z)) : 0.f;
    float* orow = a.out + row * a.V + lo;
    for (int64_t i = tid; i < n; i += kThreads) {
      const float v = SV<E>::get(sv, i);
      float o;
      if (greedy) o = (lo + i == am) ? 1.f : 0.f;
      else if (a.mode == kSoftmax) o = efn(v) * scale;
      else o = kept(comp_key(fkey(v), (uint32_t)(lo + i)), v) ? fmaxf(v, 0.f) * scale : 0.f;
      orow[i] = o;
    }
    cluster.sync();
    return;
  }

  // ---- 6b. chain: the accept test of this row's draft and this row's speculative draw ---
  // One thread records the row; the last row of a request to be recorded writes the chain.
  auto finish_row = [&](int32_t tok_f, int32_t acc_f) {
    a.ws.rowres[row] = RowRes{M, am, ctl->S1, tok_f, acc_f, {0, 0, 0}};
    __threadfence();
    const uint32_t prev = atomicAdd(&a.ws.reqcnt[req], 1u);
    if (prev != (uint32_t)a.R - 1) return;
    __threadfence();
    a.ws.reqcnt[req] = 0;
    int32_t js = D;
    for (int32_t jj = 0; jj < D; ++jj)
      if (!__ldcg(&a.ws.rowres[req * a.R + jj].acc)) {
        js = jj;
        break;
      }
    for (int32_t jj = 0; jj < a.R; ++jj) {
      const int64_t rj = req * a.R + jj;
      int32_t t = -1;
      if (jj < js) t = a.draft_tokens[req * D + jj];
      else if (jj == js) t = __ldcg(&a.ws.rowres[rj].tok);
      a.accepted_tokens[rj] = t;
      if (a.accept_index) a.accept_index[rj] = (jj <= js) ? (int32_t)rj : -1;
      if (a.logprobs) {
        float lp = 0.f;
        if (jj <= js && t >= 0 && (int64_t)t < a.V) {
          const E* xj = reinterpret_cast<const E*>(a.x) + rj * a.ld;
          const float vt = (sizeof(E) == 2) ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(xj)[t])
                                             : reinterpret_cast<const float*>(xj)[t];
          lp = (vt - __ldcg(&a.ws.rowres[rj].M)) - logf(__ldcg(&a.ws.rowres[rj].S));
        }
        a.logprobs[rj] = lp;
      }
    }
    a.accept_length[req] = js + 1;
  };
  const float uj = ctl->uj, uD = ctl->uD;
  int32_t acc = 0, tok = am;
  if (greedy) {
    acc = (j < D) && (x == am);
    cluster.sync();  // no CTA leaves while a peer may still read its statistics
    if (crank == 0 && tid == 0) finish_row(tok, acc);
    return;
  } else {
    // the draft token's weight
    uint64_t wx = 0;
    if (xvalid) {
      const float vx = ctl->vx;
      if (kept(comp_key(fkey(vx), (uint32_t)x), vx)) wx = wfn(vx);
    }
    if (fast && tk) {
      // the kept set is CTA 0's candidate list (>= C): CTA 0 draws from it, walking token
      // ids in order through a radix selection on the id digits
      if (crank == 0) {
        const int cnt = (int)ctl->gcount;
        const uint64_t Zf = Zk;  // the kept mass, the draft token included if kept
        if (j < D) acc = ((double)uj * (double)Zf < (double)wx) ? 1 : 0;
        const uint64_t Zr = Zf - wx;
        if (Zr == 0) {
          tok = (wx > 0) ? x : am;  // all the mass sits on the draft token
        } else {
          uint64_t t = (uint64_t)((double)uD * (double)Zr);
          if (t >= Zr) t = Zr - 1;  // rounding: the last token with mass
          auto wnx = [&](uint64_t c) -> uint64_t {
            return ((int32_t)comp_idx(c) == x) ? 0ull : wcomp(c);
          };
          const int idx_sh[3] = {16, 8, 0};
          uint64_t g = 0;
          (void)cta_radix<true>(gbuf, cnt, C, t + 1, wnx, idx_sh, 3, ctl, &g);
          tok = (int32_t)comp_idx(g);
        }
        if (tid == 0) finish_row(tok, acc);
      }
      return;
    } else {
      // token-id order over the slice: contiguous per-thread ranges of whole vectors
      const int64_t per = (nvec + kThreads - 1) / kThreads;
      const int64_t v0 = min(nvec, (int64_t)tid * per), v1 = min(nvec, v0 + per);
      const uint32_t ckey = (uint32_t)(C >> kIdxBits);
      const bool pretest = fast && C != 0;
      // the weight of element gi under a kept predicate (0 for the draft token)
      auto wsum = [&](auto&& keptf, float v, int64_t gi) -> float {
        if (gi == (int64_t)x) return 0.f;
        if (!keptf(comp_key(fkey(v), (uint32_t)gi), v)) return 0.f;
        return efn(v);
      };
      auto kfast = [&](uint64_t key, float) -> bool { return key >= C; };
      auto kall = [](uint64_t, float) -> bool { return true; };
      // the fp32 mass of this thread's range, in token-id order
      auto range_sum = [&](auto&& keptf) -> float {
        float acc_s = 0.f;
        for (int64_t vi = v0; vi < v1; ++vi) {
          // no element of the vector is kept if even its largest is below the threshold
          if (pretest && fkey(SV<E>::vmax(sv, vi * NV)) < ckey) continue;
          float xv[NV];
          SV<E>::vec(sv, vi * NV, xv);
#pragma unroll
          for (int q = 0; q < NV; ++q) acc_s += wsum(keptf, xv[q], lo + vi * NV + q);
        }
        return acc_s;
      };
      // the first element of this thread's range at which the running mass exceeds tf
      auto range_find = [&](auto&& keptf, float tf) -> int32_t {
        float accf = 0.f;
        int32_t found = -1, lastk = -1;
        for (int64_t vi = v0; vi < v1 && found < 0; ++vi) {
          if (pretest && fkey(SV<E>::vmax(sv, vi * NV)) < ckey) continue;
          float xv[NV];
          SV<E>::vec(sv, vi * NV, xv);
          for (int q = 0; q < NV; ++q) {
            const float w = wsum(keptf, xv[q], lo + vi * NV + q);
            if (w == 0.f) continue;
            lastk = (int32_t)(lo + vi * NV + q);
            accf += w;
            if (accf > tf) {
              found = lastk;
              break;
            }
          }
        }
        return found >= 0 ? found : lastk;
      };
      const float s = fast ? (C ? range_sum(kfast) : range_sum(kall)) : range_sum(kept);
      const uint64_t sfx = fixw(s);
      uint64_t ctot;
      const uint64_t texcl = block_excl_scan_u64(sfx, ctl, ctot);
      // CTA masses go through global memory, so that a CTA can leave without waiting for
      // its peers to read its shared memory
      uint64_t* cm = a.ws.cmass + row * 8;
      if (tid == 0) {
        cm[crank] = ctot;
        __threadfence();
      }
      cluster.sync();  // CTA masses are visible; past here no CTA reads another's smem
      uint64_t Zr = 0, cpre = 0;
      int last_nz = -1;
      for (uint32_t c = 0; c < CL; ++c) {
        const uint64_t pc = __ldcg(cm + c);
        if (c < crank) cpre += pc;
        if (pc > 0) last_nz = (int)c;
        Zr += pc;
      }
      const uint64_t Zf = Zr + wx;
      if (j < D) acc = ((double)uj * (double)Zf < (double)wx) ? 1 : 0;
      if (Zr == 0) {
        // all the mass sits on the draft token
        if (crank == 0 && tid == 0) finish_row((wx > 0) ? x : am, acc);
        return;
      }
      const uint64_t t = (uint64_t)((double)uD * (double)Zr);
      const bool past = (t >= Zr);
      const bool mine = past ? ((int)crank == last_nz) : (cpre <= t && t < cpre + ctot);
      if (!mine) return;
      const uint64_t tl = past ? 0 : t - cpre;
      const bool hit = past ? (sfx > 0 && texcl + sfx == ctot) : (texcl <= tl && tl < texcl + sfx);
      if (hit) {
        // the one thread whose range holds the target finishes the row
        const float tf = past ? INFINITY : (float)(tl - texcl) * (1.0f / kFx);
        const int32_t found =
            fast ? (C ? range_find(kfast, tf) : range_find(kall, tf)) : range_find(kept, tf);
        finish_row(found, acc);
      }
      return;
    }
  }
}

static size_t extra_smem() {
  return ((sizeof(RowCtl) + 127) & ~(size_t)127) + sizeof(uint64_t) * (size_t)kGatherCap +
         sizeof(uint32_t) * (size_t)(kThreads + kMaxCluster * kThreads);
}

static int64_t slice_elems(int64_t V, int esize, int* CL_out) {
  const int64_t bytes = V * esize;
  const int CL = (int)min((int64_t)kMaxCluster, max((int64_t)1, (bytes + kSliceTarget - 1) / kSliceTarget));
  // whole 16-element groups, so every slice starts 16-byte aligned and vectors never straddle
  const int64_t sl = ((V + CL - 1) / CL + 15) & ~(int64_t)15;
  *CL_out = CL;
  return sl;
}

int staged_max_vocab(int bf16) {
  const int esize = bf16 ? 2 : 4;
  return (int)((kSliceMax / esize) * kMaxCluster);
}

template <typename E>
static cudaError_t launch_t(const StagedArgs& a, cudaStream_t s, const char** why) {
  int CL = 1;
  const int64_t sl = slice_elems(a.V, (int)sizeof(E), &CL);
  if (sl * (int64_t)sizeof(E) > kSliceMax) {
    *why = "vocab too large for the cluster-staged kernel";
    return cudaErrorInvalidValue;
  }
  const size_t smem = (size_t)((sl * (int64_t)sizeof(E) + 127) & ~(int64_t)127) + extra_smem();
  cudaError_t e = cudaFuncSetAttribute(k_staged<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const uintptr_t base = reinterpret_cast<uintptr_t>(a.x);
  const int vec = (base % 16 == 0) && ((a.ld * (int64_t)sizeof(E)) % 16 == 0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.rows * CL));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_staged<E>, a, sl, vec);
}

cudaError_t launch_staged(const StagedArgs& a, cudaStream_t s, const char** why) {
  return a.bf16 ? launch_t<uint16_t>(a, s, why) : launch_t<float>(a, s, why);
}

cudaError_t staged_read_error(uint32_t* word, int clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_staged_err, sizeof(v));
  if (e != cudaSuccess) return e;
  *word = v;
  if (clear && v) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_staged_err, &z, sizeof(z));
  }
  return e;
}

}  // namespace tsv
