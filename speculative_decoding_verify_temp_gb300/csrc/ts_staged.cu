// Cluster-staged row kernels: one thread-block cluster per row. Each CTA of the cluster
// copies its slice of the row into shared memory with 1-D TMA bulk copies (one HBM read
// of the row), then all later passes (the max, the top-k and top-p thresholds, the
// normaliser, the draw) run over shared memory; cluster-wide sums and histograms are
// exchanged through distributed shared memory (DSMEM).
//
// Modes
//  kSoftmax  probs = softmax(x / T) per row (TokenSpeed flashinfer.py verify(): softmax)
//  kRenorm   top-k then top-p renorm of probability rows (verify(): fused_topk_topp_renorm)
//  kChain    target-only chain speculative sampling from logits with per-request T, top-k,
//            top-p (verify(): softmax + fused renorm + chain_speculative_sampling_target_only):
//            every row computes its filtered distribution p'', the accept test of its draft
//            (u_j < p''_j(x_j)) and, speculatively, its final draw (the residual p''_j without
//            x_j, or the bonus p''_D) from u_D; the last row of a request to finish writes the
//            chain.
//
// Exactness. Weights are fixed-point integers w = floor(e * 2^40) of the fp32 weight e
// (exp((x - M) / T) computed as 2^(-(M - x) * log2(e) / T)), so every sum is exact and the
// thresholds and draws are deterministic: the same inputs give the same bits on every run.
// The order "value descending, then token id ascending" is the order of 56-bit composite
// keys (an order-preserving 32-bit image of the value, then 2^24 - 1 - id); top-k and top-p
// are radix selections on these keys (8-bit digits, cluster-wide histograms), top-p with a
// leading digit that buckets the weight in eighths of an octave.
#include <stdint.h>

#include "ts_common.cuh"
#include "ts_internal.h"

namespace tsv {

static __device__ unsigned int g_staged_err;

constexpr int kThreads = 512;
constexpr int kChunks = 4;
constexpr int kMaxCluster = 8;
constexpr uint32_t kWaitLimit = 1u << 26;
constexpr int64_t kSliceTarget = 64 * 1024;   // bytes of row per CTA we aim for
constexpr int64_t kSliceMax = 192 * 1024;     // bytes of row per CTA we accept

struct RowCtl {
  // read by peer CTAs through DSMEM
  float p_max;
  int32_t p_am;
  float p_lm;
  float p_ls;
  uint64_t p_sum;
  int32_t p_tok;
  int32_t pad0;
  unsigned long long mass[2][256];
  uint32_t cnt[2][256];
  // local
  unsigned long long tot_mass[256];
  uint32_t tot_cnt[256];
  uint64_t bar[kChunks];
  uint64_t scan[kThreads / 32];
  float red_f[3][kThreads / 32];
  int32_t red_i[kThreads / 32];
  // broadcast scalars
  float M, S1;
  int32_t am;
  int32_t bin;
  int32_t bincnt;
  int32_t keep_all;
  uint64_t above;
  uint64_t target;
  uint64_t Z;
  int32_t tok;
  int32_t round;
};

template <typename E>
struct SV;
template <>
struct SV<float> {
  __device__ __forceinline__ static float get(const float* s, int64_t i) { return s[i]; }
};
template <>
struct SV<uint16_t> {
  __device__ __forceinline__ static float get(const uint16_t* s, int64_t i) {
    return bf16_bits_to_f32(s[i]);
  }
};

struct RadixOut {
  uint64_t prefix, mask, above;
  int keep_all;
};

// Cluster-wide radix selection over 64-bit composite keys.
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
      ctl->mass[buf][i] = 0;
      ctl->cnt[buf][i] = 0;
    }
    __syncthreads();
    const uint64_t pre = o.prefix, msk = o.mask;
    sweep([&](uint64_t key, float v) {
      if ((key & msk) == pre) {
        const int bin = (int)((key >> sh) & 255u);
        atomicAdd(&ctl->cnt[buf][bin], 1u);
        if (MASS) atomicAdd(&ctl->mass[buf][bin], (unsigned long long)wfn(v));
      }
    });
    __syncthreads();
    cluster.sync();
    if (tid < 256) {
      unsigned long long tm = 0;
      uint32_t tc = 0;
      for (uint32_t c = 0; c < CL; ++c) {
        RowCtl* pc = cluster.map_shared_rank(ctl, c);
        tm += pc->mass[buf][tid];
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
  constexpr int nw = kThreads / 32;
  uint64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) ctl->scan[w] = incl;
  __syncthreads();
  if (w == 0) {
    uint64_t t = lane < nw ? ctl->scan[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < nw) ctl->scan[lane] = t;
  }
  __syncthreads();
  const uint64_t before = (w > 0) ? ctl->scan[w - 1] : 0;
  total = ctl->scan[nw - 1];
  __syncthreads();
  return before + incl - v;
}

template <typename E>
__global__ void __launch_bounds__(kThreads, 2) k_staged(StagedArgs a, int64_t slice_n, int vec) {
  extern __shared__ __align__(128) unsigned char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const uint32_t crank = cluster.block_rank();
  const uint32_t CL = cluster.num_blocks();
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x / CL;
  E* sv = reinterpret_cast<E*>(smem);
  const int64_t sv_bytes = (slice_n * (int64_t)sizeof(E) + 127) & ~(int64_t)127;
  RowCtl* ctl = reinterpret_cast<RowCtl*>(smem + sv_bytes);
  const int64_t lo = (int64_t)crank * slice_n;
  const int64_t n = max((int64_t)0, min(slice_n, a.V - lo));
  const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;

  // ---- 1. stage the slice ----------------------------------------------------------
  if (tid == 0) ctl->round = 0;
  if (vec) {
    const int64_t bulk = (n * (int64_t)sizeof(E)) & ~(int64_t)15;
    int64_t cb = ((bulk / kChunks) + 15) & ~(int64_t)15;
    if (tid == 0) {
      for (int c = 0; c < kChunks; ++c) mbar_init(&ctl->bar[c], 1);
      fence_mbar_init();
      for (int c = 0; c < kChunks; ++c) {
        const int64_t off = min(bulk, c * cb);
        const int64_t len = min(bulk, off + cb) - off;
        mbar_arrive_expect_tx(&ctl->bar[c], (uint32_t)len);
        if (len > 0)
          bulk_g2s(reinterpret_cast<unsigned char*>(sv) + off,
                   reinterpret_cast<const unsigned char*>(xr + lo) + off, (uint32_t)len, &ctl->bar[c]);
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
  __syncthreads();

  // ---- 2. row maximum, argmax (lowest id), thread maxima, temperature-1 log-sum-exp ----
  const bool want_lse = (a.mode == kChain) && a.logprobs != nullptr;
  float bv = -INFINITY, lm = -INFINITY, ls = 0.f, lc = 0.f;
  int32_t bi = INT32_MAX;
  for (int64_t g = (int64_t)tid * 8; g < n; g += (int64_t)kThreads * 8) {
    float x[8];
    const int m = (int)min((int64_t)8, n - g);
    for (int k = 0; k < 8; ++k) x[k] = k < m ? SV<E>::get(sv, g + k) : -INFINITY;
    float vm = x[0];
    for (int k = 1; k < m; ++k) vm = fmaxf(vm, x[k]);
    if (vm > bv || bi == INT32_MAX) {
      for (int k = 0; k < m; ++k)
        if (x[k] == vm) {
          bi = (int32_t)(lo + g + k);
          break;
        }
      bv = vm;
    }
    if (want_lse && vm > -INFINITY) {
      const float nm = fmaxf(lm, vm);
      const float f = ex2((lm - nm) * kLog2e);
      ls *= f;
      lc *= f;
      lm = nm;
      float vs = 0.f;
      for (int k = 0; k < m; ++k) vs += ex2((x[k] - nm) * kLog2e);
      kahan_add(ls, lc, vs);
    }
  }
  ls += lc;
  // this thread's largest element as an order key (0 = the thread holds no element)
  const uint64_t tmax = (bi == INT32_MAX) ? 0ull : comp_key(fkey(bv), (uint32_t)bi);
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
      constexpr int nw = kThreads / 32;
      v = lane < nw ? ctl->red_f[0][lane] : -INFINITY;
      m = lane < nw ? ctl->red_f[1][lane] : -INFINITY;
      s = lane < nw ? ctl->red_f[2][lane] : 0.f;
      i = lane < nw ? ctl->red_i[lane] : INT32_MAX;
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
  cluster.sync();
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
  const int64_t req = (a.mode == kChain) ? row / a.R : row;
  const int32_t j = (a.mode == kChain) ? (int32_t)(row % a.R) : 0;
  float T = 1.f, tp = 1.f;
  int32_t k = 0;
  if (a.mode != kRenorm && a.temperature) T = a.temperature[req];
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

  // weight of a value: fixed point of exp((x - M)/T) (logits) or of the value (probs)
  auto efn = [&](float v) -> float {
    return is_logits ? ex2(-((M - v) * sl2)) : fminf(fmaxf(v, 0.f), 1.f);
  };
  auto wfn = [&](float v) -> uint64_t { return fixw(efn(v)); };
  // weight bucket, larger = heavier: eighths of an octave below the row maximum
  auto binkey = [&](float v) -> uint64_t {
    uint32_t b;
    if (is_logits) {
      const float d = (M - v) * sl2;
      b = (uint32_t)fminf(d * 8.f, 255.f);
    } else {
      const uint32_t vb = __float_as_uint(fmaxf(v, 0.f));
      b = (vb == 0u) ? 255u : min(255u, (pmax_bits - vb) >> 20);
    }
    return (uint64_t)(255u - b) << 56;
  };

  const bool bf16 = sizeof(E) == 2;
  const int shk_f[7] = {48, 40, 32, 24, 16, 8, 0};
  const int shk_h[5] = {48, 40, 16, 8, 0};
  const int shp_f[8] = {56, 48, 40, 32, 24, 16, 8, 0};
  const int shp_h[6] = {56, 48, 40, 16, 8, 0};

  auto slice_sweep = [&](auto&& f) {
    for (int64_t i = tid; i < n; i += kThreads) {
      const float v = SV<E>::get(sv, i);
      f(comp_key(fkey(v), (uint32_t)(lo + i)), v);
    }
  };

  // ---- 4. top-k: a bound from the thread maxima, then the exact k-th key -----------------
  RadixOut KT{0, 0, 0, 1}, KK{0, 0, 0, 1};
  if (tk) {
    if ((int64_t)k <= (int64_t)CL * kThreads) {
      KT = cluster_radix<false>(
          ctl, cluster, CL,
          [&](auto&& f) {
            if (tmax) f(tmax, 0.f);
          },
          [](float) { return (uint64_t)1; }, bf16 ? shk_h : shk_f, bf16 ? 5 : 7, (uint64_t)k, -1.f);
    }
    KK = cluster_radix<false>(
        ctl, cluster, CL,
        [&](auto&& f) {
          slice_sweep([&](uint64_t key, float v) {
            if (selected(KT, key)) f(key, v);
          });
        },
        [](float) { return (uint64_t)1; }, bf16 ? shk_h : shk_f, bf16 ? 5 : 7, (uint64_t)k, -1.f);
  }
  // The k-th key was selected among the elements that pass the thread-maxima bound, and an
  // early exit leaves the low digits of KK open: top-k membership needs both tests.
  auto keptk = [&](uint64_t key) -> bool {
    return !tk || (selected(KT, key) && selected(KK, key));
  };
  // ---- 5. top-p on the top-k survivors ----------------------------------------------------
  RadixOut PP{0, 0, 0, 1};
  if (tpa) {
    PP = cluster_radix<true>(
        ctl, cluster, CL,
        [&](auto&& f) {
          slice_sweep([&](uint64_t key, float v) {
            if (keptk(key)) f(binkey(v) | key, v);
          });
        },
        wfn, bf16 ? shp_h : shp_f, bf16 ? 6 : 8, 0, tp);
  }
  auto kept = [&](uint64_t key, float v) -> bool {
    if (!keptk(key)) return false;
    if (tpa && !selected(PP, binkey(v) | key)) return false;
    return true;
  };

  // ---- 6. outputs ----------------------------------------------------------------------
  if (a.mode == kSoftmax || a.mode == kRenorm) {
    uint64_t zt = 0;
    if (!greedy) {
      for (int64_t i = tid; i < n; i += kThreads) {
        const float v = SV<E>::get(sv, i);
        if (a.mode == kSoftmax || kept(comp_key(fkey(v), (uint32_t)(lo + i)), v)) zt += wfn(v);
      }
    }
    uint64_t tot;
    (void)block_excl_scan_u64(zt, ctl, tot);
    if (tid == 0) ctl->p_sum = tot;
    cluster.sync();
    if (tid == 0) {
      uint64_t Z = 0;
      for (uint32_t c = 0; c < CL; ++c) Z += cluster.map_shared_rank(ctl, c)->p_sum;
      ctl->Z = Z;
    }
    __syncthreads();
    const float scale = (ctl->Z > 0) ? __fdiv_rn(kFx, __ull2float_rn(ctl->Z)) : 0.f;
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

  // kChain: the accept test of this row's draft and this row's speculative draw
  const int32_t D = a.D;
  const int32_t x = (j < D) ? a.draft_tokens[req * D + j] : -1;
  const bool xvalid = x >= 0 && (int64_t)x < a.V;
  const uint64_t seed = a.seed ? (uint64_t)a.seed[req] : 0, off = a.offset ? (uint64_t)a.offset[req] : 0;
  const float uj = (j < D) ? (a.uniforms ? a.uniforms[req * a.R + j] : verify_coin(seed, off, (uint32_t)j)) : 0.f;
  const float uD = a.uniforms ? a.uniforms[req * a.R + D] : verify_coin(seed, off, (uint32_t)D);
  int32_t acc = 0, tok = am;
  if (greedy) {
    acc = (j < D) && (x == am);
  } else {
    // contiguous per-thread ranges, so that the draw can walk tokens in id order
    const int64_t cpt = (n + kThreads - 1) / kThreads;
    const int64_t r0 = min(n, (int64_t)tid * cpt), r1 = min(n, r0 + cpt);
    uint64_t zt = 0;
    for (int64_t i = r0; i < r1; ++i) {
      const float v = SV<E>::get(sv, i);
      const int64_t gi = lo + i;
      if (gi != (int64_t)x && kept(comp_key(fkey(v), (uint32_t)gi), v)) zt += wfn(v);
    }
    uint64_t ctot;
    const uint64_t texcl = block_excl_scan_u64(zt, ctl, ctot);
    if (tid == 0) ctl->p_sum = ctot;
    if (tid == 0) ctl->tok = -1;
    cluster.sync();
    // every CTA: the cluster totals, this CTA's prefix, the weight of the draft token
    uint64_t Zr = 0, cpre = 0;
    int last_nz = -1;
    for (uint32_t c = 0; c < CL; ++c) {
      const uint64_t pc = cluster.map_shared_rank(ctl, c)->p_sum;
      if (c < crank) cpre += pc;
      if (pc > 0) last_nz = (int)c;
      Zr += pc;
    }
    uint64_t wx = 0;
    if (xvalid) {
      const float vx = (sizeof(E) == 2) ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(xr)[x])
                                         : reinterpret_cast<const float*>(xr)[x];
      if (kept(comp_key(fkey(vx), (uint32_t)x), vx)) wx = wfn(vx);
    }
    const uint64_t Zf = Zr + wx;
    if (j < D) acc = ((double)uj * (double)Zf < (double)wx) ? 1 : 0;
    const uint64_t Zd = Zr;  // residual (x removed) or bonus (x = -1 removes nothing)
    if (Zd == 0) {
      tok = (wx > 0) ? x : am;  // all the mass sits on the draft token
    } else {
      const double tt = (double)uD * (double)Zd;
      uint64_t t = (uint64_t)tt;
      bool past = (t >= Zd);
      // this CTA holds the crossing iff cpre <= t < cpre + ctot (or it is the last with mass)
      const bool mine = past ? ((int)crank == last_nz) : (cpre <= t && t < cpre + ctot);
      if (mine) {
        const uint64_t tl = past ? ~0ull : t - cpre;
        const bool hit = past ? (zt > 0 && texcl + zt == ctot) : (texcl <= tl && tl < texcl + zt);
        if (hit) {
          uint64_t accw = texcl;
          int32_t found = -1, lastk = -1;
          for (int64_t i = r0; i < r1; ++i) {
            const float v = SV<E>::get(sv, i);
            const int64_t gi = lo + i;
            if (gi == (int64_t)x || !kept(comp_key(fkey(v), (uint32_t)gi), v)) continue;
            const uint64_t w = wfn(v);
            if (w == 0) continue;
            lastk = (int32_t)gi;
            if (!past && accw + w > tl) {
              found = (int32_t)gi;
              break;
            }
            accw += w;
          }
          if (found < 0) found = lastk;
          int32_t* dst = cluster.map_shared_rank(&ctl->tok, 0);
          *dst = found;
        }
      }
    }
  }
  cluster.sync();
  if (crank == 0 && tid == 0) {
    if (!greedy && ctl->tok >= 0) tok = ctl->tok;
    a.ws.rowres[row] = RowRes{M, am, ctl->S1, tok, acc, {0, 0, 0}};
    __threadfence();
    const uint32_t prev = atomicAdd(&a.ws.reqcnt[req], 1u);
    if (prev == (uint32_t)a.R - 1) {
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
    }
  }
  cluster.sync();
}

static int64_t slice_elems(int64_t V, int esize, int* CL_out) {
  int64_t bytes = V * esize;
  int CL = (int)min((int64_t)kMaxCluster, max((int64_t)1, (bytes + kSliceTarget - 1) / kSliceTarget));
  int64_t sl = ((V + CL - 1) / CL + 15) & ~(int64_t)15;
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
  const size_t smem = (size_t)((sl * (int64_t)sizeof(E) + 127) & ~(int64_t)127) + sizeof(RowCtl);
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
