// Split-row kernels for target-only chain sampling from logits (TokenSpeed flashinfer.py
// verify(): sampling_argmax for greedy requests; softmax with temperature, fused
// top-k/top-p renorm and chain_speculative_sampling_target_only for the others).
//
// k_chunk: every row is cut into chunks of 256 threads x 8 vectors (32 KB); one CTA
// loads its chunk into registers (one HBM pass, all loads in flight at once) and writes
// a small summary of it; no CTA waits for another. Every chunk gives the row statistics
// (maximum, argmax, temperature-1 log-sum-exp); by the request's knobs it adds:
//  - top-k (k <= kSTopK): the chunk's candidates for the row's top k: the elements at or
//    above a lower bound of the chunk's k-th value (the k-th largest thread maximum, or
//    for k > 256 the k-th largest of the threads' four largest values), appended to the
//    row's candidate list;
//  - neither knob: the mass of every warp step (32 consecutive vectors) relative to the
//    chunk maximum, the draft token left out;
//  - top-p alone: a histogram of the weights over sixteenth-of-an-octave buckets whose
//    edges are fixed multiples of T ln 2 / 16, so that the chunks' histograms align.
// k_finish: one CTA a row completes it from the summaries: the accept test of the row's
// draft and the row's draw; the last row of a request to finish writes the chain.
//  - top-k: the row's top k and the top-p prefix from the candidate list, the draw in
//    token-id order by a radix walk over the ids;
//  - neither: the chunk masses scaled to the row maximum locate the warp step of the
//    draw, which alone is re-read;
//  - top-p alone: the merged histogram gives the bucket where the ordered mass crosses
//    top_p; one re-read of the row gives whole-bucket masses per warp step and the
//    crossing bucket's elements, which are resolved exactly; then the draw as above.
// Rows these kernels cannot serve (top_k above kSTopK, candidate overflow, a crossing in
// the tail bucket) are flagged and left to the cluster-staged kernel.
//
// Weights are 2^((x - M) log2(e) / T) for a reference maximum M; masses that decide a
// selection are sums of floor(w * 2^40); composite keys order tokens by value, then by
// lowest id.
#include <stdint.h>

#include "ts_common.cuh"
#include "ts_internal.h"
#include "ts_select.cuh"

namespace tsv {

constexpr int kSWarps = kSThreads / 32;
constexpr int kSLocalCap = 2048;  // candidates one CTA holds in shared memory
constexpr int kSBins = 384;       // top-p buckets over 24 octaves; index kSBins is the tail
constexpr int kSSteps = kSVecs * kSWarps;  // warp steps of a chunk
constexpr double kInvFx = 1.0 / 1099511627776.0;

enum RowKind : int { kRowGreedy = 0, kRowTopK = 1, kRowPlain = 2, kRowTopP = 3, kRowStaged = 4 };

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
  __device__ __forceinline__ static float at(const float* p, int64_t i) { return p[i]; }
  __device__ __forceinline__ static void put(uint4& r, int q, float v) {
    const uint32_t b = __float_as_uint(v);
    if (q == 0) r.x = b;
    else if (q == 1) r.y = b;
    else if (q == 2) r.z = b;
    else r.w = b;
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
  __device__ __forceinline__ static float at(const uint16_t* p, int64_t i) {
    return bf16_bits_to_f32(p[i]);
  }
  __device__ __forceinline__ static void put(uint4& r, int q, float v) {
    const uint32_t h = __float_as_uint(v) >> 16;  // exact: v is a widened bf16
    uint32_t* w = (q < 2) ? &r.x : (q < 4) ? &r.y : (q < 6) ? &r.z : &r.w;
    *w = (q & 1) ? ((*w & 0x0000FFFFu) | (h << 16)) : ((*w & 0xFFFF0000u) | h);
  }
};

__device__ __forceinline__ float key_to_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ uint32_t comp_token(uint64_t c) {
  return kIdxMax - (uint32_t)(c & kIdxMax);
}

// Warp sum by butterfly: every lane ends with the same bits.
__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Exclusive scan of a double over the block in thread order (a fixed order of additions,
// so the result is reproducible); writes the block total.
__device__ __forceinline__ double excl_scan_f64(double v, double* sc, double& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sc[w] = incl;
  __syncthreads();
  if (w == 0) {
    double t = lane < kSWarps ? sc[lane] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kSWarps) sc[lane] = t;
  }
  __syncthreads();
  const double before = (w > 0) ? sc[w - 1] : 0.0;
  total = sc[kSWarps - 1];
  __syncthreads();
  return before + (incl - v);
}

// The absolute top-p bucket coordinate of a value: floor(x log2(e) / T * 16). Bucket edges
// do not depend on any maximum, so the chunks' histograms align by integer offsets.
__device__ __forceinline__ float babs(float v, float sl2) { return floorf(v * sl2 * 16.f); }

// The request's knobs and the way its rows are served.
struct Knobs {
  float T, tp;
  int32_t k;
  int kind;
};
__device__ __forceinline__ Knobs row_knobs(const SampleArgs& a, int64_t req) {
  Knobs kn;
  kn.T = a.temperature ? a.temperature[req] : 1.f;
  kn.k = a.top_k ? a.top_k[req] : 0;
  kn.tp = a.top_p ? a.top_p[req] : 1.f;
  if (!(kn.T >= kGreedyT)) kn.kind = kRowGreedy;
  else if (kn.k > 0 && (int64_t)kn.k < a.V) kn.kind = (kn.k <= kSTopK) ? kRowTopK : kRowStaged;
  else kn.kind = (kn.tp < 1.f) ? kRowTopP : kRowPlain;
  return kn;
}

// ---- k_chunk ----------------------------------------------------------------------------

struct ChunkSmem {
  sel::Scratch sc;
  union {
    uint32_t h3[3][kSBins + 1];     // top-p histogram as digit sums
    uint32_t tkeys[kSThreads * 4];  // the threads' largest keys
  } u;
  uint64_t list[kSLocalCap];
  uint32_t lcnt, wcnt, base;
  float Ms;
  float red_f[3][kSWarps];
  int32_t red_i[kSWarps];
};

template <typename E>
__global__ void __launch_bounds__(kSThreads, 3) k_chunk(SampleArgs a) {
  __shared__ ChunkSmem sm;
  constexpr int N = SVec<E>::N;
  const int S = a.splits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x / S;
  const int split = (int)(blockIdx.x % S);
  const int64_t req = row / a.R;
  const int32_t j = (int32_t)(row % a.R);
  const Knobs kn = row_knobs(a, req);
  if (kn.kind == kRowStaged) {  // the cluster-staged kernel takes this row
    if (split == 0 && tid == 0) a.ws.flag[row] = 1u;
    return;
  }
  const bool bf16 = sizeof(E) == 2;
  const int64_t V = a.V;
  const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;
  const int64_t lo = (int64_t)split * a.chunk;
  const int n = (int)min(a.chunk, V - lo);
  const int nvf = n / N;  // whole vectors of this chunk
  const uint4* vp = reinterpret_cast<const uint4*>(xr + lo);
  const uint4 ninf = make_uint4(SVec<E>::kNegInfWord, SVec<E>::kNegInfWord,
                                SVec<E>::kNegInfWord, SVec<E>::kNegInfWord);

  // ---- 1. the chunk into registers: thread t holds vectors t + 256 u ---------------------
  uint4 r[kSVecs];
#pragma unroll
  for (int u = 0; u < kSVecs; ++u) {
    const int vi = u * kSThreads + tid;
    r[u] = (vi < nvf) ? ldg_stream(vp + vi) : ninf;
  }
  if (n % N) {  // the ragged last vector, padded with -inf
    const int vt = nvf;
    if (tid == vt % kSThreads) {
      uint4 tv = ninf;
      for (int q = 0; q < n - vt * N; ++q)
        SVec<E>::put(tv, q, SVec<E>::at(xr, lo + (int64_t)vt * N + q));
#pragma unroll
      for (int u = 0; u < kSVecs; ++u)
        if (u == vt / kSThreads) r[u] = tv;
    }
  }

  // ---- 2. maximum, argmax (lowest id), temperature-1 log-sum-exp ------------------------
  float vm[kSVecs];
  float bv = -INFINITY;
#pragma unroll
  for (int u = 0; u < kSVecs; ++u) {
    vm[u] = SVec<E>::vmax(r[u]);
    bv = fmaxf(bv, vm[u]);
  }
  int32_t bi = INT32_MAX;
  {
    uint4 rb = r[0];
    int ub = -1;
#pragma unroll
    for (int u = kSVecs - 1; u >= 0; --u)
      if (vm[u] == bv) {
        rb = r[u];
        ub = u;
      }
    float xb[N];
    SVec<E>::unpack(rb, xb);
    int qb = N - 1;
#pragma unroll
    for (int q = N - 1; q >= 0; --q)
      if (xb[q] == bv) qb = q;
    const int li = (ub * kSThreads + tid) * N + qb;
    if (ub >= 0 && li < n) bi = (int32_t)(lo + li);
  }
  float lm = -INFINITY, ls = 0.f;
  if (a.logprobs && bv > -INFINITY) {
    lm = bv;
#pragma unroll
    for (int u = 0; u < kSVecs; ++u) {
      float xv[N];
      SVec<E>::unpack(r[u], xv);
      float vs = 0.f;
#pragma unroll
      for (int q = 0; q < N; ++q) vs += ex2((xv[q] - lm) * kLog2e);
      ls += vs;
    }
  }
  {
    float v = bv, m = lm, s = ls;
    int32_t i = bi;
    warp_argmax(v, i);
    warp_lse(m, s);
    if (lane == 0) {
      sm.red_f[0][warp] = v;
      sm.red_f[1][warp] = m;
      sm.red_f[2][warp] = s;
      sm.red_i[warp] = i;
    }
    __syncthreads();
    if (warp == 0) {
      v = lane < kSWarps ? sm.red_f[0][lane] : -INFINITY;
      m = lane < kSWarps ? sm.red_f[1][lane] : -INFINITY;
      s = lane < kSWarps ? sm.red_f[2][lane] : 0.f;
      i = lane < kSWarps ? sm.red_i[lane] : INT32_MAX;
      warp_argmax(v, i);
      warp_lse(m, s);
      if (lane == 0) {
        a.ws.part[row * kMaxSplits + split] = Part{v, i, m, s};
        sm.Ms = v;
        sm.lcnt = 0;
        sm.wcnt = 0;
      }
    }
  }
  if (kn.kind == kRowGreedy) return;
  __syncthreads();
  const float Ms = sm.Ms;
  const float sl2 = __fdiv_rn(kLog2e, kn.T);
  uint64_t* const rowslots = a.ws.cand + row * a.ws.cand_splits * (int64_t)kSTopK;
  uint64_t* const slots = rowslots + (int64_t)split * kSTopK;

  // ---- 3. the chunk's summary -------------------------------------------------------------
  if (kn.kind == kRowTopK) {
    const int k = kn.k;
    uint32_t tkey;
    if (k <= kSThreads) {
      // the k-th largest thread maximum bounds the chunk's k-th value from below
      sm.u.tkeys[tid] = (bv > -INFINITY) ? fkey(bv) : 0u;
      __syncthreads();
      tkey = sel::select_bound<kSThreads>(
          kSThreads, [&](int i) { return sm.u.tkeys[i]; }, (uint32_t)k, bf16 ? 2 : 4, sm.sc);
    } else {
      // the threads' four largest values
      float t4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int u = 0; u < kSVecs; ++u) {
        if (!(vm[u] > t4[3])) continue;
        float xv[N];
        SVec<E>::unpack(r[u], xv);
#pragma unroll
        for (int q = 0; q < N; ++q) {
          const float v = xv[q];
          if (!(v > t4[3])) continue;
          // insert v into the descending list t4 (equal values take a slot each)
          if (v > t4[1]) {
            t4[3] = t4[2];
            t4[2] = t4[1];
            if (v > t4[0]) {
              t4[1] = t4[0];
              t4[0] = v;
            } else {
              t4[1] = v;
            }
          } else if (v > t4[2]) {
            t4[3] = t4[2];
            t4[2] = v;
          } else {
            t4[3] = v;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) sm.u.tkeys[tid * 4 + q] = (t4[q] > -INFINITY) ? fkey(t4[q]) : 0u;
      __syncthreads();
      tkey = sel::select_bound<kSThreads>(
          kSThreads * 4, [&](int i) { return sm.u.tkeys[i]; }, (uint32_t)k, bf16 ? 2 : 4, sm.sc);
    }
    // the elements at or above the bound
#pragma unroll
    for (int u = 0; u < kSVecs; ++u) {
      if (!(vm[u] > -INFINITY) || fkey(vm[u]) < tkey) continue;
      float xv[N];
      SVec<E>::unpack(r[u], xv);
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const uint32_t kq = fkey(xv[q]);
        if (kq >= tkey && xv[q] != -INFINITY) {
          const uint32_t pos = atomicAdd(&sm.lcnt, 1u);
          if (pos < (uint32_t)kSLocalCap)
            sm.list[pos] = comp_key(kq, (uint32_t)(lo + (u * kSThreads + tid) * N + q));
        }
      }
    }
    __syncthreads();
    const uint32_t cnt = sm.lcnt;
    if (cnt > (uint32_t)kSLocalCap) {
      if (tid == 0) a.ws.flag[row] = 1u;  // too many ties at the bound
      return;
    }
    // more than kSTopK candidates: cut them to the chunk's top k, by value first, exactly
    // if ties at the k-th value remain
    uint64_t Cs = 0;
    if (cnt > (uint32_t)kSTopK) {
      const uint32_t vk = sel::select_bound<kSThreads>(
          (int)cnt, [&](int i) { return (uint32_t)(sm.list[i] >> kIdxBits); }, (uint32_t)k,
          bf16 ? 2 : 4, sm.sc);
      Cs = (uint64_t)vk << kIdxBits;
      uint32_t c2 = 0;
      for (uint32_t i = tid; i < cnt; i += kSThreads) c2 += (sm.list[i] >= Cs) ? 1u : 0u;
      if (c2) atomicAdd(&sm.wcnt, c2);
      __syncthreads();
      const uint32_t m2 = sm.wcnt;
      __syncthreads();
      if (m2 > (uint32_t)kSTopK) {
        const int shf[7] = {48, 40, 32, 24, 16, 8, 0};
        const int shh[5] = {48, 40, 16, 8, 0};
        Cs = sel::radix<kSThreads, false>(
            (int)cnt, [&](int i) { return sm.list[i]; }, 1ull, (uint64_t)k,
            [](uint64_t) { return (uint64_t)1; }, bf16 ? shh : shf, bf16 ? 5 : 7, sm.sc);
      }
    }
    if (tid == 0) sm.wcnt = 0;
    __syncthreads();
    uint32_t mine = 0;
    for (uint32_t i = tid; i < cnt; i += kSThreads) mine += (sm.list[i] >= Cs) ? 1u : 0u;
    if (mine) atomicAdd(&sm.wcnt, mine);
    __syncthreads();
    if (tid == 0) {
      sm.base = atomicAdd(&a.ws.ccount[row], sm.wcnt);
      sm.lcnt = 0;
    }
    __syncthreads();
    uint64_t* dst = rowslots + sm.base;
    for (uint32_t i = tid; i < cnt; i += kSThreads) {
      const uint64_t c = sm.list[i];
      if (c >= Cs) dst[atomicAdd(&sm.lcnt, 1u)] = c;
    }
  } else if (kn.kind == kRowPlain) {
    // the mass of every warp step relative to the chunk maximum, the draft token left out;
    // warp step u * 8 + w covers the vectors 256 u + 32 w .. 256 u + 32 w + 31
    const int32_t x = (j < a.D) ? a.draft_tokens[req * a.D + j] : -1;
    const int64_t xl64 = (int64_t)x - lo;
    const int xl = (x >= 0 && xl64 >= 0 && xl64 < n) ? (int)xl64 : -1;
    const int xv_i = (xl >= 0) ? xl / N : -1;  // the vector holding the draft token
#pragma unroll
    for (int u = 0; u < kSVecs; ++u) {
      float xv[N];
      SVec<E>::unpack(r[u], xv);
      const int xq = (xv_i == u * kSThreads + tid) ? xl % N : -1;
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const float w = ex2((xv[q] - Ms) * sl2);
        s += (q == xq) ? 0.f : w;
      }
      const uint64_t f = fixw(warp_sum_f32(s));
      if (lane == 0) slots[u * kSWarps + warp] = f;
    }
  } else {
    // the top-p histogram relative to the chunk maximum, on absolute bucket edges
    for (int i = tid; i < 3 * (kSBins + 1); i += kSThreads) (&sm.u.h3[0][0])[i] = 0;
    __syncthreads();
    const float bs = babs(Ms, sl2);
    uint64_t tail = 0;
#pragma unroll
    for (int u = 0; u < kSVecs; ++u) {
      float xv[N];
      SVec<E>::unpack(r[u], xv);
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const uint64_t w = fixw(ex2((xv[q] - Ms) * sl2));
        if (w == 0) continue;
        const float off = bs - babs(xv[q], sl2);
        if (off < (float)kSBins) {
          const int b = (int)off;
          sel::add3(&sm.u.h3[0][b], &sm.u.h3[1][b], &sm.u.h3[2][b], w);
        } else {
          tail += w;
        }
      }
    }
    tail = warp_sum_u64(tail);
    if (lane == 0 && tail)
      sel::add3(&sm.u.h3[0][kSBins], &sm.u.h3[1][kSBins], &sm.u.h3[2][kSBins], tail);
    __syncthreads();
    for (int i = tid; i <= kSBins; i += kSThreads)
      slots[i] = sel::get3(sm.u.h3[0][i], sm.u.h3[1][i], sm.u.h3[2][i]);
    if (tid == 0) slots[kSBins + 1] = (uint64_t)__float_as_uint(bs);
  }
}

// ---- k_finish ---------------------------------------------------------------------------

struct FinishSmem {
  sel::Scratch sc;
  uint64_t list[kSLocalCap];
  double rowmass[kSBins];
  double dscan[32];
  double scale[kMaxSplits];
  uint32_t lcnt;
  float M, S1;
  int32_t am;
  float uj, uD, vx;
  int32_t owner, sstar;
  uint64_t res_u;
  double res_d;
};

template <typename E>
__global__ void __launch_bounds__(kSThreads) k_finish(SampleArgs a) {
  __shared__ FinishSmem sm;
  constexpr int N = SVec<E>::N;
  const int S = a.splits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int64_t req = row / a.R;
  const int32_t j = (int32_t)(row % a.R);
  const Knobs kn = row_knobs(a, req);
  if (kn.kind == kRowStaged) return;
  const bool bf16 = sizeof(E) == 2;
  const int64_t V = a.V;
  const int64_t CH = a.chunk;
  const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;
  const int32_t D = a.D;
  const int32_t x = (j < D) ? a.draft_tokens[req * D + j] : -1;
  const bool xvalid = x >= 0 && (int64_t)x < V;
  uint64_t* const rowslots = a.ws.cand + row * a.ws.cand_splits * (int64_t)kSTopK;
  const int shf[7] = {48, 40, 32, 24, 16, 8, 0};
  const int shh[5] = {48, 40, 16, 8, 0};
  const int* cs = bf16 ? shh : shf;
  const int ncs = bf16 ? 5 : 7;

  if (tid < 32) {
    float v = -INFINITY, m = -INFINITY, s = 0.f;
    int32_t i = INT32_MAX;
    for (int q = lane; q < S; q += 32) {
      const Part* pp = &a.ws.part[row * kMaxSplits + q];
      argmax_merge(v, i, __ldcg(&pp->v), __ldcg(&pp->i));
      lse_merge(m, s, __ldcg(&pp->m), __ldcg(&pp->s));
    }
    warp_argmax(v, i);
    warp_lse(m, s);
    if (lane == 0) {
      sm.M = v;
      sm.am = (i == INT32_MAX) ? 0 : i;
      sm.S1 = s;
      const uint64_t seed = a.seed ? (uint64_t)a.seed[req] : 0;
      const uint64_t off = a.offset ? (uint64_t)a.offset[req] : 0;
      const bool coins = kn.kind != kRowGreedy;
      sm.uj = (coins && j < D)
                  ? (a.uniforms ? a.uniforms[req * a.R + j] : verify_coin(seed, off, (uint32_t)j))
                  : 0.f;
      sm.uD = coins ? (a.uniforms ? a.uniforms[req * a.R + D] : verify_coin(seed, off, (uint32_t)D))
                    : 0.f;
      sm.vx = xvalid ? SVec<E>::at(xr, x) : 0.f;
    }
  }
  __syncthreads();
  const uint32_t total = (kn.kind == kRowTopK) ? __ldcg(&a.ws.ccount[row]) : 0u;
  const bool flagged = (kn.kind != kRowGreedy) && __ldcg(&a.ws.flag[row]) != 0u;
  __syncthreads();
  if (tid == 0 && kn.kind == kRowTopK) a.ws.ccount[row] = 0;
  if (flagged) return;  // the cluster-staged kernel finishes the row
  const float M = sm.M;
  const int32_t am = sm.am;
  const float uj = sm.uj, uD = sm.uD, vx = sm.vx;
  const float sl2 = (kn.kind == kRowGreedy) ? 0.f : __fdiv_rn(kLog2e, kn.T);
  const float tp = kn.tp;
  auto wfn = [&](float v) -> uint64_t { return fixw(ex2((v - M) * sl2)); };
  auto wcomp = [&](uint64_t c) -> uint64_t {
    return wfn(key_to_value((uint32_t)(c >> kIdxBits)));
  };

  // records the row; the last row of its request to be recorded writes the chain
  auto finish_row = [&](int32_t tok_f, int32_t acc_f) {
    a.ws.rowres[row] = RowRes{M, am, sm.S1, tok_f, acc_f, {0, 0, 0}};
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
        if (jj <= js && t >= 0 && (int64_t)t < V) {
          const E* xj = reinterpret_cast<const E*>(a.x) + rj * a.ld;
          lp = (SVec<E>::at(xj, t) - __ldcg(&a.ws.rowres[rj].M)) - logf(__ldcg(&a.ws.rowres[rj].S));
        }
        a.logprobs[rj] = lp;
      }
    }
    a.accept_length[req] = js + 1;
  };

  if (kn.kind == kRowGreedy) {
    if (tid == 0) finish_row(am, (j < D && x == am) ? 1 : 0);
    return;
  }

  const int64_t nvr = V / N;  // whole vectors of the row; the rest is a scalar tail
  const int64_t nvall = (V + N - 1) / N;
  const uint4* rp = reinterpret_cast<const uint4*>(xr);
  auto load_vec = [&](int64_t vi, float* xv) {
    if (vi < nvr) {
      SVec<E>::unpack(__ldcg(rp + vi), xv);
    } else {
      for (int q = 0; q < N; ++q) {
        const int64_t i = vi * N + q;
        xv[q] = (i < V) ? SVec<E>::at(xr, i) : -INFINITY;
      }
    }
  };
  // Warp 0 walks the warp step starting at row vector v0 (32 vectors, one a lane) and
  // returns the first element at which the running weight exceeds tf (the last element
  // with weight if none does, e.g. by rounding; -1 if the step has no weight).
  auto walk_step = [&](int64_t v0, float tf, auto&& wgt) -> int32_t {
    const int64_t vi = v0 + lane;
    float xv[N];
    float vs = 0.f;
    if (vi < nvall) {
      load_vec(vi, xv);
#pragma unroll
      for (int q = 0; q < N; ++q) vs += wgt(xv[q], vi * N + q);
    }
    float inc = vs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const unsigned cross = __ballot_sync(0xffffffffu, vs > 0.f && inc > tf);
    const unsigned nz = __ballot_sync(0xffffffffu, vs > 0.f);
    const int wl = cross ? __ffs(cross) - 1 : (nz ? 31 - __clz(nz) : -1);
    int32_t f = -1;
    if (lane == wl) {
      float accf = inc - vs;
      for (int q = 0; q < N; ++q) {
        const float w = wgt(xv[q], vi * N + q);
        if (w == 0.f) continue;
        f = (int32_t)(vi * N + q);
        accf += w;
        if (cross && accf > tf) break;
      }
    }
    return (wl >= 0) ? __shfl_sync(0xffffffffu, f, wl) : -1;
  };

  if (kn.kind == kRowTopK) {
    // ---- top-k from the chunks' candidates -------------------------------------------------
    const int k = kn.k;
    const int ng = (int)total;
    const uint64_t Ck = sel::radix<kSThreads, false>(
        ng, [&](int i) { return __ldcg(rowslots + i); }, 1ull, (uint64_t)k,
        [](uint64_t) { return (uint64_t)1; }, cs, ncs, sm.sc);
    if (tid == 0) sm.lcnt = 0;
    __syncthreads();
    for (int i = tid; i < ng; i += kSThreads) {
      const uint64_t c = __ldcg(rowslots + i);
      if (c >= Ck) sm.list[atomicAdd(&sm.lcnt, 1u)] = c;  // at most k <= kSTopK items
    }
    __syncthreads();
    const int nl = (int)sm.lcnt;
    auto item = [&](int i) { return sm.list[i]; };
    auto mass_from = [&](uint64_t c0) -> uint64_t {
      uint64_t sum = 0;
      for (int i = tid; i < nl; i += kSThreads) {
        const uint64_t c = sm.list[i];
        if (c >= c0) sum += wcomp(c);
      }
      uint64_t tot;
      (void)sel::excl_scan<kSThreads>(sum, sm.sc, tot);
      return tot;
    };
    uint64_t C = Ck, Z = mass_from(Ck);
    if (tp < 1.f) {
      const double want = ceil((double)tp * (double)Z);
      const uint64_t P = (want > (double)Z) ? Z : (uint64_t)want;
      C = sel::radix<kSThreads, true>(nl, item, Ck, P, wcomp, cs, ncs, sm.sc);
      Z = mass_from(C);
    }
    uint64_t wx = 0;
    if (xvalid && comp_key(fkey(vx), (uint32_t)x) >= C) wx = wfn(vx);
    const int32_t acc = (j < D) && ((double)uj * (double)Z < (double)wx) ? 1 : 0;
    const uint64_t Zr = Z - wx;
    int32_t tok;
    if (Zr == 0) {
      tok = (wx > 0) ? x : am;
    } else {
      uint64_t t = (uint64_t)((double)uD * (double)Zr);
      if (t >= Zr) t = Zr - 1;
      const int idx_sh[3] = {16, 8, 0};
      uint64_t g = 0;
      (void)sel::radix<kSThreads, true>(
          nl, item, C, t + 1,
          [&](uint64_t c) { return ((int32_t)comp_token(c) == x) ? 0ull : wcomp(c); }, idx_sh, 3,
          sm.sc, &g);
      tok = (int32_t)comp_token(g);
    }
    if (tid == 0) finish_row(tok, acc);
    return;
  }

  if (kn.kind == kRowPlain) {
    // ---- neither knob: the chunks' warp-step masses, scaled to the row maximum ----------
    if (tid < S)
      sm.scale[tid] = exp2((double)((__ldcg(&a.ws.part[row * kMaxSplits + tid].v) - M) * sl2));
    __syncthreads();
    const int64_t E_ = (int64_t)S * kSSteps;
    const int64_t per = (E_ + kSThreads - 1) / kSThreads;
    const int64_t e0 = min(E_, (int64_t)tid * per), e1 = min(E_, e0 + per);
    auto entry = [&](int64_t e) -> double {
      const int64_t s = e / kSSteps, w = e - s * kSSteps;
      return (double)__ldcg(rowslots + s * kSTopK + w) * kInvFx * sm.scale[s];
    };
    double mine = 0.0;
    for (int64_t e = e0; e < e1; ++e) mine += entry(e);
    double Zr;
    const double ex = excl_scan_f64(mine, sm.dscan, Zr);
    const double wx = xvalid ? exp2((double)((vx - M) * sl2)) : 0.0;
    const int32_t acc = (j < D) && ((double)uj * (Zr + wx) < wx) ? 1 : 0;
    if (!(Zr > 0.0)) {
      if (tid == 0) finish_row((wx > 0.0) ? x : am, acc);
      return;
    }
    const double t = (double)uD * Zr;
    if (tid == 0) sm.owner = -1;
    __syncthreads();
    if (mine > 0.0 && ex <= t && t < ex + mine) sm.owner = tid;
    __syncthreads();
    if (sm.owner < 0) {  // rounding: the last thread with mass
      if (mine > 0.0) atomicMax(&sm.owner, tid);
      __syncthreads();
    }
    if (tid == sm.owner) {
      double accd = ex;
      int64_t es = -1, elast = -1;
      double rs = 0.0, rlast = 0.0;
      for (int64_t e = e0; e < e1; ++e) {
        const double m = entry(e);
        if (m <= 0.0) continue;
        elast = e;
        rlast = accd;
        if (t < accd + m) {
          es = e;
          rs = accd;
          break;
        }
        accd += m;
      }
      if (es < 0) {
        es = elast;
        rs = rlast;
      }
      const int64_t s = es / kSSteps;
      sm.sstar = (int32_t)s;
      sm.res_u = (uint64_t)es;
      // the residual in the chunk's own weight units (relative to its maximum)
      sm.res_d = (t - rs) / sm.scale[s];
    }
    __syncthreads();
    if (warp != 0) return;
    const int s = sm.sstar;
    const int64_t es = (int64_t)sm.res_u;
    const float Mss = __ldcg(&a.ws.part[row * kMaxSplits + s].v);
    const int64_t v0 = (int64_t)s * (CH / N) + (es - (int64_t)s * kSSteps) * 32;
    const int32_t tok = walk_step(v0, (float)sm.res_d, [&](float v, int64_t gi) -> float {
      return (gi == (int64_t)x) ? 0.f : ex2((v - Mss) * sl2);
    });
    if (lane == 0) finish_row(tok >= 0 ? tok : am, acc);
    return;
  }

  // ---- top-p alone: merged histogram, crossing bucket, one re-read of the row ------------
  if (tp <= 0.f) {  // only the argmax is kept
    if (tid == 0) finish_row(am, (j < D && x == am) ? 1 : 0);
    return;
  }
  const float bM = babs(M, sl2);
  for (int i = tid; i < kSBins; i += kSThreads) sm.rowmass[i] = 0.0;
  __syncthreads();
  double tailm = 0.0;
  for (int s = 0; s < S; ++s) {
    const uint64_t* hs = rowslots + (int64_t)s * kSTopK;
    const float bs = __uint_as_float((uint32_t)__ldcg(hs + kSBins + 1));
    const double sc =
        exp2((double)((__ldcg(&a.ws.part[row * kMaxSplits + s].v) - M) * sl2)) * kInvFx;
    const float d = bM - bs;  // >= 0: the chunk's buckets sit d buckets lower in the row
    for (int i = tid; i <= kSBins; i += kSThreads) {
      const uint64_t h = __ldcg(hs + i);
      if (h == 0) continue;
      const float ri = (i == kSBins) ? 1.0e9f : (float)i + d;
      if (ri < (float)kSBins) sm.rowmass[(int)ri] += (double)h * sc;
      else tailm += (double)h * sc;
    }
    __syncthreads();
  }
  // row buckets in order 0..383: thread t holds buckets t and t + 256; the tail is last
  const double h0 = sm.rowmass[tid];
  const double h1 = (tid + kSThreads < kSBins) ? sm.rowmass[tid + kSThreads] : 0.0;
  double tail_all, Zb, Zb2;
  (void)excl_scan_f64(tailm, sm.dscan, tail_all);
  const double ex0 = excl_scan_f64(h0, sm.dscan, Zb);
  const double ex1 = excl_scan_f64(h1, sm.dscan, Zb2);
  const double Zt = Zb + Zb2 + tail_all;
  const double P = (double)tp * Zt;
  if (tid == 0) sm.owner = -1;
  __syncthreads();
  if (h0 > 0.0 && ex0 < P && P <= ex0 + h0) {
    sm.owner = tid;
    sm.res_d = ex0;
  }
  if (h1 > 0.0 && Zb + ex1 < P && P <= Zb + ex1 + h1) {
    sm.owner = tid + kSThreads;
    sm.res_d = Zb + ex1;
  }
  __syncthreads();
  const int bstar = sm.owner;
  const double pre = sm.res_d;
  __syncthreads();
  if (bstar < 0) {  // the crossing lies in the tail bucket: the cluster kernel takes it
    if (tid == 0) a.ws.flag[row] = 1u;
    return;
  }
  // the re-read: whole-bucket masses per row warp step, the crossing bucket's elements
  const float fb = (float)bstar;
  if (tid == 0) sm.lcnt = 0;
  __syncthreads();
  uint64_t* const steps = rowslots;  // the chunk histograms are merged: reuse their slots
  const int64_t nst = (nvall + 31) / 32;
  for (int64_t g = warp; g < nst; g += kSWarps) {
    const int64_t vi = g * 32 + lane;
    float s = 0.f;
    if (vi < nvall) {
      float xv[N];
      load_vec(vi, xv);
      float vmx = xv[0];
#pragma unroll
      for (int q = 1; q < N; ++q) vmx = fmaxf(vmx, xv[q]);
      if (vmx > -INFINITY && bM - babs(vmx, sl2) <= fb) {  // else every element is lighter
#pragma unroll
        for (int q = 0; q < N; ++q) {
          const float v = xv[q];
          if (v == -INFINITY) continue;
          const float off = bM - babs(v, sl2);
          const int64_t gi = vi * N + q;
          if (off < fb) {
            if (gi != (int64_t)x) s += ex2((v - M) * sl2);
          } else if (off == fb && wfn(v) > 0) {
            const uint32_t pos = atomicAdd(&sm.lcnt, 1u);
            if (pos < (uint32_t)kSLocalCap) sm.list[pos] = comp_key(fkey(v), (uint32_t)gi);
          }
        }
      }
    }
    const uint64_t f = fixw(warp_sum_f32(s));
    if (lane == 0) steps[g] = f;
  }
  __syncthreads();
  const uint32_t cnt = sm.lcnt;
  if (cnt > (uint32_t)kSLocalCap || cnt == 0) {
    if (tid == 0) a.ws.flag[row] = 1u;
    return;
  }
  const double want = ceil((P - pre) * 1099511627776.0);
  const uint64_t Pb = want < 1.0 ? 1ull : (uint64_t)want;
  const uint64_t C = sel::radix<kSThreads, true>((int)cnt, [&](int i) { return sm.list[i]; }, 1ull,
                                                 Pb, wcomp, cs, ncs, sm.sc);
  // the kept elements of the crossing bucket join their steps
  for (uint32_t i = tid; i < cnt; i += kSThreads) {
    const uint64_t c = sm.list[i];
    const uint32_t gi = comp_token(c);
    if (c >= C && (int32_t)gi != x)
      atomicAdd(reinterpret_cast<unsigned long long*>(steps + (gi / N) / 32),
                (unsigned long long)wcomp(c));
  }
  __syncthreads();
  auto kept = [&](float v, int64_t gi) -> bool {
    const float off = bM - babs(v, sl2);
    if (off < fb) return true;
    return off == fb && comp_key(fkey(v), (uint32_t)gi) >= C;
  };
  uint64_t wx = 0;
  if (xvalid && kept(vx, x)) wx = wfn(vx);
  const int64_t per = (nst + kSThreads - 1) / kSThreads;
  const int64_t g0 = min(nst, (int64_t)tid * per), g1 = min(nst, g0 + per);
  uint64_t mine = 0;
  for (int64_t g = g0; g < g1; ++g) mine += __ldcg(steps + g);
  uint64_t Zr;
  const uint64_t ex = sel::excl_scan<kSThreads>(mine, sm.sc, Zr);
  const int32_t acc = (j < D) && ((double)uj * (double)(Zr + wx) < (double)wx) ? 1 : 0;
  if (Zr == 0) {
    if (tid == 0) finish_row((wx > 0) ? x : am, acc);
    return;
  }
  uint64_t t = (uint64_t)((double)uD * (double)Zr);
  if (t >= Zr) t = Zr - 1;
  if (mine > 0 && ex <= t && t < ex + mine) {
    uint64_t accu = ex;
    int64_t gs = g1 - 1;
    for (int64_t g = g0; g < g1; ++g) {
      const uint64_t m = __ldcg(steps + g);
      if (t < accu + m) {
        gs = g;
        break;
      }
      accu += m;
    }
    sm.res_u = (uint64_t)gs;
    sm.res_d = (double)(t - accu) * kInvFx;
  }
  __syncthreads();
  if (warp != 0) return;
  const int64_t gs = (int64_t)sm.res_u;
  const int32_t tok = walk_step(gs * 32, (float)sm.res_d, [&](float v, int64_t gi) -> float {
    if (gi == (int64_t)x || v == -INFINITY || !kept(v, gi)) return 0.f;
    return ex2((v - M) * sl2);
  });
  if (lane == 0) finish_row(tok >= 0 ? tok : am, acc);
}

cudaError_t launch_sample(const SampleArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)(a.rows * a.splits));
  if (a.bf16) {
    k_chunk<uint16_t><<<grid, kSThreads, 0, s>>>(a);
    k_finish<uint16_t><<<(unsigned)a.rows, kSThreads, 0, s>>>(a);
  } else {
    k_chunk<float><<<grid, kSThreads, 0, s>>>(a);
    k_finish<float><<<(unsigned)a.rows, kSThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace tsv
