// Row-streaming kernel for the top-k/top-p renormalisation of probability rows (TokenSpeed
// flashinfer.py verify(): fused_topk_topp_renorm). Its row machinery was first written for
// chain sampling as well; chain sampling from logits now runs in ts_chain.cu, and only
// the renorm mode (RN = true) is instantiated.
//
// A persistent CTA (2 an SM) takes one row after another from a tiered order that every
// CTA computes alike (large top-k and general rows, then top-p rows, then the rest; no
// workspace). A producer warp streams each row through a ring of kRNSt shared-memory
// stages of 16 KB (bulk copies completing on mbarriers, the next row's stages already in
// flight while a row is finished); 8 consumer warps copy their vectors of a stage to
// registers, free the slot, keep running row state, and finish the row after its last
// stage:
//  - top-k (k <= kSTopK): a candidate list in shared memory above a running threshold:
//    first a lower bound of the row's k-th value from the first stage (its k-th largest
//    vector maximum, or for k > 256 its k-th largest value), later the k-th largest
//    candidate value whenever the list fills; at the end the row's top k and the top-p
//    prefix within it;
//  - neither knob: the row's exact mass;
//  - top-p alone: a histogram over linear buckets (the float's exponent and leading
//    mantissa bits) of the probabilities relative to their bucket's upper edge; at the
//    end the bucket where the ordered mass crosses top_p, one more read of the row for the
//    mass above it and the crossing bucket's elements (resolved exactly).
// Renorm rows are read once more through the ring to write max(p, 0) / Z or 0. Rows the
// summaries cannot serve (top_k above kSTopK, candidate overflow, a row maximum far
// above the first stage's, an oversized crossing bucket) take a general path: radix
// selections over the whole row, read again from memory.
//
// Weights are 2^((x - M) log2(e) / T) for the row maximum M (probabilities: p); masses
// that decide a selection are sums of floor(w * 2^40); composite keys order tokens by
// value, then by lowest id. Every wait on an mbarrier is bounded by the SM clock; a wait
// that gives up raises the CTA's abort flag and sets the reported error word
// (ts_device_error); the producer then issues no more copies and waits for those in
// flight, and the consumers leave the rows they have not written, all at the next row
// boundary, before the CTA exits. A later launch starts clean.
#include <stdint.h>

#include "ts_common.cuh"
#include "ts_internal.h"
#include "ts_rowutil.cuh"
#include "ts_select.cuh"

namespace tsv {

constexpr int kRCons = 256;                  // consumer threads (8 warps)
constexpr int kRWarps = kRCons / 32;
constexpr int kRThreads = kRCons + 32;       // + the producer warp
constexpr int kRNSt = 4;                     // ring stages
constexpr int kRStageBytes = 16384;          // 1024 vectors of 16 bytes
constexpr int kRStageVecs = kRStageBytes / 16;
constexpr int kRVecs = kRStageVecs / kRCons;  // vectors per consumer thread and stage
constexpr int kRListCap = 2048;              // the first part of the candidate space
constexpr int kRSmallE = 4;                  // lists of up to 128 candidates: one warp
constexpr int kRSoft = 3072;                 // top-k list size that triggers a compaction
constexpr int kRBins = 2048;                 // top-p buckets (128 octaves)
constexpr int kRHead = 1024;                 // buckets above the first stage's maximum
constexpr int kRBPT = kRBins / kRCons;       // buckets per consumer thread at the end
constexpr int kRCrossCap = kRListCap + (2 * kRBins * 4) / 8;  // top-k or crossing elements
constexpr int kRNList = 512;                 // renorm rows a CTA can list (tiered order)
constexpr long long kRWaitCycles = 1ll << 32;  // a stage wait gives up after 2^32 SM
                                               // clock cycles (about 2 s)
constexpr double kInvFx = 1.0 / 1099511627776.0;

static __device__ unsigned int g_row_err;

enum RowKind : int { kRowGreedy = 0, kRowTopK = 1, kRowPlain = 2, kRowTopP = 3, kRowStaged = 4 };

__device__ __forceinline__ void cbar() { sel::ConsumerBar::sync(); }

// Exclusive scan of a double over the consumer threads in thread order (a fixed order of
// additions, so the result is reproducible); writes the total.
__device__ __forceinline__ double excl_scan_f64(double v, double* sc, double& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sc[w] = incl;
  cbar();
  if (w == 0) {
    double t = lane < kRWarps ? sc[lane] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < kRWarps) sc[lane] = t;
  }
  cbar();
  const double before = (w > 0) ? sc[w - 1] : 0.0;
  total = sc[kRWarps - 1];
  cbar();
  return before + (incl - v);
}

// The absolute top-p bucket coordinate of a value: floor(x log2(e) / T * 16).
__device__ __forceinline__ float babs(float v, float sl2) { return floorf(v * sl2 * 16.f); }
// The upper edge of linear probability bucket b (b <= 2032: p <= 1): the float whose bits
// are (b + 1) << 19.
__device__ __forceinline__ float rn_edge(float b) {
  return __uint_as_float(((uint32_t)b + 1u) << 19);
}

// The CTA's abort flag: raised by a wait that gave up. It is the CTA's own, so that one
// launch's error never reaches a later launch (the global word only reports).
__device__ __forceinline__ bool row_error(const int32_t* ab) {
  return *reinterpret_cast<const volatile int32_t*>(ab) != 0;
}

// Waits for the phase of `bar` with the given parity; gives up after kRWaitCycles of this
// SM's clock (monotonic) or once the CTA has aborted, raising the CTA's abort flag and
// setting the reported error word. Returns whether the phase completed.
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, int32_t* ab) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0 && (clock64() - t0 > kRWaitCycles || row_error(ab))) {
      *reinterpret_cast<volatile int32_t*>(ab) = 1;
      atomicOr(&g_row_err, 1u);
      return false;
    }
  }
}

// As bounded_wait, but only the time limit ends it: used to let the copies a CTA has
// issued land before it exits, also after an error.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kRWaitCycles) {
      atomicOr(&g_row_err, 1u);
      return;
    }
}

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

struct RowSmem {
  uint64_t full[kRNSt];
  uint64_t empty[kRNSt];
  int64_t srow[kRNSt];  // the row of each stage in the ring, -1: no more rows
  sel::Scratch sc;
  union {
    struct {
      uint64_t list[kRListCap];  // top-k candidates
      union {
        uint32_t h2[2][kRBins];       // top-p histogram: 13-bit digit sums
        uint32_t tkeys[kRStageVecs];  // the first stage's vector maxima
      } u;
    } t;
    uint64_t cross[kRCrossCap];  // top-k candidates; at the end of a top-p row the crossing
                                 // bucket's elements
  } w;
  double dscan[32];
  double tab[16];  // 2^(-q/16)
  float redf[3][kRWarps];
  int32_t redi[kRWarps];
  uint32_t lcnt, tau;
  int32_t bad;
  int32_t abort_flag;
  float base;
  float M, S1;
  int32_t am;
  float uj, uD, vx;
  int32_t owner;
  uint64_t res_u;
  double res_d;
  // renorm: this CTA's rows in the cost-tiered order, and the counts that build it
  int32_t rnrows[kRNList];
  uint32_t tcnt[3];
  uint32_t wtc[kRThreads / 32][3];
};

template <typename E, bool RN>
__global__ void __launch_bounds__(kRThreads, 2) k_row(SampleArgs a) {
  extern __shared__ __align__(128) unsigned char dsm[];
  constexpr int N = SVec<E>::N;
  constexpr int SE = kRStageBytes / (int)sizeof(E);  // elements per stage
  unsigned char* ring = dsm;
  RowSmem& sm = *reinterpret_cast<RowSmem*>(dsm + kRNSt * kRStageBytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t V = a.V;
  const int nst = (int)((V + SE - 1) / SE);  // stages per row

  if (tid == 0) {
    for (int s = 0; s < kRNSt; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kRWarps);
    }
    fence_mbar_init();
    sm.abort_flag = 0;
  }
  if (tid < 16) {
    sm.tab[tid] = exp2(-(double)tid / 16.0);
  }
  if (tid < 3) sm.tcnt[tid] = 0;
  __syncthreads();

  // Renorm rows (no workspace, so no shared counter): every CTA orders the rows the same
  // way, by cost tier (large top-k and general rows, then top-p rows, then the rest) and
  // by row within a tier, and takes every gridDim.x-th row of that order from its own
  // index on, so that each CTA gets about the same number of rows of each tier. Rows in
  // turn when the list would not fit.
  int32_t rn_n = -1;
  if constexpr (RN) {
    if (a.rows <= (int64_t)kRNList * (int64_t)gridDim.x) {
      auto tier_of = [&](int64_t r) -> int {
        const Knobs kq = row_knobs(a, r);
        if (kq.kind == kRowStaged || (kq.kind == kRowTopK && kq.k > kRCons)) return 0;
        return (kq.kind == kRowTopP) ? 1 : 2;
      };
      uint32_t cnt3[3] = {0u, 0u, 0u};
      for (int64_t r = tid; r < a.rows; r += kRThreads) ++cnt3[tier_of(r)];
      for (int t = 0; t < 3; ++t)
        if (cnt3[t]) atomicAdd(&sm.tcnt[t], cnt3[t]);
      __syncthreads();
      uint32_t run[3] = {0u, sm.tcnt[0], sm.tcnt[0] + sm.tcnt[1]};  // next position per tier
      const uint32_t lt = (1u << lane) - 1u;
      for (int64_t r0 = 0; r0 < a.rows; r0 += kRThreads) {
        const int64_t r = r0 + tid;
        const int t = (r < a.rows) ? tier_of(r) : 3;
        uint32_t before = 0;
        for (int q = 0; q < 3; ++q) {
          const uint32_t m = __ballot_sync(0xffffffffu, t == q);
          if (lane == 0) sm.wtc[warp][q] = (uint32_t)__popc(m);
          if (t == q) before = (uint32_t)__popc(m & lt);
        }
        __syncthreads();
        if (t < 3) {
          uint32_t pos = run[t] + before;
          for (int w = 0; w < warp; ++w) pos += sm.wtc[w][t];
          if (pos % gridDim.x == blockIdx.x) sm.rnrows[pos / gridDim.x] = (int32_t)r;
        }
        for (int q = 0; q < 3; ++q)
          for (int w = 0; w < kRThreads / 32; ++w) run[q] += sm.wtc[w][q];
        __syncthreads();
      }
      rn_n = (a.rows > (int64_t)blockIdx.x)
                 ? (int32_t)((a.rows - 1 - (int64_t)blockIdx.x) / gridDim.x + 1)
                 : 0;
    }
  }

  // ---- producer warp ------------------------------------------------------------------
  if (warp == kRWarps) {
    if (lane == 0) {
      uint32_t g = 0;  // stages issued so far
      bool ok = true;
      int64_t rr = blockIdx.x;
      int32_t q = 0;
      while (ok) {
        int64_t row = -1;
        if constexpr (RN) {  // renorm: the listed rows, else rows in turn
          if (rn_n >= 0) {
            row = (q < rn_n) ? (int64_t)sm.rnrows[q] : -1;
            ++q;
          } else {
            row = (rr < a.rows) ? rr : -1;
            rr += gridDim.x;
          }
        } else {
          // rows are taken from a shared counter, so that CTAs with cheap rows take more.
          // The counter runs over the rows four times, taking on each round the rows of one
          // cost tier, longest first (top-p and general rows, then large top-k, then the
          // other sampled rows, then greedy rows): the step then ends on short rows.
          const uint64_t idx = atomicAdd(reinterpret_cast<unsigned long long*>(a.ws.work), 1ull);
          if (idx < 4ull * (uint64_t)a.rows) {
            const int tier = (int)(idx / (uint64_t)a.rows);
            row = (int64_t)(idx % (uint64_t)a.rows);
            const Knobs kq = row_knobs(a, row / a.R);
            int t = 3;
            if (kq.kind == kRowTopP || kq.kind == kRowStaged) t = 0;
            else if (kq.kind == kRowTopK && kq.k > kRCons) t = 1;
            else if (kq.kind != kRowGreedy) t = 2;
            if (t != tier) continue;
          }
        }
        if (row < 0) {  // one last stage tells the consumers to stop
          const int slot = (int)(g % kRNSt);
          const uint32_t use = g / kRNSt;
          if ((use > 0 && !bounded_wait(&sm.empty[slot], (use - 1) & 1u, &sm.abort_flag)) || row_error(&sm.abort_flag)) break;
          sm.srow[slot] = -1;
          mbar_arrive_expect_tx(&sm.full[slot], 0u);
          ++g;  // (the marker is the latest use of its slot)
          break;
        }
        const unsigned char* src =
            reinterpret_cast<const unsigned char*>(a.x) + row * a.ld * (int64_t)sizeof(E);
        // top-p rows are streamed twice (the histogram, then the kept masses); renorm rows
        // once more to write the output
        const int npass = ((row_knobs(a, row / a.R).kind == kRowTopP) ? 2 : 1) + (RN ? 1 : 0);
        for (int cc = 0; cc < npass * nst; ++cc, ++g) {
          const int c = cc % nst;
          const int slot = (int)(g % kRNSt);
          const uint32_t use = g / kRNSt;
          // after an error nothing more is issued (a slot may still be in use)
          if ((use > 0 && !bounded_wait(&sm.empty[slot], (use - 1) & 1u, &sm.abort_flag)) || row_error(&sm.abort_flag)) {
            ok = false;
            break;
          }
          const int64_t nc = min((int64_t)SE, V - (int64_t)c * SE);
          const uint32_t bytes = (uint32_t)((nc * (int64_t)sizeof(E)) & ~(int64_t)15);
          sm.srow[slot] = row;
          mbar_arrive_expect_tx(&sm.full[slot], bytes);
          if (bytes)
            bulk_g2s(ring + slot * kRStageBytes, src + (int64_t)c * kRStageBytes, bytes,
                     &sm.full[slot]);
        }
      }
      // no copy of this CTA may still be in flight when it exits: wait for the last use
      // of every slot (the consumers have normally waited for them already)
      for (uint32_t h = (g > (uint32_t)kRNSt ? g - (uint32_t)kRNSt : 0u); h < g; ++h)
        drain_wait(&sm.full[h % kRNSt], (h / kRNSt) & 1u);
    }
    return;
  }

  // ---- consumers ----------------------------------------------------------------------
  const bool bf16 = sizeof(E) == 2;
  const int lowv = bf16 ? 16 : 0;  // value key bits below this follow from the higher ones
  const uint4 ninf = make_uint4(SVec<E>::kNegInfWord, SVec<E>::kNegInfWord,
                                SVec<E>::kNegInfWord, SVec<E>::kNegInfWord);
  const int64_t nvr = V / N;  // whole vectors of a row; the rest is a scalar tail
  const int64_t nvall = (V + N - 1) / N;
  const int vbase = warp * (kRVecs * 32) + lane;  // warp w: a stage's vectors 128 w ..
  uint32_t g = 0;

  for (int64_t nrow = 0; nrow < a.rows; ++nrow) {
    // the row of the next stage, or the end
    int64_t row;
    {
      const int slot = (int)(g % kRNSt);
      bounded_wait(&sm.full[slot], (g / kRNSt) & 1u, &sm.abort_flag);
      row = *reinterpret_cast<volatile int64_t*>(&sm.srow[slot]);
      // every consumer takes the same decision: the flag is read between two barriers
      cbar();
      const bool ab = row_error(&sm.abort_flag);
      cbar();
      if (ab || row < 0 || row >= a.rows) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
        break;
      }
    }
    const int64_t req = row / a.R;
    const int32_t j = (int32_t)(row % a.R);
    const Knobs kn = row_knobs(a, req);
    const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;
    const uint4* rp = reinterpret_cast<const uint4*>(xr);
    // vector vi of the stage held at sv (first element c0, nc elements, nvf whole vectors);
    // the ragged last vector of the row comes from global memory, padded with -inf
    auto stage_vec = [&](const uint4* sv, int64_t c0, int nc, int nvf, int vi) -> uint4 {
      if (vi < nvf) return sv[vi];
      if (vi > nvf || nc % N == 0) return ninf;
      uint32_t w[4] = {SVec<E>::kNegInfWord, SVec<E>::kNegInfWord, SVec<E>::kNegInfWord,
                       SVec<E>::kNegInfWord};
      for (int q = 0; q < nc - nvf * N; ++q) {
        const int64_t gi = c0 + (int64_t)vi * N + q;
        if (sizeof(E) == 2) {
          const uint32_t h = reinterpret_cast<const uint16_t*>(xr)[gi];
          w[q >> 1] = (q & 1) ? ((w[q >> 1] & 0x0000FFFFu) | (h << 16)) : ((w[q >> 1] & 0xFFFF0000u) | h);
        } else {
          w[q] = reinterpret_cast<const uint32_t*>(xr)[gi];
        }
      }
      return make_uint4(w[0], w[1], w[2], w[3]);
    };
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
    const int32_t D = a.D;
    const int32_t x = (j < D) ? a.draft_tokens[req * D + j] : -1;
    const bool xvalid = x >= 0 && (int64_t)x < V;
    const float sl2 = (kn.kind == kRowGreedy) ? 0.f : __fdiv_rn(kLog2e, kn.T);
    const int32_t k = kn.k;
    // top-p buckets, whether an element has weight, and its weight relative to the upper
    // edge of its bucket b. Logits: b = floor(16 log2 w) of w = e^(x/T). Probabilities:
    // the exponent and leading 4 mantissa bits of p (16 linear buckets an octave; the
    // float's bits order them exactly)
    auto live = [&](float v) -> bool {
      if constexpr (RN) return v > 0.f;
      else return v != -INFINITY;
    };
    auto bucket_of = [&](float v) -> float {
      if constexpr (RN) return (float)(__float_as_uint(fminf(v, 1.f)) >> 19);
      else return babs(v, sl2);
    };
    auto edge_w = [&](float v, float b) -> float {
      if constexpr (RN) return __fdividef(fminf(v, 1.f), rn_edge(b));
      else return ex2(fmaf(v, sl2, -(b + 1.f) * 0.0625f));
    };
    uint64_t* const rowslots =
        RN ? nullptr : a.ws.cand + row * a.ws.cand_splits * (int64_t)kSTopK;
    uint64_t zsum = 0;  // renorm rows without knobs: the row's exact mass
    if (tid == 0) {
      sm.lcnt = 0;
      sm.bad = 0;
      sm.tau = 0;
    }
    if (kn.kind == kRowTopP)
      for (int i = tid; i < 2 * kRBins; i += kRCons) (&sm.w.t.u.h2[0][0])[i] = 0;
    cbar();

    float bv = -INFINITY, lm = -INFINITY, ls = 0.f, lc = 0.f;
    float tl = 0.f;  // top-p renorm: this thread's tail mass
    int64_t bvi = -1;  // the row vector holding this thread's maximum (first one)

    // ---- the stages of the row -------------------------------------------------------
    for (int c = 0; c < nst; ++c, ++g) {
      const int slot = (int)(g % kRNSt);
      bounded_wait(&sm.full[slot], (g / kRNSt) & 1u, &sm.abort_flag);
      const uint4* sv = reinterpret_cast<const uint4*>(ring + slot * kRStageBytes);
      const int64_t c0 = (int64_t)c * SE;  // the stage's first element
      const int nc = (int)min((int64_t)SE, V - c0);
      const int nvf = nc / N;
      auto vec_at = [&](int vi) -> uint4 { return stage_vec(sv, c0, nc, nvf, vi); };
      // warp w takes the stage's vectors 128 w .. 128 w + 127, lane l those l + 32 u; the
      // warp frees the slot once its vectors are in registers
      uint4 rv[kRVecs];
#pragma unroll
      for (int u = 0; u < kRVecs; ++u) rv[u] = vec_at(vbase + u * 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
      float vmv[kRVecs];
#pragma unroll
      for (int u = 0; u < kRVecs; ++u) {
        const int vi = vbase + u * 32;
        const uint4 r = rv[u];
        const float vm = SVec<E>::vmax(r);
        vmv[u] = vm;
        if (vm > bv || (bvi < 0 && vi * N < nc)) {  // (an all -inf row keeps its lowest id)
          bv = vm;
          bvi = (int64_t)c * (SE / N) + vi;
        }
        if (a.logprobs && vm > -INFINITY) {
          float xv[N];
          SVec<E>::unpack(r, xv);
          const float nm = fmaxf(lm, vm);
          const float f = ex2((lm - nm) * kLog2e);
          ls *= f;
          lc *= f;
          lm = nm;
          float vs = 0.f;
#pragma unroll
          for (int q = 0; q < N; ++q) vs += ex2((xv[q] - nm) * kLog2e);
          kahan_add(ls, lc, vs);
        }
      }

      if (kn.kind == kRowTopK) {
        if (c == 0) {
          // a lower bound of the row's k-th value from the first stage: the k-th largest
          // vector maximum (k <= 256), else the stage's own k-th largest value
          uint32_t t0;
          if (k <= kRCons) {
#pragma unroll
            for (int u = 0; u < kRVecs; ++u)
              sm.w.t.u.tkeys[vbase + u * 32] = (vmv[u] > -INFINITY) ? fkey(vmv[u]) : 0u;
            cbar();
            t0 = sel::select_bound<kRCons, sel::ConsumerBar>(
                kRStageVecs, [&](int i) { return sm.w.t.u.tkeys[i]; }, (uint32_t)k, bf16 ? 2 : 4,
                sm.sc);
          } else {
            // the stage's order keys, from registers into the (still empty) candidate area
            uint32_t* skeys = reinterpret_cast<uint32_t*>(sm.w.cross);
#pragma unroll
            for (int u = 0; u < kRVecs; ++u) {
              float xv[N];
              SVec<E>::unpack(rv[u], xv);
#pragma unroll
              for (int q = 0; q < N; ++q)
                skeys[(vbase + u * 32) * N + q] = (xv[q] > -INFINITY) ? fkey(xv[q]) : 0u;
            }
            cbar();
            t0 = sel::select_bound<kRCons, sel::ConsumerBar>(
                nc, [&](int i) { return skeys[i]; }, (uint32_t)k, bf16 ? 2 : 4, sm.sc);
          }
          if (tid == 0) sm.tau = t0;
          cbar();
        }
        // the elements at or above the threshold
        const uint32_t tau = sm.tau;
        uint32_t m32 = 0;
#pragma unroll
        for (int u = 0; u < kRVecs; ++u) {
          if (!(vmv[u] > -INFINITY) || fkey(vmv[u]) < tau) continue;
          float xv[N];
          SVec<E>::unpack(rv[u], xv);
#pragma unroll
          for (int q = 0; q < N; ++q)
            if (fkey(xv[q]) >= tau && xv[q] != -INFINITY) m32 |= 1u << (u * N + q);
        }
        if (__any_sync(0xffffffffu, m32 != 0u)) {
          const uint32_t pos = warp_reserve(&sm.lcnt, (uint32_t)__popc(m32), lane);
          append_candidates<E>(m32, rv, (int)c0, vbase, pos, sm.w.cross, (uint32_t)kRCrossCap);
        }
      } else if (RN && kn.kind == kRowPlain) {
        // renorm without knobs: the row's exact mass
#pragma unroll
        for (int u = 0; u < kRVecs; ++u) {
          float xv[N];
          SVec<E>::unpack(rv[u], xv);
#pragma unroll
          for (int q = 0; q < N; ++q) zsum += fixw(fminf(fmaxf(xv[q], 0.f), 1.f));
        }
      } else if (kn.kind == kRowPlain) {
        // warp w's 128 vectors of the stage: their mass relative to their own maximum, the
        // draft token left out
        float em = fmaxf(fmaxf(vmv[0], vmv[1]), fmaxf(vmv[2], vmv[3]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) em = fmaxf(em, __shfl_xor_sync(0xffffffffu, em, o));
        float s = 0.f;
        if (em > -INFINITY) {
#pragma unroll
          for (int u = 0; u < kRVecs; ++u) {
            const int vi = vbase + u * 32;
            float xv[N];
            SVec<E>::unpack(rv[u], xv);
#pragma unroll
            for (int q = 0; q < N; ++q) {
              const float w = ex2((xv[q] - em) * sl2);
              s += (c0 + (int64_t)vi * N + q == (int64_t)x) ? 0.f : w;
            }
          }
        }
        s = warp_sum_f32(s);
        if (lane == 0)
          rowslots[(int64_t)c * kRWarps + warp] =
              ((uint64_t)__float_as_uint(em) << 32) | __float_as_uint(s);
      } else if (kn.kind == kRowTopP) {
        if (c == 0) {
          // the bucket window: kRHead buckets above the first stage's maximum, kRBins down
          float m = fmaxf(fmaxf(vmv[0], vmv[1]), fmaxf(vmv[2], vmv[3]));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) sm.redf[0][warp] = m;
          cbar();
          if (tid == 0) {
            float mm = sm.redf[0][0];
            for (int w = 1; w < kRWarps; ++w) mm = fmaxf(mm, sm.redf[0][w]);
            sm.base = live(mm) ? bucket_of(mm) + (float)kRHead : 0.f;
            if (!live(mm)) sm.bad = 1;
          }
          cbar();
        }
        const float base = sm.base;
        // probabilities: vectors lighter than 2^-24 of this thread's running maximum skip
        // the histogram and add to the thread's tail sum. Their total is below V 2^-24 of
        // the row's mass, so for top_p <= 1 - V 2^-24 the crossing lies above them; the
        // finish checks that it does and otherwise leaves the row to the general path.
        // Vectors below 2^-41 of it weigh nothing in the fixed-point masses (2^-40 units)
        // and are skipped.
        const float tail_below = bv * 5.9604644775390625e-8f;
        const float zero_below = bv * 4.547473508864641e-13f;
        bool out = false;
#pragma unroll
        for (int u = 0; u < kRVecs; ++u) {
          if (!live(vmv[u]) || (RN && vmv[u] < zero_below)) continue;
          float xv[N];
          SVec<E>::unpack(rv[u], xv);
          if (RN && vmv[u] < tail_below) {
#pragma unroll
            for (int q = 0; q < N; ++q)
              if (live(xv[q])) tl += xv[q];
            continue;
          }
#pragma unroll
          for (int q = 0; q < N; ++q) {
            const float v = xv[q];
            if (!live(v)) continue;
            const float b = bucket_of(v);
            const float idx = base - b;
            if (idx < 0.f) {
              out = true;  // above the window
              continue;
            }
            if (idx >= (float)kRBins) continue;  // below 2^-64 of the maximum: negligible
            // the weight relative to its bucket's upper edge, in (2^-1/16, 1], 25 bits
            const uint32_t r = __float2uint_rz(edge_w(v, b) * 33554432.f);
            const int ib = (int)idx;
            atomicAdd(&sm.w.t.u.h2[0][ib], r & 0x1FFFu);
            atomicAdd(&sm.w.t.u.h2[1][ib], r >> 13);
          }
        }
        if (out) sm.bad = 1;
      }

      // the candidate count is checked every few stages (and after the last): a stage adds
      // few candidates once the threshold has settled. Large k is checked every stage: a
      // first-stage threshold at k = 1000 passes a quarter of a 4096-entry fp32 stage, so
      // two stages could fill the list past its capacity
      const int cstride = (k > kRCons) ? 1 : 8;
      const uint32_t soft = (k > kRCons) ? (uint32_t)kRListCap : (uint32_t)kRSoft;
      if (kn.kind == kRowTopK && ((c + 1) % cstride == 0 || c == nst - 1)) {
        cbar();
        const uint32_t cnt = sm.lcnt;
        if (cnt > (uint32_t)kRCrossCap) {
          if (tid == 0) {
            sm.bad = 1;
            sm.tau = 0xFFFFFFFFu;  // stop collecting; the staged kernel takes the row
            sm.lcnt = 0;
          }
          cbar();
        } else if (cnt > soft) {
          // compaction: keep the candidates at or above the k-th largest value
          const uint32_t vk = sel::select_bound<kRCons, sel::ConsumerBar>(
              (int)cnt, [&](int i) { return (uint32_t)(sm.w.cross[i] >> kIdxBits); },
              (uint32_t)k, bf16 ? 2 : 4, sm.sc);
          // in two halves, so that a thread holds at most 8 candidates: survivors of the
          // first half go below 2048, the second half is read before it is overwritten
          if (tid == 0) sm.tau = max(sm.tau, vk);
          for (int half = 0; half < 2; ++half) {
            uint64_t keep[kRListCap / kRCons];
#pragma unroll
            for (int m = 0; m < kRListCap / kRCons; ++m) {
              const uint32_t i = (uint32_t)(half * kRListCap + m * kRCons + tid);
              keep[m] = (i < cnt) ? sm.w.cross[i] : 0ull;
            }
            cbar();
            if (half == 0 && tid == 0) sm.lcnt = 0;
            cbar();
#pragma unroll
            for (int m = 0; m < kRListCap / kRCons; ++m)
              if ((uint32_t)(keep[m] >> kIdxBits) >= vk && keep[m] != 0ull)
                sm.w.cross[atomicAdd(&sm.lcnt, 1u)] = keep[m];
            cbar();
          }
          cbar();
          if (sm.lcnt > soft) {  // ties at the k-th value fill the list
            if (tid == 0) {
              sm.bad = 1;
              sm.tau = 0xFFFFFFFFu;
              sm.lcnt = 0;
            }
          }
          cbar();
        }
      }
    }

    // ---- the row's statistics ---------------------------------------------------------
    ls += lc;
    int32_t bi = INT32_MAX;
    if (bvi >= 0) {  // the first element of the best vector equal to the maximum
      float xv[N];
      load_vec(bvi, xv);
      int qb = N - 1;
#pragma unroll
      for (int q = N - 1; q >= 0; --q)
        if (xv[q] == bv) qb = q;
      bi = (int32_t)(bvi * N + qb);
    }
    {
      float v = bv, m = lm, s = ls;
      int32_t i = bi;
      warp_argmax(v, i);
      warp_lse(m, s);
      if (lane == 0) {
        sm.redf[0][warp] = v;
        sm.redf[1][warp] = m;
        sm.redf[2][warp] = s;
        sm.redi[warp] = i;
      }
      cbar();
      if (warp == 0) {
        v = lane < kRWarps ? sm.redf[0][lane] : -INFINITY;
        m = lane < kRWarps ? sm.redf[1][lane] : -INFINITY;
        s = lane < kRWarps ? sm.redf[2][lane] : 0.f;
        i = lane < kRWarps ? sm.redi[lane] : INT32_MAX;
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
      cbar();
    }
    const float M = sm.M;
    const int32_t am = sm.am;
    const float uj = sm.uj, uD = sm.uD, vx = sm.vx;
    const bool bad = sm.bad != 0;
    auto wfn = [&](float v) -> uint64_t {
      if constexpr (RN) return fixw(fminf(fmaxf(v, 0.f), 1.f));
      else return fixw(ex2((v - M) * sl2));
    };
    auto wcomp = [&](uint64_t cc) -> uint64_t {
      return wfn(key_to_value((uint32_t)(cc >> kIdxBits)));
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
            lp = (SVec<E>::at(xj, t) - __ldcg(&a.ws.rowres[rj].M)) -
                 logf(__ldcg(&a.ws.rowres[rj].S));
          }
          a.logprobs[rj] = lp;
        }
      }
      a.accept_length[req] = js + 1;
    };
    // Warp 0 walks the 32 vectors from row vector v0 (one a lane) and returns the first
    // element at which the running weight exceeds tf (the last element with weight if
    // none does, e.g. by rounding; -1 if no element has weight).
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
    // The same over the kRVecs * 32 vectors from v0, a step of 32 at a time.
    auto walk_range = [&](int64_t v0, float tf, auto&& wgt) -> int32_t {
      int lastu = -1;
      for (int u = 0; u < kRVecs; ++u) {
        const int64_t vi = v0 + u * 32 + lane;
        float vs = 0.f;
        if (vi < nvall) {
          float xv[N];
          load_vec(vi, xv);
#pragma unroll
          for (int q = 0; q < N; ++q) vs += wgt(xv[q], vi * N + q);
        }
        const float tot = warp_sum_f32(vs);
        if (tot > tf) return walk_step(v0 + u * 32, tf, wgt);
        if (tot > 0.f) {
          tf -= tot;
          lastu = u;
        }
      }
      // rounding: the last element with weight
      return (lastu >= 0) ? walk_step(v0 + lastu * 32, INFINITY, wgt) : -1;
    };

    // The general path for the rows the streamed summaries cannot serve (top_k above
    // kSTopK, candidate overflow, a maximum above the bucket window, a crossing bucket too
    // large): radix selections over the whole row, read again from memory for every
    // digit, in the order top-k, top-p within it, then the draw in token-id order.
    auto general_select = [&](uint64_t& Cout, uint64_t& Zout) {
      const int n = (int)V;
      auto gitem = [&](int i) -> uint64_t {
        return comp_key(fkey(SVec<E>::at(xr, i)), (uint32_t)i);
      };
      auto gmass = [&](uint64_t c0) -> uint64_t {
        uint64_t sum = 0;
        for (int i = tid; i < n; i += kRCons) {
          const uint64_t cc = gitem(i);
          if (cc >= c0) sum += wcomp(cc);
        }
        uint64_t tot;
        (void)sel::excl_scan<kRCons, sel::ConsumerBar>(sum, sm.sc, tot);
        return tot;
      };
      const bool tk = k > 0 && (int64_t)k < V;
      uint64_t C = 1;  // every composite key is at least 1
      if (tk)
        C = sel::radix_adaptive<kRCons, false, sel::ConsumerBar>(
            n, gitem, 1ull, (uint64_t)k, [](uint64_t) { return (uint64_t)1; }, lowv, sm.sc);
      uint64_t Z = gmass(C);
      if (kn.tp < 1.f) {
        const double want = ceil((double)kn.tp * (double)Z);
        const uint64_t P = (want > (double)Z) ? Z : (uint64_t)want;
        C = sel::radix_adaptive<kRCons, true, sel::ConsumerBar>(n, gitem, C, P, wcomp, lowv, sm.sc);
        Z = gmass(C);
      }
      Cout = C;
      Zout = Z;
    };
    auto general = [&]() {
      const int n = (int)V;
      auto gitem = [&](int i) -> uint64_t {
        return comp_key(fkey(SVec<E>::at(xr, i)), (uint32_t)i);
      };
      uint64_t C, Z;
      general_select(C, Z);
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
        uint64_t gsel = 0;
        (void)sel::radix<kRCons, true, sel::ConsumerBar>(
            n, gitem, C, t + 1,
            [&](uint64_t cc) { return ((int32_t)comp_token(cc) == x) ? 0ull : wcomp(cc); },
            idx_sh, 3, sm.sc, &gsel);
        tok = (int32_t)comp_token(gsel);
      }
      if (tid == 0) finish_row(tok, acc);
    };

    // the consumers' sum of a float (top-p tail masses)
    auto consumer_sum = [&](float v) -> double {
      v = warp_sum_f32(v);
      if (lane == 0) sm.redf[1][warp] = v;
      cbar();
      double t = 0.0;
      for (int w = 0; w < kRWarps; ++w) t += (double)sm.redf[1][w];
      cbar();
      return t;
    };

    // ---- finish the row -----------------------------------------------------------------
    if constexpr (RN) {
      // renorm: the kept set (a threshold composite C, and for top-p rows the bucket rule)
      // and its exact mass Z, then one more pass that writes max(p, 0) / Z or 0
      uint64_t C = 0, Z = 0;
      bool bucket_rule = false;
      float fbk = 0.f;
      const float base = sm.base;
      if (kn.kind == kRowTopP) {
        bool active = !bad && kn.tp > 0.f;
        int bstar = -1;
        double pre = 0.0, P = 0.0;
        if (active) {
          // mass of bucket i = (digit sums) 2^-25 (upper edge of bucket base - i)
          double hm[kRBPT];
          double hsum = 0.0;
#pragma unroll
          for (int q = 0; q < kRBPT; ++q) {
            const int i = kRBPT * tid + q;
            const uint64_t h = (uint64_t)sm.w.t.u.h2[0][i] + ((uint64_t)sm.w.t.u.h2[1][i] << 13);
            hm[q] = h ? (double)h * (1.0 / 33554432.0) * (double)rn_edge(base - (float)i) : 0.0;
            hsum += hm[q];
          }
          const double ttail = consumer_sum(tl);
          double Zt;
          const double hex = excl_scan_f64(hsum, sm.dscan, Zt);
          P = (double)kn.tp * (Zt + ttail);
          if (tid == 0) sm.owner = -1;
          cbar();
          double acc_b = hex;
#pragma unroll
          for (int q = 0; q < kRBPT; ++q) {
            if (hm[q] > 0.0 && acc_b < P && P <= acc_b + hm[q]) {
              sm.owner = kRBPT * tid + q;
              sm.res_d = acc_b;
            }
            acc_b += hm[q];
          }
          cbar();
          bstar = sm.owner;
          pre = sm.res_d;
          // (a crossing among the tail's weights is left to the general path)
          active = bstar >= 0 &&
                   (ttail == 0.0 ||
                    __uint_as_float((uint32_t)(base - (float)bstar) << 19) >= M * 1.1920929e-7f);
        }
        if (tid == 0) sm.lcnt = 0;
        cbar();
        // the second pass: the exact mass above the crossing bucket, and its elements
        const float fb = (float)bstar;
        uint64_t zab = 0;
        for (int c = 0; c < nst; ++c, ++g) {
          const int slot = (int)(g % kRNSt);
          bounded_wait(&sm.full[slot], (g / kRNSt) & 1u, &sm.abort_flag);
          const int64_t c0 = (int64_t)c * SE;
          uint4 rv[kRVecs];
          if (active) {
            const uint4* sv = reinterpret_cast<const uint4*>(ring + slot * kRStageBytes);
            const int nc = (int)min((int64_t)SE, V - c0);
            const int nvf = nc / N;
#pragma unroll
            for (int u = 0; u < kRVecs; ++u) rv[u] = stage_vec(sv, c0, nc, nvf, vbase + u * 32);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.empty[slot]);
          if (active) {
            uint32_t mk[kRVecs];
            uint32_t nsel = 0;
#pragma unroll
            for (int u = 0; u < kRVecs; ++u) {
              mk[u] = 0;
              const float vm = SVec<E>::vmax(rv[u]);
              if (!live(vm) || base - bucket_of(vm) > fb) continue;  // all lighter
              float xv[N];
              SVec<E>::unpack(rv[u], xv);
#pragma unroll
              for (int q = 0; q < N; ++q) {
                const float v = xv[q];
                if (!live(v)) continue;
                const float idx = base - bucket_of(v);
                if (idx < fb) zab += wfn(v);
                else if (idx == fb && wfn(v) > 0) mk[u] |= 1u << q;
              }
              nsel += (uint32_t)__popc(mk[u]);
            }
            if (__any_sync(0xffffffffu, nsel != 0)) {
              const uint32_t pos = warp_reserve(&sm.lcnt, nsel, lane);
              uint32_t m32 = 0;
#pragma unroll
              for (int u = 0; u < kRVecs; ++u) m32 |= mk[u] << (u * N);
              append_candidates<E>(m32, rv, (int)c0, vbase, pos, sm.w.cross, (uint32_t)kRCrossCap);
            }
          }
        }
        cbar();
        const uint32_t cnt = sm.lcnt;
        if (kn.tp <= 0.f) {  // only the argmax is kept
          C = comp_key(fkey(M), (uint32_t)am);
          Z = wfn(M);
        } else if (!active || cnt > (uint32_t)kRCrossCap || cnt == 0) {
          general_select(C, Z);
        } else {
          const double want = ceil((P - pre) * 1099511627776.0);
          const uint64_t Pb = want < 1.0 ? 1ull : (uint64_t)want;
          C = sel::radix_adaptive<kRCons, true, sel::ConsumerBar>(
              (int)cnt, [&](int i) { return sm.w.cross[i]; }, 1ull, Pb, wcomp, lowv, sm.sc);
          uint64_t mine = zab;
          for (uint32_t i = tid; i < cnt; i += kRCons) {
            const uint64_t cc = sm.w.cross[i];
            if (cc >= C) mine += wcomp(cc);
          }
          (void)sel::excl_scan<kRCons, sel::ConsumerBar>(mine, sm.sc, Z);
          bucket_rule = true;
          fbk = fb;
        }
      } else if (bad || kn.kind == kRowStaged) {
        general_select(C, Z);
      } else if (kn.kind == kRowTopK) {
        const int nl = (int)sm.lcnt;
        auto item = [&](int i) { return sm.w.cross[i]; };
        const uint64_t Ck = sel::radix_adaptive<kRCons, false, sel::ConsumerBar>(
            nl, item, 1ull, (uint64_t)k, [](uint64_t) { return (uint64_t)1; }, lowv, sm.sc);
        auto mass_from = [&](uint64_t c0) -> uint64_t {
          uint64_t sum = 0;
          for (int i = tid; i < nl; i += kRCons) {
            const uint64_t cc = sm.w.cross[i];
            if (cc >= c0) sum += wcomp(cc);
          }
          uint64_t tot;
          (void)sel::excl_scan<kRCons, sel::ConsumerBar>(sum, sm.sc, tot);
          return tot;
        };
        C = Ck;
        Z = mass_from(Ck);
        if (kn.tp < 1.f) {
          const double want = ceil((double)kn.tp * (double)Z);
          const uint64_t P = (want > (double)Z) ? Z : (uint64_t)want;
          C = sel::radix_adaptive<kRCons, true, sel::ConsumerBar>(nl, item, Ck, P, wcomp, lowv, sm.sc);
          Z = mass_from(C);
        }
      } else {  // no knobs: everything is kept
        (void)sel::excl_scan<kRCons, sel::ConsumerBar>(zsum, sm.sc, Z);
      }
      // a wait that gave up: the row (and the rest) is left unwritten
      {
        cbar();
        const bool ab = row_error(&sm.abort_flag);
        cbar();
        if (ab) break;
      }
      // the write pass
      const float scale = (Z > 0) ? __fdiv_rn(kFx, __ull2float_rn(Z)) : 0.f;
      float* orow = a.out + row * V;
      const bool vout = ((reinterpret_cast<uintptr_t>(orow) & 15) == 0);
      for (int c = 0; c < nst; ++c, ++g) {
        const int slot = (int)(g % kRNSt);
        bounded_wait(&sm.full[slot], (g / kRNSt) & 1u, &sm.abort_flag);
        const uint4* sv = reinterpret_cast<const uint4*>(ring + slot * kRStageBytes);
        const int64_t c0 = (int64_t)c * SE;
        const int nc = (int)min((int64_t)SE, V - c0);
        const int nvf = nc / N;
        uint4 rw[kRVecs];
#pragma unroll
        for (int u = 0; u < kRVecs; ++u) rw[u] = stage_vec(sv, c0, nc, nvf, vbase + u * 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
#pragma unroll
        for (int u = 0; u < kRVecs; ++u) {
          const int vi = vbase + u * 32;
          if (vi * N >= nc) continue;
          float xv[N], y[N];
          SVec<E>::unpack(rw[u], xv);
#pragma unroll
          for (int q = 0; q < N; ++q) {
            const float v = xv[q];
            const int64_t gi = c0 + (int64_t)vi * N + q;
            bool kp = comp_key(fkey(v), (uint32_t)gi) >= C;
            if (bucket_rule && live(v)) {
              const float idx = base - bucket_of(v);
              kp = idx < fbk || (idx == fbk && kp);
            }
            y[q] = kp ? fmaxf(v, 0.f) * scale : 0.f;
          }
          const int64_t e0 = c0 + (int64_t)vi * N;
          if (vout && vi < nvf) {
            __stcs(reinterpret_cast<float4*>(orow + e0), make_float4(y[0], y[1], y[2], y[3]));
          } else {
            for (int q = 0; q < N; ++q)
              if (e0 + q < V) orow[e0 + q] = y[q];
          }
        }
      }
    } else if (kn.kind == kRowTopP) {
      // top-p alone: bucket masses (thread t holds buckets 8t .. 8t + 7), the crossing
      // bucket, then the second pass over the row
      const float base = sm.base;
      bool active = !bad && kn.tp > 0.f;
      int bstar = -1;
      double pre = 0.0, P = 0.0;
      if (active) {
        // mass of bucket i = (digit sums) 2^-25 2^((base - i + 1)/16 - M log2(e)/T)
        const double F = exp2((double)(base + 1.f) / 16.0 - (double)M * (double)sl2) *
                         (1.0 / 33554432.0);
        double hm[kRBPT];
        double hsum = 0.0;
#pragma unroll
        for (int q = 0; q < kRBPT; ++q) {
          const int i = kRBPT * tid + q;
          const uint64_t h = (uint64_t)sm.w.t.u.h2[0][i] + ((uint64_t)sm.w.t.u.h2[1][i] << 13);
          hm[q] = ldexp((double)h * F * sm.tab[i & 15], -(i >> 4));
          hsum += hm[q];
        }
        double Zt;
        const double hex = excl_scan_f64(hsum, sm.dscan, Zt);
        P = (double)kn.tp * Zt;
        if (tid == 0) sm.owner = -1;
        cbar();
        double acc_b = hex;
#pragma unroll
        for (int q = 0; q < kRBPT; ++q) {
          if (hm[q] > 0.0 && acc_b < P && P <= acc_b + hm[q]) {
            sm.owner = kRBPT * tid + q;
            sm.res_d = acc_b;
          }
          acc_b += hm[q];
        }
        cbar();
        bstar = sm.owner;
        pre = sm.res_d;
        active = bstar >= 0;
      }
      if (tid == 0) sm.lcnt = 0;
      cbar();
      // the second pass: per (stage, warp) range of 128 vectors the mass of the whole
      // buckets above the crossing one (the draft token left out), and the crossing
      // bucket's elements; the stages are consumed in any case
      const float fb = (float)bstar;
      for (int c = 0; c < nst; ++c, ++g) {
        const int slot = (int)(g % kRNSt);
        bounded_wait(&sm.full[slot], (g / kRNSt) & 1u, &sm.abort_flag);
        if (active) {
          const uint4* sv = reinterpret_cast<const uint4*>(ring + slot * kRStageBytes);
          const int64_t c0 = (int64_t)c * SE;
          const int nc = (int)min((int64_t)SE, V - c0);
          const int nvf = nc / N;
          float s = 0.f;
#pragma unroll
          for (int u = 0; u < kRVecs; ++u) {
            const int vi = vbase + u * 32;
            const uint4 r = stage_vec(sv, c0, nc, nvf, vi);
            const float vm = SVec<E>::vmax(r);
            if (!(vm > -INFINITY) || base - babs(vm, sl2) > fb) continue;  // all lighter
            float xv[N];
            SVec<E>::unpack(r, xv);
#pragma unroll
            for (int q = 0; q < N; ++q) {
              const float v = xv[q];
              if (v == -INFINITY) continue;
              const float idx = base - babs(v, sl2);
              const int64_t gi = c0 + (int64_t)vi * N + q;
              if (idx < fb) {
                if (gi != (int64_t)x) s += ex2((v - M) * sl2);
              } else if (idx == fb) {
                // (a candidate of zero fixed-point weight sorts after every positive one,
                // so it never moves the mass cut)
                const uint32_t pos = atomicAdd(&sm.lcnt, 1u);
                if (pos < (uint32_t)kRCrossCap) sm.w.cross[pos] = comp_key(fkey(v), (uint32_t)gi);
              }
            }
          }
          const uint64_t f = fixw(warp_sum_f32(s));
          if (lane == 0) rowslots[(int64_t)c * kRWarps + warp] = f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
      }
      cbar();
      const uint32_t cnt = sm.lcnt;
      if (kn.tp <= 0.f) {  // only the argmax is kept
        if (tid == 0) finish_row(am, (j < D && x == am) ? 1 : 0);
      } else if (!active || cnt > (uint32_t)kRCrossCap || cnt == 0) {
        general();
      } else {
        const double want = ceil((P - pre) * 1099511627776.0);
        const uint64_t Pb = want < 1.0 ? 1ull : (uint64_t)want;
        const uint64_t C = sel::radix_adaptive<kRCons, true, sel::ConsumerBar>(
            (int)cnt, [&](int i) { return sm.w.cross[i]; }, 1ull, Pb, wcomp, lowv, sm.sc);
        // the kept elements of the crossing bucket join their ranges
        for (uint32_t i = tid; i < cnt; i += kRCons) {
          const uint64_t cc = sm.w.cross[i];
          const uint32_t gi = comp_token(cc);
          if (cc >= C && (int32_t)gi != x)
            atomicAdd(reinterpret_cast<unsigned long long*>(rowslots + (gi / N) / (kRVecs * 32)),
                      (unsigned long long)wcomp(cc));
        }
        cbar();
        auto kept = [&](float v, int64_t gi) -> bool {
          const float idx = base - babs(v, sl2);
          if (idx < fb) return true;
          return idx == fb && comp_key(fkey(v), (uint32_t)gi) >= C;
        };
        uint64_t wx = 0;
        if (xvalid && kept(vx, x)) wx = wfn(vx);
        const int64_t E_ = (int64_t)nst * kRWarps;
        const int64_t per = (E_ + kRCons - 1) / kRCons;
        const int64_t e0 = min(E_, (int64_t)tid * per), e1 = min(E_, e0 + per);
        uint64_t mine = 0;
        for (int64_t e = e0; e < e1; ++e) mine += __ldcg(rowslots + e);
        uint64_t Zr;
        const uint64_t ex = sel::excl_scan<kRCons, sel::ConsumerBar>(mine, sm.sc, Zr);
        const int32_t acc = (j < D) && ((double)uj * (double)(Zr + wx) < (double)wx) ? 1 : 0;
        if (Zr == 0) {
          if (tid == 0) finish_row((wx > 0) ? x : am, acc);
        } else {
          uint64_t t = (uint64_t)((double)uD * (double)Zr);
          if (t >= Zr) t = Zr - 1;
          if (mine > 0 && ex <= t && t < ex + mine) {
            uint64_t accu = ex;
            int64_t esel = e1 - 1;
            for (int64_t e = e0; e < e1; ++e) {
              const uint64_t m = __ldcg(rowslots + e);
              if (t < accu + m) {
                esel = e;
                break;
              }
              accu += m;
            }
            sm.res_u = (uint64_t)esel;
            sm.res_d = (double)(t - accu) * kInvFx;
          }
          cbar();
          if (warp == 0) {
            const int64_t es = (int64_t)sm.res_u;
            const int64_t v0 = (es / kRWarps) * (SE / N) + (es % kRWarps) * (kRVecs * 32);
            const int32_t tok = walk_range(v0, (float)sm.res_d, [&](float v, int64_t gi) -> float {
              if (gi == (int64_t)x || v == -INFINITY || !kept(v, gi)) return 0.f;
              return ex2((v - M) * sl2);
            });
            if (lane == 0) finish_row(tok >= 0 ? tok : am, acc);
          }
        }
      }
    } else if (kn.kind == kRowGreedy) {
      if (tid == 0) finish_row(am, (j < D && x == am) ? 1 : 0);
    } else if (bad || kn.kind == kRowStaged) {
      general();
    } else if (kn.kind == kRowTopK && (int)sm.lcnt <= 32 * kRSmallE) {
      // few candidates: one warp finishes the row (sorts in registers, scans by shuffles)
      if (warp == 0) {
        const int nl = (int)sm.lcnt;
        uint64_t v[kRSmallE], w[kRSmallE];
#pragma unroll
        for (int e = 0; e < kRSmallE; ++e) {
          const int i = e * 32 + lane;
          v[e] = (i < nl) ? sm.w.cross[i] : 0ull;
        }
        warp_bitonic_asc(v);  // element i has descending rank 32 E - 1 - i
#pragma unroll
        for (int e = 0; e < kRSmallE; ++e) {
          const int r = 32 * kRSmallE - 1 - (e * 32 + lane);
          w[e] = (v[e] != 0ull && r < k) ? wcomp(v[e]) : 0ull;
        }
        uint64_t incl[kRSmallE];
#pragma unroll
        for (int e = 0; e < kRSmallE; ++e) incl[e] = w[e];
        const uint64_t Zk = warp_scan_incl(incl);
        // top-p within the top k: rank r kept iff r = 0 or the mass before it is below P
        uint64_t P = Zk;
        if (kn.tp < 1.f) {
          const double want = ceil((double)kn.tp * (double)Zk);
          P = (want > (double)Zk) ? Zk : (uint64_t)want;
        }
        uint64_t Z = 0, wx = 0;
        bool kept[kRSmallE];
#pragma unroll
        for (int e = 0; e < kRSmallE; ++e) {
          const int r = 32 * kRSmallE - 1 - (e * 32 + lane);
          const uint64_t before = Zk - incl[e];
          kept[e] = v[e] != 0ull && r < k && (r == 0 || before < P);
          if (kept[e]) {
            Z += w[e];
            if ((int32_t)comp_token(v[e]) == x) wx = w[e];
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          Z += __shfl_xor_sync(0xffffffffu, Z, o);
          wx += __shfl_xor_sync(0xffffffffu, wx, o);
        }
        const int32_t acc = (j < D) && ((double)uj * (double)Z < (double)wx) ? 1 : 0;
        const uint64_t Zr = Z - wx;
        int32_t tok = (wx > 0) ? x : am;
        if (Zr > 0) {
          uint64_t t = (uint64_t)((double)uD * (double)Zr);
          if (t >= Zr) t = Zr - 1;
          // the kept tokens in id order, the draft token without weight
          uint64_t key2[kRSmallE], cw[kRSmallE];
#pragma unroll
          for (int e = 0; e < kRSmallE; ++e)
            key2[e] = kept[e] ? (((uint64_t)comp_token(v[e]) << 32) | (uint32_t)(v[e] >> kIdxBits))
                              : ~0ull;
          warp_bitonic_asc(key2);
#pragma unroll
          for (int e = 0; e < kRSmallE; ++e)
            cw[e] = (key2[e] != ~0ull && (int32_t)(key2[e] >> 32) != x)
                        ? wfn(key_to_value((uint32_t)key2[e]))
                        : 0ull;
          (void)warp_scan_incl(cw);
          // the first token whose inclusive prefix mass exceeds t
          int32_t f = INT32_MAX;
#pragma unroll
          for (int e = 0; e < kRSmallE; ++e) {
            const uint64_t wi = (key2[e] != ~0ull && (int32_t)(key2[e] >> 32) != x)
                                    ? wfn(key_to_value((uint32_t)key2[e]))
                                    : 0ull;
            if (wi > 0 && cw[e] > t && cw[e] - wi <= t) f = (int32_t)(key2[e] >> 32);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) f = min(f, __shfl_xor_sync(0xffffffffu, f, o));
          if (f != INT32_MAX) tok = f;
        }
        if (lane == 0) finish_row(tok, acc);
      }
    } else if (kn.kind == kRowTopK) {
      const int nl = (int)sm.lcnt;
      auto item = [&](int i) { return sm.w.cross[i]; };
      const uint64_t Ck = sel::radix_adaptive<kRCons, false, sel::ConsumerBar>(
          nl, item, 1ull, (uint64_t)k, [](uint64_t) { return (uint64_t)1; }, lowv, sm.sc);
      auto mass_from = [&](uint64_t c0) -> uint64_t {
        uint64_t sum = 0;
        for (int i = tid; i < nl; i += kRCons) {
          const uint64_t cc = sm.w.cross[i];
          if (cc >= c0) sum += wcomp(cc);
        }
        uint64_t tot;
        (void)sel::excl_scan<kRCons, sel::ConsumerBar>(sum, sm.sc, tot);
        return tot;
      };
      uint64_t C = Ck, Z = mass_from(Ck);
      if (kn.tp < 1.f) {
        const double want = ceil((double)kn.tp * (double)Z);
        const uint64_t P = (want > (double)Z) ? Z : (uint64_t)want;
        C = sel::radix_adaptive<kRCons, true, sel::ConsumerBar>(nl, item, Ck, P, wcomp, lowv, sm.sc);
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
        uint64_t gsel = 0;
        (void)sel::radix<kRCons, true, sel::ConsumerBar>(
            nl, item, C, t + 1,
            [&](uint64_t cc) { return ((int32_t)comp_token(cc) == x) ? 0ull : wcomp(cc); },
            idx_sh, 3, sm.sc, &gsel);
        tok = (int32_t)comp_token(gsel);
      }
      if (tid == 0) finish_row(tok, acc);
    } else if (kn.kind == kRowPlain) {
      // the warp steps scaled to the row maximum, in token order
      const int64_t E_ = (int64_t)nst * kRWarps;
      const int64_t per = (E_ + kRCons - 1) / kRCons;
      const int64_t e0 = min(E_, (int64_t)tid * per), e1 = min(E_, e0 + per);
      auto entry = [&](int64_t e, float* emax) -> double {
        const uint64_t p = __ldcg(rowslots + e);
        const float em = __uint_as_float((uint32_t)(p >> 32));
        *emax = em;
        if (!(em > -INFINITY)) return 0.0;
        return (double)__uint_as_float((uint32_t)p) * (double)ex2((em - M) * sl2);
      };
      double mine = 0.0;
      float emd;
      for (int64_t e = e0; e < e1; ++e) mine += entry(e, &emd);
      double Zr;
      const double ex = excl_scan_f64(mine, sm.dscan, Zr);
      const double wx = xvalid ? (double)ex2((vx - M) * sl2) : 0.0;
      const int32_t acc = (j < D) && ((double)uj * (Zr + wx) < wx) ? 1 : 0;
      if (!(Zr > 0.0)) {
        if (tid == 0) finish_row((wx > 0.0) ? x : am, acc);
      } else {
        const double t = (double)uD * Zr;
        if (tid == 0) sm.owner = -1;
        cbar();
        if (mine > 0.0 && ex <= t && t < ex + mine) sm.owner = tid;
        cbar();
        if (sm.owner < 0) {  // rounding: the last thread with mass
          if (mine > 0.0) atomicMax(&sm.owner, tid);
          cbar();
        }
        if (tid == sm.owner) {
          double accd = ex, rs = 0.0, rlast = 0.0;
          int64_t es = -1, elast = -1;
          for (int64_t e = e0; e < e1; ++e) {
            float em;
            const double m = entry(e, &em);
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
          float em;
          const double m = entry(es, &em);
          sm.res_u = (uint64_t)es;
          sm.redf[0][0] = em;
          // the residual in the step's own weight units (relative to its maximum)
          sm.res_d = (t - rs) / (m > 0.0 ? (double)ex2((em - M) * sl2) : 1.0);
        }
        cbar();
        if (warp == 0) {
          const int64_t es = (int64_t)sm.res_u;
          const float em = sm.redf[0][0];
          const int64_t v0 = (es / kRWarps) * (SE / N) + (es % kRWarps) * (kRVecs * 32);
          const int32_t tok = walk_range(v0, (float)sm.res_d, [&](float v, int64_t gi) -> float {
            return (gi == (int64_t)x || v == -INFINITY) ? 0.f : ex2((v - em) * sl2);
          });
          if (lane == 0) finish_row(tok >= 0 ? tok : am, acc);
        }
      }
    }
    cbar();  // the row's shared state is free for the next row
  }
  // the last CTA to finish leaves the row counter at zero for the next call
  if (!RN && tid == 0) {
    __threadfence();
    if (atomicAdd(&a.ws.work[2], 1u) == gridDim.x - 1) {
      *reinterpret_cast<unsigned long long*>(a.ws.work) = 0ull;
      a.ws.work[2] = 0u;
    }
  }
}

namespace {
template <typename E, bool RN>
cudaError_t launch_row_kernel(const SampleArgs& a, cudaStream_t s) {
  int dev = 0, nsm = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t want = (int64_t)nsm * 2;  // two CTAs an SM
  const unsigned grid = (unsigned)(a.rows < want ? a.rows : want);
  const size_t dyn = (size_t)kRNSt * kRStageBytes + sizeof(RowSmem);
  e = cudaFuncSetAttribute(k_row<E, RN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  k_row<E, RN><<<grid, kRThreads, dyn, s>>>(a);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_renorm_rows(const SampleArgs& a, cudaStream_t s) {
  if (a.rows <= 0 || a.bf16 || !a.out) return cudaErrorInvalidValue;
  return launch_row_kernel<float, true>(a, s);
}

cudaError_t row_read_error(uint32_t* word, int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_row_err, sizeof(v));
  if (e != cudaSuccess) return e;
  *word = v;
  if (clear && v) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_row_err, &z, sizeof(z));
  }
  return e;
}

}  // namespace tsv
