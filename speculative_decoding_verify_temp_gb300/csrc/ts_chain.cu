// Row-streaming kernel for target-only chain sampling from logits (TokenSpeed
// flashinfer.py verify(): sampling_argmax for greedy requests; softmax with temperature,
// fused top-k/top-p renorm and chain_speculative_sampling_target_only for the others).
//
// Three launches per call (four with a probability output, one more with draft
// probabilities):
//  - k_chain_plan (one CTA) orders the rows by cost tier (top-p and general rows first,
//    then large top-k rows, then the other sampled rows, greedy rows last), so that the
//    step ends on short rows, and clears the per-launch state: the row claim counter, the
//    per-request row counts and accept_length (0 until a request's chain is written).
//    A ragged batch (qo_indptr) schedules each request's own window of packed rows.
//  - k_chain: persistent CTAs (two an SM) of a producer warp and 7 compute warps. The
//    producer keeps a ring of kCNSt shared-memory stages of 14 KB filled with bulk copies
//    that complete on mbarriers, and claims the next row from the planned order when the
//    current one has kCNSt + 1 stages left to issue (the claim's latency hides behind
//    them, and a CTA never holds more than its current and next rows). Each compute warp
//    copies its four 16-byte vectors of a stage to registers, releases the slot, and
//    keeps running row state in a loop specialised for the row's kind:
//     - every row: maximum and its first token id (lowest id among equal values), and
//       the temperature-1 log-sum-exp when logprobs are asked for;
//     - top-k (k <= kSTopK): a candidate list in shared memory above a threshold: first a
//       lower bound of the row's k-th value from the first stage, later the k-th largest
//       candidate value whenever the list fills; at the end the row's top k, the top-p
//       prefix within it, and the draw in token-id order;
//     - neither knob: the mass of every warp's 128 vectors of a stage relative to their
//       maximum; at the end these ranges, scaled to the row maximum, locate the draw, and
//       only that range is read again;
//     - top-p alone: three passes over the row, the first from HBM, the other two from L2
//       (the first two passes load with an evict-last cache policy, every other load
//       evict-first). Pass 1: a histogram of the weights over 32 octaves below a window
//       top set by the first stage's maximum, one column of bins per thread (no shared
//       atomics); it locates the octave where the ordered mass crosses top_p. Pass 2 (the
//       row maximum now known): the row's mass and a histogram over sixteenths of the two
//       octaves around the crossing, which locates the crossing sixteenth. Pass 3: the
//       kept mass of each warp range above the two sixteenths around the crossing and
//       the elements within them, resolved exactly; then the draw.
//    Rows the summaries cannot serve (top_k above kSTopK, candidate overflow, a top-p
//    crossing outside its windows) take a general path: radix selections over the whole
//    row, read again from memory. Top-k rows apply min_p to their list, and with the
//    joint order measure top_p on the whole row's mass (one more pass over the row);
//    other rows with min_p take one more pass that keeps the tokens above its bound
//    (top-p rows only when that bound lies above their nucleus cut).
//  - k_chain_write: the chain of every request whose rows are all recorded (accepted
//    tokens, accept index, logprobs, accept_length), one warp a request. A row only
//    stores its record and counts itself, without waiting on the count.
//  - k_chain_resid (draft probabilities): the residual draw of each rejected row.
//  - k_chain_probs (single-step sampling with a probability output): each row's kept
//    distribution, rebuilt from the row's record.
// The same launches serve single-step sampling (TokenSpeed sample(); TensorRT-LLM
// fused_sample_from_logits_with_probs) as chains of one row and no draft.
//
// Weights are 2^((x - M) log2(e) / T) for the row maximum M; masses that decide a
// selection are sums of floor(w * 2^40); composite keys order tokens by value, then by
// lowest id. Every wait on an mbarrier is bounded: a stage wait by the launch's
// wait_cycles of SM clock. A wait that gives up sets the CTA's abort flag and the
// library's sticky error word (ts_device_error); the CTA then issues no more copies,
// leaves its current row unwritten at the next row boundary, waits for the copies it has
// in flight and exits. The requests it leaves keep accept_length = 0 from the planning
// launch, and the next launch starts from a clean state.
#include <stdint.h>

#include <type_traits>

#include "ts_common.cuh"
#include "ts_internal.h"
#include "ts_rowutil.cuh"
#include "ts_select.cuh"

namespace tsv {
namespace {

constexpr int kCC = 224;                       // compute threads (7 warps)
constexpr int kCW = kCC / 32;
constexpr int kCThreads = kCC + 32;            // + the producer warp
constexpr int kCNSt = 4;                       // ring stages
constexpr int kCVecs = 4;                      // vectors per compute thread and stage
constexpr int kCStageVecs = kCC * kCVecs;      // 896 vectors of 16 bytes
constexpr int kCStageBytes = kCStageVecs * 16;  // 14336
constexpr int kCCap = 4096;                    // candidate / crossing list capacity
constexpr int kCHalf = kCCap / 2;
constexpr int kCSmallE = 4;                    // lists of up to 128 candidates: one warp
constexpr int kCMerge = 128;                   // top-k: k up to this takes its first bound
                                               // from the first stage's vector maxima and
                                               // is compacted only at the end
constexpr int kPB = 32;                        // top-p bins per level
constexpr int kPHead = 8;                      // octaves of the window above the first stage
constexpr long long kCDrainCycles = 1ll << 32;
constexpr uint32_t kNoRow = 0xFFFFFFFFu;
constexpr uint32_t kRowMask = (1u << 30) - 1u;
constexpr double kCInvFx = 1.0 / 1099511627776.0;  // 2^-40
constexpr float kFx1 = 17592186044416.f;            // 2^44: top-p pass 1's mass scale
constexpr double kCInvFx1 = 1.0 / 17592186044416.0;  // 2^-44

enum CKind : int { kCGreedy = 0, kCTopK = 1, kCPlain = 2, kCTopP = 3, kCGeneral = 4 };

template <int K>
using KindTag = std::integral_constant<int, K>;

}  // namespace

static __device__ unsigned int g_chain_err;

namespace {

struct CKnobs {
  float T, tp, mp;
  int32_t k;
  int kind;
};

// The request's knobs and the way its rows are served. top_p <= 0 keeps only the argmax,
// which is the greedy distribution. min_p is clamped to [0, 1].
__device__ __forceinline__ CKnobs cknobs(const SampleArgs& a, int64_t req) {
  CKnobs kn;
  kn.T = a.temperature ? a.temperature[req] : 1.f;
  kn.k = a.top_k ? a.top_k[req] : 0;
  kn.tp = a.top_p ? a.top_p[req] : 1.f;
  kn.mp = a.min_p ? fminf(fmaxf(a.min_p[req], 0.f), 1.f) : 0.f;
  const bool tk = kn.k > 0 && (int64_t)kn.k < a.V;
  if (!(kn.T >= kGreedyT)) kn.kind = kCGreedy;
  else if (tk) kn.kind = (kn.k <= kSTopK) ? kCTopK : kCGeneral;
  else if (kn.tp < 1.f) kn.kind = (kn.tp > 0.f) ? kCTopP : kCGreedy;
  else kn.kind = kCPlain;
  return kn;
}

// The seed, offset and coin position of a row's draw coin: a chain's request and its
// position D (the request's own draft count), or, when sampling, the row's request and
// its position within it.
struct CCoin {
  int64_t sreq;
  uint32_t pos;
};
__device__ __forceinline__ CCoin ccoin(const SampleArgs& a, int64_t req, int32_t D) {
  if (a.sample_n > 0) return CCoin{req / a.sample_n, (uint32_t)(req % a.sample_n)};
  return CCoin{req, (uint32_t)D};
}

__device__ __forceinline__ int ctier(const CKnobs& kn) {
  if (kn.kind == kCTopP || kn.kind == kCGeneral) return 0;
  if (kn.kind == kCTopK && kn.k > kCMerge) return 1;
  return (kn.kind != kCGreedy) ? 2 : 3;
}

__device__ __forceinline__ bool ld_abort(const int32_t* f) {
  return *reinterpret_cast<const volatile int32_t*>(f) != 0;
}

// One non-blocking probe of the phase of `bar` with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 "
      "%0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity; gives up after `budget` cycles of
// this SM's clock or as soon as the CTA's abort flag is up, raising it (and the sticky
// error word). Returns whether the phase completed. Budgets below 2^20 cycles poll
// without suspending (a suspended probe may outlast a short budget).
__device__ __forceinline__ bool cwait(uint64_t* bar, uint32_t parity, unsigned long long budget,
                                      int32_t* abort_flag) {
  const bool short_budget = budget < (1ull << 20);
  if (short_budget ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t it = 1;; ++it) {
    if (short_budget ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u &&
        (ld_abort(abort_flag) || (unsigned long long)(clock64() - t0) > budget)) {
      *reinterpret_cast<volatile int32_t*>(abort_flag) = 1;
      atomicOr(&g_chain_err, 1u);
      return false;
    }
  }
}

// Waits, on the long budget only, for a copy this CTA issued: no copy may be in flight
// when the CTA exits.
__device__ __forceinline__ void cdrain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kCDrainCycles) {
      atomicOr(&g_chain_err, 2u);
      return;
    }
}

// 1-D bulk copy global -> shared with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_pol(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// The compute warps' barrier (named barrier 1; the producer warp never takes part).
struct CBar {
  __device__ __forceinline__ static void sync() { asm volatile("bar.sync 1, 224;" ::: "memory"); }
};
static_assert(kCC == 224, "CBar counts 224 threads");
__device__ __forceinline__ void cbar() { CBar::sync(); }

struct alignas(16) CSmem {
  uint64_t full[kCNSt];
  uint64_t empty[kCNSt];
  int64_t srow[kCNSt];
  sel::Scratch sc;
  union {
    uint64_t list[kCCap];       // top-k candidates; top-p crossing elements
    float hist[kPB * kCC];      // top-p: bin b of compute thread t at b * kCC + t
    struct {
      uint64_t lo[kCHalf];
      uint32_t keys[kCStageVecs];  // top-k: the first stage's vector maxima
    } tk;
  } w;
  double dscan[32];
  double hb[kPB];
  float hw[kCW][kPB];
  uint64_t red2[2][kCW];
  float redf[3][kCW];
  int32_t redi[kCW];
  uint32_t lcnt, tau;
  int32_t bad, abort_flag, owner, am;
  float M, S1, uj, uD, vx, qx;
  int32_t pbi;
  int32_t gtop, gl, gh;
  uint64_t res_u, zall, ptarget;
  double res_d;
};

// The ragged last vector of a row (n < N valid elements from e0 on), read from global
// memory and padded with -inf; kept out of line so that the stage loops stay small.
template <typename E>
__device__ __noinline__ uint4 ragged_vec(const E* xr, int e0, int n) {
  uint32_t wv[4] = {SVec<E>::kNegInfWord, SVec<E>::kNegInfWord, SVec<E>::kNegInfWord,
                    SVec<E>::kNegInfWord};
  for (int q = 0; q < n; ++q) {
    if (sizeof(E) == 2) {
      const uint32_t h = reinterpret_cast<const uint16_t*>(xr)[e0 + q];
      wv[q >> 1] = (q & 1) ? ((wv[q >> 1] & 0x0000FFFFu) | (h << 16))
                           : ((wv[q >> 1] & 0xFFFF0000u) | h);
    } else {
      wv[q] = reinterpret_cast<const uint32_t*>(xr)[e0 + q];
    }
  }
  return make_uint4(wv[0], wv[1], wv[2], wv[3]);
}

// two CTAs an SM: their rings and state fit the SM's 228 KB of shared memory (1 KB of it
// reserved per CTA)
static_assert(2 * (kCNSt * kCStageBytes + sizeof(CSmem) + 1024) <= 233472, "two CTAs an SM");

// The packed rows of request b: [first, first + count); count 0 for a ragged window that
// does not fit (outside the rows, or more than R rows), which is left unverified.
struct CWin {
  int64_t first;
  int32_t count;
};
__device__ __forceinline__ CWin cwin(const SampleArgs& a, int64_t b) {
  if (!a.qo) return CWin{b * a.R, a.R};
  const int64_t f = a.qo[b], e = a.qo[b + 1];
  if (f < 0 || e > a.rows || e - f < 1 || e - f > a.R) return CWin{0, 0};
  return CWin{f, (int32_t)(e - f)};
}

// Orders the rows by cost tier (stable within a tier) and clears the per-launch state. A
// request's rows share its knobs, so the order is built over requests: the rows of a
// request take consecutive claim positions, after the rows of the requests before it in
// its tier. Each entry holds the row and, in bits 30-31, its number of passes minus one;
// positions past the last scheduled row hold kNoRow. A ragged batch also records the
// request of every packed row.
__global__ void __launch_bounds__(1024) k_chain_plan(SampleArgs a) {
  __shared__ uint32_t cnt[4];
  __shared__ uint32_t wc[32][4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t B = a.nreq;
  if (tid < 4) cnt[tid] = 0u;
  if (tid == 0) {
    a.ws.work[0] = 0u;  // top-k candidates collected (all rows)
    a.ws.work[1] = 0u;  // top-k lists compacted at the end
    a.ws.work[2] = 0u;  // rows the general path served
    a.ws.work[3] = 0u;  // row claims
  }
  uint32_t c[4] = {0u, 0u, 0u, 0u};
  for (int64_t b = tid; b < B; b += 1024) {
    a.ws.creq[b] = 0u;
    a.accept_length[b] = 0;
    const int t = ctier(cknobs(a, b));
    const int32_t n = cwin(a, b).count;
    c[t] += (uint32_t)n;
    if (n == 0)  // a ragged window that does not fit: its outputs read as unused
      for (int32_t jj = 0; jj < a.R; ++jj) {
        a.accepted_tokens[b * a.R + jj] = -1;
        if (a.accept_index) a.accept_index[b * a.R + jj] = -1;
        if (a.logprobs) a.logprobs[b * a.R + jj] = 0.f;
      }
  }
  __syncthreads();
  for (int q = 0; q < 4; ++q)
    if (c[q]) atomicAdd(&cnt[q], c[q]);
  __syncthreads();
  uint32_t r[4] = {0u, cnt[0], cnt[0] + cnt[1], cnt[0] + cnt[1] + cnt[2]};
  const uint32_t total = r[3] + cnt[3];
  for (int64_t bb = 0; bb < B; bb += 1024) {
    const int64_t b = bb + tid;
    int t = 4;
    uint32_t np = 0u;
    CWin wn{0, 0};
    if (b < B) {
      const CKnobs kn = cknobs(a, b);
      t = ctier(kn);
      np = (kn.kind == kCTopP) ? 2u : 0u;  // passes - 1
      wn = cwin(a, b);
    }
    uint32_t before = 0u;
    for (int q = 0; q < 4; ++q) {
      const uint32_t v = (t == q) ? (uint32_t)wn.count : 0u;
      uint32_t inc = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
      }
      if (lane == 31) wc[warp][q] = inc;
      if (t == q) before = inc - v;
    }
    __syncthreads();
    if (t < 4) {
      uint32_t pos = r[t] + before;
      for (int w = 0; w < warp; ++w) pos += wc[w][t];
      for (int32_t jj = 0; jj < wn.count; ++jj) {
        const int64_t row = wn.first + jj;
        if ((int64_t)pos + jj < a.rows) a.ws.order[(int64_t)pos + jj] = (uint32_t)row | (np << 30);
        if (a.qo) a.ws.rreq[row] = (uint32_t)b;
      }
    }
    for (int w = 0; w < 32; ++w)
      for (int q = 0; q < 4; ++q) r[q] += wc[w][q];
    __syncthreads();
  }
  for (int64_t p = (int64_t)total + tid; p < a.rows; p += 1024) a.ws.order[p] = kNoRow;
}

// The min_p pass of a row (one warp a range at a time, ranges warp, warp + kCW, ...):
// range e (stage e / kCW, warp e % kCW of it: kCVecs x 32 vectors) gets the sum of the
// fixed-point weights of its tokens with x - M >= bound, the draft token x left out.
// Returns the lane's smallest passing value key (at most fkey(M)). Kept out of line: it
// runs once for a few rows, and inlined it would raise the register need of the
// streaming loops.
template <typename E>
__device__ __noinline__ uint32_t minp_ranges(const E* xr, int64_t V, int64_t nranges, int SE,
                                             float M, float bound, float sl2, int32_t x,
                                             uint64_t* rowslots) {
  constexpr int N = SVec<E>::N;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint4* rp = reinterpret_cast<const uint4*>(xr);
  const int64_t nvr = V / N, nvall = (V + N - 1) / N;
  uint32_t kmin = fkey(M);
  for (int64_t e = warp; e < nranges; e += kCW) {
    const int64_t v0 = (e / kCW) * (SE / N) + (e % kCW) * (kCVecs * 32);
    uint64_t sum = 0;
    for (int u = 0; u < kCVecs; ++u) {
      const int64_t vi = v0 + u * 32 + lane;
      if (vi >= nvall) continue;
      float xv[N];
      if (vi < nvr) {
        SVec<E>::unpack(__ldcg(rp + vi), xv);
      } else {
        for (int q = 0; q < N; ++q) xv[q] = (vi * N + q < V) ? SVec<E>::at(xr, vi * N + q) : -INFINITY;
      }
#pragma unroll
      for (int q = 0; q < N; ++q) {
        if (!(xv[q] - M >= bound)) continue;
        kmin = min(kmin, fkey(xv[q]));
        if (vi * N + q != (int64_t)x) sum += fixw(ex2((xv[q] - M) * sl2));
      }
    }
    sum = warp_sum_u64(sum);
    if (lane == 0) rowslots[e] = sum;
  }
  return kmin;
}

// EXT: the kernel also serves min_p and the joint filter order (a separate
// instantiation, so that calls without them run the smaller kernel).
template <typename E, bool EXT>
__global__ void __launch_bounds__(kCThreads, 2) k_chain(SampleArgs a) {
  extern __shared__ __align__(128) unsigned char dsm[];
  constexpr int N = SVec<E>::N;
  constexpr int SE = kCStageBytes / (int)sizeof(E);  // elements per stage
  unsigned char* ring = dsm;
  CSmem& sm = *reinterpret_cast<CSmem*>(dsm + kCNSt * kCStageBytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t V = a.V;
  const int nst = (int)((V + SE - 1) / SE);  // stages per pass
  const unsigned long long budget = a.wait_cycles;
  constexpr bool bf16 = sizeof(E) == 2;
  constexpr int lowv = bf16 ? 16 : 0;  // value key bits below this follow from the higher ones

  if (tid == 0) {
    for (int s = 0; s < kCNSt; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kCW);
    }
    fence_mbar_init();
    sm.abort_flag = 0;
  }
  __syncthreads();

  // ---- producer warp: the ring's refills ------------------------------------------------
  if (warp == kCW) {
    if (lane == 0) {
      uint64_t pol_first, pol_last;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_first));
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_last));
      auto order_at = [&](uint32_t pos) -> uint32_t {
        return (pos < (uint64_t)a.rows) ? __ldcg(&a.ws.order[pos]) : kNoRow;
      };
      uint32_t gi = 0;  // stages issued
      // A row is claimed when the previous one has a ring's depth of stages left to issue,
      // so that the claim's latency is hidden while a CTA holds at most the row it is
      // streaming and the next one's first stages (the last rows of a step stay spread).
      uint32_t pend = atomicAdd(&a.ws.work[3], 1u);  // the claim of the next row
      for (;;) {
        const uint32_t e = order_at(pend);
        if (e == kNoRow) {  // one last stage tells the consumers to stop
          const int slot = (int)(gi % kCNSt);
          const uint32_t use = gi / kCNSt;
          if ((use > 0 && !cwait(&sm.empty[slot], (use - 1) & 1u, budget, &sm.abort_flag)) ||
              ld_abort(&sm.abort_flag))
            break;
          sm.srow[slot] = -1;
          mbar_arrive_expect_tx(&sm.full[slot], 0u);
          ++gi;
          break;
        }
        const int64_t irow = (int64_t)(e & kRowMask);
        const int inp = (int)(e >> 30) + 1;
        const int total = inp * nst;
        const int claim_at = max(0, total - (kCNSt + 1));  // stage index that claims the next row
        const unsigned char* src =
            reinterpret_cast<const unsigned char*>(a.x) + irow * a.ld * (int64_t)sizeof(E);
        bool ok = true;
        for (int cs = 0; cs < total; ++cs, ++gi) {
          const int pass = cs / nst, c = cs - pass * nst;
          // top-p rows: the first two passes are kept in L2 for the ones that follow
          const uint64_t pol = (inp > 1 && pass < 2) ? pol_last : pol_first;
          const int slot = (int)(gi % kCNSt);
          const uint32_t use = gi / kCNSt;
          // after an error nothing more is issued (a slot may still be in use)
          if ((use > 0 && !cwait(&sm.empty[slot], (use - 1) & 1u, budget, &sm.abort_flag)) ||
              ld_abort(&sm.abort_flag)) {
            ok = false;
            break;
          }
          if (cs == claim_at) pend = atomicAdd(&a.ws.work[3], 1u);
          const int64_t nc = min((int64_t)SE, V - (int64_t)c * SE);
          const uint32_t bytes = (uint32_t)((nc * (int64_t)sizeof(E)) & ~(int64_t)15);
          sm.srow[slot] = irow;
          mbar_arrive_expect_tx(&sm.full[slot], bytes);
          if (bytes)
            bulk_g2s_pol(ring + slot * kCStageBytes, src + (int64_t)c * kCStageBytes, bytes,
                         &sm.full[slot], pol);
        }
        if (!ok) break;
      }
      // no copy of this CTA may still be in flight when it exits: wait for the last use of
      // every slot (normally complete already)
      for (uint32_t h = (gi > (uint32_t)kCNSt ? gi - (uint32_t)kCNSt : 0u); h < gi; ++h)
        cdrain(&sm.full[h % kCNSt], (h / kCNSt) & 1u);
    }
    return;
  }

  // ---- the rows -----------------------------------------------------------------------------
  const uint4 ninf = make_uint4(SVec<E>::kNegInfWord, SVec<E>::kNegInfWord,
                                SVec<E>::kNegInfWord, SVec<E>::kNegInfWord);
  const int64_t nvr = V / N;  // whole vectors of a row; the rest is a scalar tail
  const int64_t nvall = (V + N - 1) / N;
  const int vbase = warp * (kCVecs * 32) + lane;  // warp w: a stage's vectors 128 w ..
  uint32_t g = 0;                                 // the next stage to consume

  auto stage_ptr = [&](uint32_t gg) -> const uint4* {
    const int slot = (int)(gg % kCNSt);
    cwait(&sm.full[slot], (gg / kCNSt) & 1u, budget, &sm.abort_flag);
    return reinterpret_cast<const uint4*>(ring + slot * kCStageBytes);
  };
  auto stage_release = [&](uint32_t gg) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[gg % kCNSt]);
  };

  for (;;) {
    int64_t row;
    {
      const int slot = (int)(g % kCNSt);
      cwait(&sm.full[slot], (g / kCNSt) & 1u, budget, &sm.abort_flag);
      row = *reinterpret_cast<volatile int64_t*>(&sm.srow[slot]);
    }
    cbar();
    const bool ab = ld_abort(&sm.abort_flag);
    if (tid == 0) {
      sm.lcnt = 0;
      sm.bad = 0;
      sm.tau = 0;
    }
    cbar();
    if (ab || row < 0 || row >= a.rows) break;

    // the row's request, its position j in the request's window of rows (first row
    // rbase) and the request's drafts D (a ragged window verifies count - 1 of them);
    // the padded layouts (drafts, draft probabilities, coins, outputs) hold DP = a.D
    const int64_t req = a.qo ? (int64_t)__ldcg(&a.ws.rreq[row]) : row / a.R;
    const CWin win = cwin(a, req);
    const int64_t rbase = win.first;
    const int32_t j = (int32_t)(row - rbase);
    const int32_t D = win.count - 1;
    const int32_t DP = a.D;
    const CKnobs kn = cknobs(a, req);
    const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;
    const uint4* rp = reinterpret_cast<const uint4*>(xr);
    const int32_t x = (j < D) ? a.draft_tokens[req * DP + j] : -1;
    const bool xvalid = x >= 0 && (int64_t)x < V;
    const float sl2 = (kn.kind == kCGreedy) ? 0.f : __fdiv_rn(kLog2e, kn.T);
    const float s16 = sl2 * 16.f;  // sixteenths of an octave per logit unit
    const int32_t k = kn.k;
    uint64_t* const rowslots = a.ws.cand + row * a.ws.cand_splits * (int64_t)kSTopK;
    const bool want_lse = a.logprobs != nullptr;

    // vector vi of the stage held at sv (first element c0, nc elements, nvf whole
    // vectors); the ragged last vector of the row comes from global memory, padded with
    // -inf
    auto stage_vec = [&](const uint4* sv, int c0, int nc, int vi) -> uint4 {
      const int nvf = nc / N;
      if (vi < nvf) return sv[vi];
      if (vi > nvf || nc % N == 0) return ninf;
      return ragged_vec<E>(xr, c0 + vi * N, nc - nvf * N);
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
    // The sixteenth-of-an-octave bucket of a logit's weight: floor(v s16), with the
    // product taken exactly and rounded down, clamped to +-2^22 (monotone in v), from the
    // bits of v s16 + 1.5 2^23 (one fused multiply-add rounding toward -inf; no
    // conversion instruction). Its octave is the bucket >> 4.
    auto six_i = [&](float v) -> int {
      float t = __fmaf_rd(v, s16, 12582912.f);
      t = fminf(fmaxf(t, 8388608.f), 16777216.f);
      return __float_as_int(t) - 0x4B400000;
    };

    // running statistics of this thread's vectors
    float bv = -INFINITY;   // maximum
    int32_t bi = INT32_MAX;  // its first token id
    float lm = -INFINITY, ls = 0.f, lc = 0.f;  // temperature-1 log-sum-exp (Kahan)
    auto lse_vec = [&](const uint4& r, float vm) {
      if (!(vm > -INFINITY)) return;
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
    };

    // Keeps the list's candidates at or above the k-th largest value (cnt <= kCCap) and
    // returns that value's key; the list keeps its order of survivors in each half.
    auto compact = [&](uint32_t cnt) -> uint32_t {
      const uint32_t vk = sel::select_bound<kCC, CBar>(
          (int)cnt, [&](int i) { return (uint32_t)(sm.w.list[i] >> kIdxBits); }, (uint32_t)k,
          bf16 ? 2 : 4, sm.sc);
      // in two halves, so that a thread holds at most ceil(2048 / 224) candidates:
      // survivors of the first half go below 2048, the second half is read before it is
      // overwritten
      constexpr int KP = (kCHalf + kCC - 1) / kCC;
      for (int half = 0; half < 2; ++half) {
        uint64_t keep[KP];
#pragma unroll
        for (int m = 0; m < KP; ++m) {
          const uint32_t i = (uint32_t)(half * kCHalf + m * kCC + tid);
          keep[m] = (i < cnt && i < (uint32_t)((half + 1) * kCHalf)) ? sm.w.list[i] : 0ull;
        }
        cbar();
        if (half == 0 && tid == 0) sm.lcnt = 0;
        cbar();
#pragma unroll
        for (int m = 0; m < KP; ++m)
          if ((uint32_t)(keep[m] >> kIdxBits) >= vk && keep[m] != 0ull)
            sm.w.list[atomicAdd(&sm.lcnt, 1u)] = keep[m];
        cbar();
      }
      return vk;
    };
    uint64_t z1 = 0;  // top-p pass 1: the row's mass in 2^-44 units of 2^(pbi + 1)

    // One pass over the row's stages: the statistics every row keeps, and the kind's own
    // summary. PASS is the top-p pass (1 for every other kind).
    auto stream = [&](auto kind_tag, auto pass_tag) {
      constexpr int KIND = decltype(kind_tag)::value;
      constexpr int PASS = decltype(pass_tag)::value;
      for (int c = 0; c < nst; ++c, ++g) {
        const uint4* sv = stage_ptr(g);
        const int c0 = c * SE;  // the stage's first element
        const int nc = min(SE, (int)V - c0);
        uint4 rv[kCVecs];
        if (nc == SE) {
#pragma unroll
          for (int u = 0; u < kCVecs; ++u) rv[u] = sv[vbase + u * 32];
        } else {
#pragma unroll
          for (int u = 0; u < kCVecs; ++u) rv[u] = stage_vec(sv, c0, nc, vbase + u * 32);
        }
        stage_release(g);
        float vmv[kCVecs];
#pragma unroll
        for (int u = 0; u < kCVecs; ++u) vmv[u] = SVec<E>::vmax(rv[u]);
        if (PASS == 1) {
          // the thread's maximum and its first token id: the stage's four vector maxima
          // against the running maximum, searched only when it rises
          const float m4 = fmaxf(fmaxf(vmv[0], vmv[1]), fmaxf(vmv[2], vmv[3]));
          if (m4 > bv) {
            int qb = -1;
#pragma unroll
            for (int u = kCVecs - 1; u >= 0; --u) {
              if (vmv[u] != m4) continue;
              float xv[N];
              SVec<E>::unpack(rv[u], xv);
#pragma unroll
              for (int q = N - 1; q >= 0; --q)
                if (xv[q] == m4) qb = (vbase + u * 32) * N + q;
            }
            bv = m4;
            bi = c0 + qb;
          }
          if (want_lse) {
#pragma unroll
            for (int u = 0; u < kCVecs; ++u) lse_vec(rv[u], vmv[u]);
          }
        }

        if constexpr (KIND == kCTopK) {
          if (c == 0) {
            // a lower bound of the row's k-th value from the first stage. k <= 128: the k-th
            // largest of the stage's 896 vector maxima (distinct elements, so at least k of
            // the row's elements lie at or above it), built two key bits a round: each
            // thread counts its four maxima at or above the candidates C + {1, 2, 3}
            // 2^(bit - 1), one barrier a round sums the warps (two slots, alternating; the
            // counts are at most 896 and pack in 16 bits). Larger k: the stage's k-th
            // largest value, the same way over its elements.
            if (k <= kCMerge) {
              uint32_t kv[kCVecs];
#pragma unroll
              for (int u = 0; u < kCVecs; ++u) kv[u] = (vmv[u] > -INFINITY) ? fkey(vmv[u]) : 0u;
              static_assert(((32 - lowv) & 1) == 0, "the key bits pair up");
              uint32_t C = 0;
#pragma unroll 1
              for (int bit = 31; bit > lowv; bit -= 2) {
                const uint32_t c1 = C | (1u << (bit - 1)), c2 = C | (2u << (bit - 1)),
                               c3 = C | (3u << (bit - 1));
                uint32_t n12 = 0, n3 = 0;
#pragma unroll
                for (int u = 0; u < kCVecs; ++u) {
                  n12 += ((kv[u] >= c1) ? 1u : 0u) + ((kv[u] >= c2) ? 0x10000u : 0u);
                  n3 += (kv[u] >= c3) ? 1u : 0u;
                }
                n12 = __reduce_add_sync(0xffffffffu, n12);
                n3 = __reduce_add_sync(0xffffffffu, n3);
                const int slot = (bit >> 1) & 1;
                if (lane == 0) sm.red2[slot][warp] = (uint64_t)n12 | ((uint64_t)n3 << 32);
                cbar();
                uint64_t tot = 0;
#pragma unroll
                for (int w2 = 0; w2 < kCW; ++w2) tot += sm.red2[slot][w2];
                const uint32_t t1 = (uint32_t)(tot & 0xFFFFu), t2 = (uint32_t)((tot >> 16) & 0xFFFFu),
                               t3 = (uint32_t)(tot >> 32);
                if (t3 >= (uint32_t)k) C = c3;
                else if (t2 >= (uint32_t)k) C = c2;
                else if (t1 >= (uint32_t)k) C = c1;
              }
              if (tid == 0) sm.tau = C;
              cbar();
            } else {
              // the k-th largest of the stage's pair maxima (the larger of each two
              // neighbouring elements: distinct elements, so at least k of the row's
              // elements lie at or above it; half the keys of an element-wise bound, and a
              // little looser), built two bits at a time from the top: the largest C with
              // at least k pair maxima at or above it (bf16 keys carry 16 bits). Each round
              // every compute thread counts its own keys at or above the three candidates
              // C + {1, 2, 3} 2^(bit - 1); one barrier a round sums the warps (two slots,
              // alternating; a warp's counts are at most 512 and the stage's at most 3584,
              // so they pack in 16 bits). The thread's keys (0 for -inf) sit in its own
              // column of the list area (key i of thread t at i * kCC + t: no bank
              // conflicts).
              constexpr int NP = N / 2;  // pairs a vector
              uint32_t* skeys = reinterpret_cast<uint32_t*>(sm.w.list) + tid;
#pragma unroll
              for (int u = 0; u < kCVecs; ++u) {
                float xv[N];
                SVec<E>::unpack(rv[u], xv);
#pragma unroll
                for (int q = 0; q < NP; ++q) {
                  const float pm = fmaxf(xv[2 * q], xv[2 * q + 1]);
                  skeys[(u * NP + q) * kCC] = (pm > -INFINITY) ? fkey(pm) : 0u;
                }
              }
              static_assert(((32 - lowv) & 1) == 0, "the key bits pair up");
              uint32_t C = 0;
#pragma unroll 1
              for (int bit = 31; bit > lowv; bit -= 2) {
                const uint32_t c1 = C | (1u << (bit - 1)), c2 = C | (2u << (bit - 1)),
                               c3 = C | (3u << (bit - 1));
                uint32_t n12 = 0, n3 = 0;
#pragma unroll 8
                for (int i = 0; i < kCVecs * NP; ++i) {
                  const uint32_t key = skeys[i * kCC];
                  n12 += ((key >= c1) ? 1u : 0u) + ((key >= c2) ? 0x10000u : 0u);
                  n3 += (key >= c3) ? 1u : 0u;
                }
                n12 = __reduce_add_sync(0xffffffffu, n12);
                n3 = __reduce_add_sync(0xffffffffu, n3);
                const int slot = (bit >> 1) & 1;
                if (lane == 0) sm.red2[slot][warp] = (uint64_t)n12 | ((uint64_t)n3 << 32);
                cbar();
                uint64_t tot = 0;
#pragma unroll
                for (int w2 = 0; w2 < kCW; ++w2) tot += sm.red2[slot][w2];
                const uint32_t t1 = (uint32_t)(tot & 0xFFFFu), t2 = (uint32_t)((tot >> 16) & 0xFFFFu),
                               t3 = (uint32_t)(tot >> 32);
                if (t3 >= (uint32_t)k) C = c3;
                else if (t2 >= (uint32_t)k) C = c2;
                else if (t1 >= (uint32_t)k) C = c1;
              }
              if (tid == 0) sm.tau = C;
              cbar();
            }
          }
          // the elements at or above the threshold (a key at or below that of -inf keeps
          // every finite element)
          const uint32_t tau = sm.tau;
          const float tf = (tau <= 0x007FFFFFu) ? -INFINITY : key_to_value(tau);
          // a stage rarely holds a candidate once the bound is set: the warp tests its
          // stage maximum first
          const float m4 = fmaxf(fmaxf(vmv[0], vmv[1]), fmaxf(vmv[2], vmv[3]));
          if (__any_sync(0xffffffffu, m4 > -INFINITY && m4 >= tf)) {
            uint32_t mk[kCVecs];
            uint32_t nsel = 0;
  #pragma unroll
            for (int u = 0; u < kCVecs; ++u) {
              mk[u] = 0u;
              if (vmv[u] > -INFINITY && vmv[u] >= tf) {
                float xv[N];
                SVec<E>::unpack(rv[u], xv);
  #pragma unroll
                for (int q = 0; q < N; ++q)
                  if (xv[q] >= tf && xv[q] != -INFINITY) mk[u] |= 1u << q;
                nsel += (uint32_t)__popc(mk[u]);
              }
            }
            if (__any_sync(0xffffffffu, nsel != 0u)) {
              const uint32_t pos = warp_reserve(&sm.lcnt, nsel, lane);
              uint32_t m32 = 0;
#pragma unroll
              for (int u = 0; u < kCVecs; ++u) m32 |= mk[u] << (u * N);
              append_candidates<E>(m32, rv, c0, vbase, pos, sm.w.list, (uint32_t)kCCap);
            }
          }
          // k > 128: the list is checked every few stages (and after the last) and compacted
          // when it passes half its capacity. k <= 128 lists are only checked at the end.
          if (k > kCMerge && ((c + 1) % 8 == 0 || c == nst - 1)) {
            cbar();
            const uint32_t cnt = sm.lcnt;
            cbar();
            if (cnt > (uint32_t)kCCap) {
              if (tid == 0) {
                sm.bad = 1;
                sm.tau = 0xFFFFFFFFu;  // stop collecting; the general path takes the row
                sm.lcnt = 0;
              }
              cbar();
            } else if (cnt > (uint32_t)kCHalf) {
              const uint32_t vk = compact(cnt);
              if (tid == 0) sm.tau = max(sm.tau, vk);
              cbar();
              if (sm.lcnt > (uint32_t)kCHalf) {  // ties at the k-th value fill the list
                cbar();
                if (tid == 0) {
                  sm.bad = 1;
                  sm.tau = 0xFFFFFFFFu;
                  sm.lcnt = 0;
                }
              }
              cbar();
            }
          }
        } else if constexpr (KIND == kCPlain) {
          // warp w's 128 vectors of the stage: their mass relative to their own maximum,
          // the draft token left out
          float em = fmaxf(fmaxf(vmv[0], vmv[1]), fmaxf(vmv[2], vmv[3]));
          em = warp_max(em);
          float s = 0.f;
          if (em > -INFINITY) {
#pragma unroll
            for (int u = 0; u < kCVecs; ++u) {
              const int e0 = c0 + (vbase + u * 32) * N;
              float xv[N];
              SVec<E>::unpack(rv[u], xv);
              float vs = 0.f;
              if ((unsigned)(x - e0) < (unsigned)N) {
#pragma unroll
                for (int q = 0; q < N; ++q)
                  vs += (e0 + q == x) ? 0.f : ex2((xv[q] - em) * sl2);
              } else {
#pragma unroll
                for (int q = 0; q < N; ++q) vs += ex2((xv[q] - em) * sl2);
              }
              s += vs;
            }
          }
          s = warp_sum_f32(s);
          if (lane == 0)
            rowslots[c * kCW + warp] =
                ((uint64_t)__float_as_uint(em) << 32) | __float_as_uint(s);
        } else if constexpr (KIND == kCTopP && PASS == 1) {
          // pass 1: weights relative to 2^(pbi + 1), the window top (kPHead octaves above
          // the first stage's maximum): the row's mass, and octave bins below the window
          // top (bin d: octave pbi - d; the lowest bin also takes every deeper element),
          // one column per compute thread (no shared atomics; -inf elements add 0)
          if (c == 0) {
            float m = fmaxf(fmaxf(vmv[0], vmv[1]), fmaxf(vmv[2], vmv[3]));
            m = warp_max(m);
            if (lane == 0) sm.redf[0][warp] = m;
#pragma unroll
            for (int b = 0; b < kPB; ++b) sm.w.hist[b * kCC + tid] = 0.f;
            cbar();
            if (tid == 0) {
              float mm = sm.redf[0][0];
              for (int w2 = 1; w2 < kCW; ++w2) mm = fmaxf(mm, sm.redf[0][w2]);
              sm.pbi = (mm > -INFINITY) ? (six_i(mm) >> 4) + kPHead : 0;
              if (!(mm > -INFINITY)) sm.bad = 1;
            }
            cbar();
          }
          const int pbi = sm.pbi;
          const float ptop = (float)(pbi + 1);
          float zs = 0.f;
#pragma unroll
          for (int u = 0; u < kCVecs; ++u) {
            float xv[N];
            SVec<E>::unpack(rv[u], xv);
            // the octave below the window top: from the weight's exponent (wv = 2^t, t =
            // v sl2 - pbi - 1, so d = pbi - floor(v sl2) = 126 - biased exponent; a zero
            // weight falls in the last bin). An element the fast 2^t puts one octave off
            // near an octave edge only moves the window the later exact passes check.
            // The vector maximum has the vector's smallest d: below 0, an element lies
            // above the window (the row goes to the general path).
            const int dv = 126 - (int)(__float_as_uint(ex2(fmaf(vmv[u], sl2, -ptop))) >> 23);
            if (dv < 0) sm.bad = 1;
            if (__all_sync(0xffffffffu, dv >= kPB - 1)) {
              // the warp's vectors lie in the lowest bin, whose mass no crossing uses
              // (a crossing there sends the row to the general path): the row's mass only
#pragma unroll
              for (int q = 0; q < N; ++q) zs += ex2(fmaf(xv[q], sl2, -ptop));
            } else {
#pragma unroll
              for (int q = 0; q < N; ++q) {
                const float wv = ex2(fmaf(xv[q], sl2, -ptop));
                zs += wv;
                const unsigned d = (unsigned)(126 - (int)(__float_as_uint(wv) >> 23));
                sm.w.hist[min(d, (unsigned)(kPB - 1)) * kCC + tid] += wv;
              }
            }
          }
          // at most 32 weights of at most 1 each (else the row is flagged above): the
          // stage's share in 2^-44 units of the window top, rounded to nearest
          z1 += __float2ull_rn(zs * kFx1);
        } else if constexpr (KIND == kCTopP && PASS == 2) {
          // pass 2 (the row maximum known): sixteenth bins over the window's two octaves,
          // weights relative to the maximum
          const float M = sm.M;
          const int gt = sm.gtop;
#pragma unroll
          for (int u = 0; u < kCVecs; ++u) {
            const bool meets = vmv[u] > -INFINITY && six_i(vmv[u]) >= gt - (kPB - 1) &&
                               six_i(SVec<E>::vmin(rv[u])) <= gt;
            if (!__any_sync(0xffffffffu, meets)) continue;  // the warp's vectors miss it
            float xv[N];
            SVec<E>::unpack(rv[u], xv);
#pragma unroll
            for (int q = 0; q < N; ++q) {
              const float v = xv[q];
              const unsigned f = (unsigned)(gt - six_i(v));
              if (meets && f < (unsigned)kPB) sm.w.hist[f * kCC + tid] += ex2((v - M) * sl2);
            }
          }
        } else if constexpr (KIND == kCTopP && PASS == 3) {
          // pass 3: per warp range the kept mass above the collected sixteenths (the
          // draft token left out), and the elements within them
          const float M = sm.M;
          const int gh = sm.gh, gl = sm.gl;
          float s = 0.f;
          uint32_t mk[kCVecs];
          uint32_t nsel = 0;
#pragma unroll
          for (int u = 0; u < kCVecs; ++u) {
            mk[u] = 0u;
            const bool any = vmv[u] > -INFINITY && six_i(vmv[u]) >= gl;
            if (!__any_sync(0xffffffffu, any)) continue;  // the warp's vectors are lighter
            const int e0 = c0 + (vbase + u * 32) * N;
            float xv[N];
            SVec<E>::unpack(rv[u], xv);
#pragma unroll
            for (int q = 0; q < N; ++q) {
              const float v = xv[q];
              const int gx = six_i(v);  // -inf: the lowest bucket, below the window
              const float wv = ex2((v - M) * sl2);
              s += (any && gx > gh && e0 + q != x) ? wv : 0.f;
              mk[u] |= (any && gx >= gl && gx <= gh) ? (1u << q) : 0u;
            }
            nsel += (uint32_t)__popc(mk[u]);
          }
          if (__any_sync(0xffffffffu, nsel != 0u)) {
            const uint32_t pos = warp_reserve(&sm.lcnt, nsel, lane);
            uint32_t m32 = 0;
#pragma unroll
            for (int u = 0; u < kCVecs; ++u) m32 |= mk[u] << (u * N);
            append_candidates<E>(m32, rv, c0, vbase, pos, sm.w.list, (uint32_t)kCCap);
          }
          // the warp's sum (each lane's below 2^46: 32 weights of at most 1) by two 32-bit
          // reductions, of the low 24 bits and of the rest; none where the range keeps nothing
          const uint64_t fl = __float2ull_rz(s * kFx);
          uint64_t f = 0ull;
          if (__any_sync(0xffffffffu, fl != 0ull)) {
            const uint32_t lo = __reduce_add_sync(0xffffffffu, (uint32_t)(fl & 0xFFFFFFu));
            const uint32_t hi = __reduce_add_sync(0xffffffffu, (uint32_t)(fl >> 24));
            f = ((uint64_t)hi << 24) + lo;
          }
          if (lane == 0) rowslots[c * kCW + warp] = f;
        }
      }
    };

    // ---- the streaming passes ---------------------------------------------------------------
    switch (kn.kind) {
      case kCTopK: stream(KindTag<kCTopK>{}, KindTag<1>{}); break;
      case kCPlain: stream(KindTag<kCPlain>{}, KindTag<1>{}); break;
      case kCTopP: stream(KindTag<kCTopP>{}, KindTag<1>{}); break;
      default: stream(KindTag<kCGreedy>{}, KindTag<1>{}); break;
    }

    // ---- the row's statistics ---------------------------------------------------------------
    ls += lc;
    {
      float v = bv, m = lm, s = ls;
      int32_t i = bi;
      warp_argmax(v, i);
      if (want_lse) warp_lse(m, s);
      if (lane == 0) {
        sm.redf[0][warp] = v;
        sm.redf[1][warp] = m;
        sm.redf[2][warp] = s;
        sm.redi[warp] = i;
      }
      cbar();
      if (warp == 0) {
        v = lane < kCW ? sm.redf[0][lane] : -INFINITY;
        m = lane < kCW ? sm.redf[1][lane] : -INFINITY;
        s = lane < kCW ? sm.redf[2][lane] : 0.f;
        i = lane < kCW ? sm.redi[lane] : INT32_MAX;
        warp_argmax(v, i);
        if (want_lse) warp_lse(m, s);
        if (lane == 0) {
          sm.M = v;
          sm.am = (i == INT32_MAX) ? 0 : i;
          sm.S1 = s;
          // greedy rows need neither coins nor the draft token's logit
          float uj0 = 0.f, uD0 = 0.f, vx0 = 0.f, qx0 = 0.f;
          if (kn.kind != kCGreedy) {
            const CCoin cc = ccoin(a, req, D);
            const uint64_t seed = a.seed ? (uint64_t)a.seed[cc.sreq] : 0;
            const uint64_t off = a.offset ? (uint64_t)a.offset[cc.sreq] : 0;
            if (j < D)
              uj0 = a.uniforms ? a.uniforms[req * a.R + j] : verify_coin(seed, off, (uint32_t)j);
            uD0 = a.uniforms ? a.uniforms[req * a.R + D] : verify_coin(seed, off, cc.pos);
            vx0 = xvalid ? SVec<E>::at(xr, x) : 0.f;
            qx0 = (a.q && j < D && xvalid) ? a.q[(req * DP + j) * a.ld_q + x] : 0.f;
          }
          sm.uj = uj0;
          sm.uD = uD0;
          sm.vx = vx0;
          sm.qx = qx0;
        }
      }
      cbar();
    }
    const float M = sm.M;
    const int32_t am = sm.am;
    const float uj = sm.uj, uD = sm.uD, vx = sm.vx;
    auto wfn = [&](float v) -> uint64_t { return fixw(ex2((v - M) * sl2)); };
    auto wcomp = [&](uint64_t cc) -> uint64_t {
      return wfn(key_to_value((uint32_t)(cc >> kIdxBits)));
    };

    // ---- top-p: locate the crossing (passes 2 and 3) ------------------------------------------
    // Sums bin b over the compute threads' columns into sm.hb[b] (warp w, lane b takes the
    // entries of threads 32w .. 32w + 31 in a skewed order, free of bank conflicts).
    auto bin_totals = [&]() {
      float acc = 0.f;
#pragma unroll 8
      for (int i = 0; i < 32; ++i) acc += sm.w.hist[lane * kCC + warp * 32 + ((i + lane) & 31)];
      sm.hw[warp][lane] = acc;
      cbar();
      if (warp == 0) {
        double t = 0.0;
        for (int w2 = 0; w2 < kCW; ++w2) t += (double)sm.hw[w2][lane];
        sm.hb[lane] = t;
      }
      cbar();
    };
    if (kn.kind == kCTopP) {
      // pass 1's octave bins (weights relative to 2^(pbi + 1)) and the row's mass
      {
        const uint64_t z = warp_sum_u64(z1);
        if (lane == 0) sm.red2[0][warp] = z;
      }
      bin_totals();
      if (warp == 0) {
        uint64_t zt = 0;
        for (int w2 = 0; w2 < kCW; ++w2) zt += sm.red2[0][w2];
        const double zrel = (double)zt * kCInvFx1;  // the row's mass, units of 2^(pbi + 1)
        const double mb = sm.hb[lane];
        double incl = mb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const double P1 = (double)kn.tp * zrel;
        const double before = incl - mb;
        const unsigned hm = __ballot_sync(0xffffffffu, mb > 0.0 && before < P1 && P1 <= incl);
        const int bs = hm ? __ffs(hm) - 1 : -1;
        const double bbefore = __shfl_sync(0xffffffffu, before, bs >= 0 ? bs : 0);
        const double bmass = __shfl_sync(0xffffffffu, mb, bs >= 0 ? bs : 0);
        // the fine window: the crossing octave and its neighbour on the nearer side
        const bool okb = bs >= 0 && bs < kPB - 2;  // else the crossing is in or below the lowest bins
        const int bt = (okb && (P1 - bbefore) / bmass < 0.5 && bs > 0) ? bs - 1 : (okb ? bs : 0);
        const double above = __shfl_sync(0xffffffffu, before, bt);  // the bins above bt
        if (lane == 0) {
          // 2^40 times the weight of 2^(pbi + 1) relative to the row maximum's
          const double K =
              exp2((double)(sm.pbi + 1) - (double)M * (double)sl2) * 1099511627776.0;
          const double zm = zrel * K;
          const double want = ceil((double)kn.tp * zm);
          sm.ptarget = (want >= zm) ? (uint64_t)zm : (uint64_t)want;
          if (!okb) sm.bad = 1;
          sm.gtop = 16 * (sm.pbi - bt) + 15;
          sm.res_d = above * K;  // the mass above the window, 2^-40 units of the maximum
          // A crossing octave that holds few tokens (each weighs at least half its top
          // edge, so its mass bounds their number) is collected whole by pass 3, and
          // pass 2 is skipped: its sixteenths bound the crossing elements instead.
          sm.gh = 0;
          sm.gl = 1;  // gl > gh: pass 2 decides the window
          if (okb && bmass * exp2((double)(bs + 1)) <= 3500.0) {
            sm.gh = 16 * (sm.pbi - bs) + 15;
            sm.gl = 16 * (sm.pbi - bs);
          }
        }
      }
      cbar();
      const bool bad1 = sm.bad != 0;
      const bool skip2 = sm.gl <= sm.gh;  // the crossing octave is the window of pass 3
      // pass 2 (its stages are consumed in any case)
      if (!bad1 && !skip2) {
#pragma unroll
        for (int b = 0; b < kPB; ++b) sm.w.hist[b * kCC + tid] = 0.f;
      }
      cbar();
      if (!bad1 && !skip2) {
        stream(KindTag<kCTopP>{}, KindTag<2>{});
      } else {
        for (int c = 0; c < nst; ++c, ++g) {
          (void)stage_ptr(g);
          stage_release(g);
        }
      }
      cbar();
      if (!skip2) bin_totals();
      if (warp == 0 && !bad1 && !skip2) {
        // sixteenth f (0: the window's highest) in 2^-40 units of the maximum's weight,
        // after the mass above the window
        const double mf = sm.hb[lane] * 1099511627776.0;
        double incl = mf;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const double P = (double)sm.ptarget;
        const double before = sm.res_d + incl - mf;
        const unsigned hm = __ballot_sync(0xffffffffu, mf > 0.0 && before < P && P <= before + mf);
        const int fs = hm ? __ffs(hm) - 1 : -1;
        const double fbefore = __shfl_sync(0xffffffffu, before, fs >= 0 ? fs : 0);
        const double fmass = __shfl_sync(0xffffffffu, mf, fs >= 0 ? fs : 0);
        if (lane == 0) {
          if (fs < 0) {
            sm.bad = 1;
          } else {
            // the crossing sixteenth and its neighbour on the nearer side
            const double frac = (P - fbefore) / fmass;
            int f0 = fs, f1 = fs;
            if (frac < 0.5) f0 = (fs > 0) ? fs - 1 : fs;
            else f1 = (fs < kPB - 1) ? fs + 1 : fs;
            sm.gh = sm.gtop - f0;
            sm.gl = sm.gtop - f1;
          }
        }
      }
      cbar();
      const bool bad2 = sm.bad != 0;
      if (tid == 0) sm.lcnt = 0;
      cbar();
      if (!bad2) {
        stream(KindTag<kCTopP>{}, KindTag<3>{});
      } else {
        for (int c = 0; c < nst; ++c, ++g) {
          (void)stage_ptr(g);
          stage_release(g);
        }
      }
      cbar();
    }

    // a wait that gave up: leave the row (and the rest) unwritten
    {
      const bool ab2 = ld_abort(&sm.abort_flag);
      cbar();
      if (ab2) break;
    }
    // a top-k list that overflowed goes to the general path; one longer than a warp
    // takes is compacted to the row's top k first
    if (kn.kind == kCTopK && sm.bad == 0) {
      const uint32_t cnt = sm.lcnt;
      if (tid == 0) {
        atomicAdd(&a.ws.work[0], cnt);
        if (cnt > (uint32_t)(32 * kCSmallE)) atomicAdd(&a.ws.work[1], 1u);
      }
      if (cnt > (uint32_t)kCCap) {
        cbar();
        if (tid == 0) sm.bad = 1;
      } else if (cnt > (uint32_t)(32 * kCSmallE) && k <= kCMerge) {
        (void)compact(cnt);
      }
      cbar();
    }
    const bool bad = sm.bad != 0;

    // The accept test on the kept mass Z (the draft token's weight wx included):
    // target-only u < p(x), with draft probabilities u q(x) < p(x).
    const bool qmode = a.q != nullptr;
    const float qx = sm.qx;
    // Relaxed acceptance (target-only, a threshold in (0, 1); any other value means 1):
    // p(x) >= threshold_single or u threshold_acc < p(x).
    const float ts = (a.thr_single > 0.f && a.thr_single < 1.f) ? a.thr_single : 1.f;
    const float ta = (a.thr_acc > 0.f && a.thr_acc < 1.f) ? a.thr_acc : 1.f;
    const bool relaxed = !qmode && (ts < 1.f || ta < 1.f);
    auto accept = [&](double Z, double wx) -> int32_t {
      if (j >= D) return 0;
      if (relaxed)
        return (wx >= (double)ts * Z || (double)uj * (double)ta * Z < wx) ? 1 : 0;
      return (qmode ? (double)uj * (double)qx * Z < wx : (double)uj * Z < wx) ? 1 : 0;
    };
    // With draft probabilities the residual draw of a rejected row needs the draft row:
    // rows before the last record their kept set and leave the draw to k_chain_resid.
    const bool skip_draw = qmode && j < D;
    // records the row (k_chain_write then writes the chains of complete requests)
    auto finish_row = [&](int32_t tok_f, int32_t acc_f, int32_t kset = 0, uint64_t Cf = 0,
                          uint64_t Zf = 0) {
      RowRes rr{M, am, sm.S1, tok_f, acc_f, {0, 0, 0}, Cf, Zf, 0, 0, kset, 0};
      if (kset == 3) {
        rr.gh = sm.gh;
        rr.gl = sm.gl;
      }
      a.ws.rowres[row] = rr;
      // the request's count of recorded rows (k_chain_write, the next launch, writes the
      // chains of the requests whose rows are all recorded)
      asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(&a.ws.creq[req]) : "memory");
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
    // The same over the kCVecs * 32 vectors from v0, a step of 32 at a time.
    auto walk_range = [&](int64_t v0, float tf, auto&& wgt) -> int32_t {
      int lastu = -1;
      for (int u = 0; u < kCVecs; ++u) {
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
    // The draw over per-range masses (stage c, warp w at c * kCW + w; the draft token left
    // out) with coin uD, then a walk of the chosen range with weights wgt: warp 0 records
    // the row. Zr is the ranges' total.
    const int64_t e1max = (int64_t)nst * kCW;  // the row's ranges
    auto draw_ranges = [&](uint64_t mine, uint64_t ex, uint64_t Zr, int64_t e0, int64_t e1,
                           int32_t acc, int32_t kset, uint64_t Cf, uint64_t Zf, auto&& wgt) {
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
        sm.res_d = (double)(t - accu) * kCInvFx;
      }
      cbar();
      if (warp == 0) {
        const int64_t es = min((int64_t)(sm.res_u % (uint64_t)e1max), e1max - 1);
        const int64_t v0 = (es / kCW) * (SE / N) + (es % kCW) * (kCVecs * 32);
        const int32_t tok = walk_range(v0, (float)sm.res_d, wgt);
        if (lane == 0) finish_row(tok >= 0 ? tok : am, acc, kset, Cf, Zf);
      }
    };

    // min_p: a token stays iff x - M >= T ln(min_p) (a value bound; the argmax passes)
    const bool use_mp = EXT && kn.mp > 0.f;
    const float mp_thr = use_mp ? kn.T * logf(kn.mp) : -INFINITY;
    auto mp_keep = [&](uint64_t cc) -> bool {
      return !use_mp || key_to_value((uint32_t)(cc >> kIdxBits)) - M >= mp_thr;
    };
    // The weight of a token in a draw over ranges (the draft token left out): top-p rows
    // keep the sixteenths above dr_gh and those in dr_gl..dr_gh at or above the composite
    // dr_C; min_p rows (dr_bound) keep the tokens above the value bound.
    bool dr_bound = false;
    uint64_t dr_C = 0;
    int dr_gh = 0, dr_gl = 0;
    auto dr_wgt = [&](float v, int64_t gidx) -> float {
      if (gidx == (int64_t)x || v == -INFINITY) return 0.f;
      if (dr_bound) {
        if (!(v - M >= mp_thr)) return 0.f;
      } else {
        const int gx = six_i(v);
        if (!(gx > dr_gh || (gx >= dr_gl && comp_key(fkey(v), (uint32_t)gidx) >= dr_C))) return 0.f;
      }
      return ex2((v - M) * sl2);
    };
    // min_p without top-k: the kept set is every token with x - M >= T ln(min_p) (top-p
    // rows take this path when that bound lies above their nucleus cut). One pass over
    // the row: each warp sums the fixed-point weights of the passing tokens of its ranges
    // (the draft token left out) into the range slots, and notes the smallest passing
    // value; then the accept test and the draw over the ranges, as for top-p rows.
    auto minp_path = [&](auto) {  // generic: instantiated only where called (EXT)
      const int64_t E_ = (int64_t)nst * kCW;
      uint32_t kmin = minp_ranges<E>(xr, V, E_, SE, M, mp_thr, sl2, x, rowslots);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
      if (lane == 0) sm.redi[warp] = (int32_t)kmin;
      cbar();
      uint32_t km = 0xFFFFFFFFu;
      for (int w2 = 0; w2 < kCW; ++w2) km = min(km, (uint32_t)sm.redi[w2]);
      const uint64_t Cm = comp_key(km, kIdxMax);
      const int64_t per = (E_ + kCC - 1) / kCC;
      const int64_t e0 = min(E_, (int64_t)tid * per), e1 = min(E_, e0 + per);
      uint64_t mine = 0;
      for (int64_t e = e0; e < e1; ++e) mine += __ldcg(rowslots + e);
      uint64_t Zr;
      const uint64_t ex = sel::excl_scan<kCC, CBar>(mine, sm.sc, Zr);
      const uint64_t wx = (xvalid && vx - M >= mp_thr) ? wfn(vx) : 0ull;
      const int32_t acc = accept((double)(Zr + wx), (double)wx);
      if (skip_draw) {
        if (tid == 0) finish_row(-1, acc, 1, Cm, Zr + wx);
      } else if (Zr == 0) {
        if (tid == 0) finish_row((wx > 0) ? x : am, acc, 1, Cm, Zr + wx);
      } else {
        dr_bound = true;
        draw_ranges(mine, ex, Zr, e0, e1, acc, 1, Cm, Zr + wx, dr_wgt);
      }
    };

    // The general path for the rows the streamed summaries cannot serve (top_k above
    // kSTopK, candidate overflow, a top-p crossing outside its windows): radix selections
    // over the whole row, read again from memory for every digit, in the order top-k,
    // top-p within it, then the draw in token-id order.
    auto general = [&]() {
      if (tid == 0) atomicAdd(&a.ws.work[2], 1u);
      const int n = (int)V;
      auto gitem = [&](int i) -> uint64_t {
        return comp_key(fkey(SVec<E>::at(xr, i)), (uint32_t)i);
      };
      auto gmass = [&](uint64_t c0) -> uint64_t {
        uint64_t sum = 0;
        for (int64_t vi = tid; vi < nvall; vi += kCC) {
          float xv[N];
          load_vec(vi, xv);
#pragma unroll
          for (int q = 0; q < N; ++q) {
            const int64_t i = vi * N + q;
            const uint64_t cc = comp_key(fkey(xv[q]), (uint32_t)i);
            if (i < n && cc >= c0) sum += wfn(xv[q]);
          }
        }
        uint64_t tot;
        (void)sel::excl_scan<kCC, CBar>(sum, sm.sc, tot);
        return tot;
      };
      const bool tk = k > 0 && (int64_t)k < V;
      uint64_t C = 1;  // every composite key is at least 1
      if (tk)
        C = sel::radix_adaptive<kCC, false, CBar, 4>(
            n, gitem, 1ull, (uint64_t)k, [](uint64_t) { return (uint64_t)1; }, lowv, sm.sc);
      uint64_t Z = gmass(C);
      if (kn.tp < 1.f) {
        // top-k first: the nucleus of the top-k set; joint: the nucleus of the whole row,
        // intersected with the top-k set (the larger threshold)
        const bool jt = EXT && a.joint && tk;
        const uint64_t Zref = jt ? gmass(1ull) : Z;
        const double want = ceil((double)kn.tp * (double)Zref);
        const uint64_t P = (want > (double)Zref) ? Zref : (uint64_t)want;
        const uint64_t Cp =
            sel::radix_adaptive<kCC, true, CBar, 4>(n, gitem, jt ? 1ull : C, P, wcomp, lowv, sm.sc);
        C = max(C, Cp);
        Z = gmass(C);
      }
      if (use_mp) {
        // min_p: of the kept tokens, those with x - M >= T ln(min_p); the passing values
        // form a top segment, so the smallest passing key bounds them (the argmax passes)
        const float thr = kn.T * logf(kn.mp);
        uint32_t kmin = 0xFFFFFFFFu;
        for (int64_t vi = tid; vi < nvall; vi += kCC) {
          float xv[N];
          load_vec(vi, xv);
#pragma unroll
          for (int q = 0; q < N; ++q)
            if (xv[q] - M >= thr) kmin = min(kmin, fkey(xv[q]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
        if (lane == 0) sm.redi[warp] = (int32_t)kmin;
        cbar();
        uint32_t km = 0xFFFFFFFFu;
        for (int w2 = 0; w2 < kCW; ++w2) km = min(km, (uint32_t)sm.redi[w2]);
        cbar();
        const uint64_t Cm = comp_key(min(km, fkey(M)), kIdxMax);
        if (Cm > C) {
          C = Cm;
          Z = gmass(C);
        }
      }
      uint64_t wx = 0;
      if (xvalid && comp_key(fkey(vx), (uint32_t)x) >= C) wx = wfn(vx);
      const int32_t acc = accept((double)Z, (double)wx);
      if (skip_draw) {
        if (tid == 0) finish_row(-1, acc, 1, C, Z);
        return;
      }
      const uint64_t Zr = Z - wx;
      int32_t tok;
      if (Zr == 0) {
        tok = (wx > 0) ? x : am;
      } else {
        uint64_t t = (uint64_t)((double)uD * (double)Zr);
        if (t >= Zr) t = Zr - 1;
        const int idx_sh[3] = {16, 8, 0};
        uint64_t gsel = 0;
        (void)sel::radix<kCC, true, CBar, 4>(
            n, gitem, C, t + 1,
            [&](uint64_t cc) { return ((int32_t)comp_token(cc) == x) ? 0ull : wcomp(cc); },
            idx_sh, 3, sm.sc, &gsel);
        tok = (int32_t)comp_token(gsel);
      }
      if (tid == 0) finish_row(tok, acc, 1, C, Z);
    };

    // Top-k rows with the joint order measure top_p on the whole row's mass (one more
    // pass over the row, every compute thread); with min_p they keep only the tokens at
    // or above the value bound thr_v (x - M >= T ln(min_p)).
    const bool jrow = EXT && a.joint && kn.kind == kCTopK && kn.tp < 1.f && !bad;
    uint64_t Zall = 0;
    if (jrow) {
      uint64_t sum = 0;
      for (int64_t vi = tid; vi < nvall; vi += kCC) {
        float xv[N];
        load_vec(vi, xv);
#pragma unroll
        for (int q = 0; q < N; ++q) sum += wfn(xv[q]);
      }
      (void)sel::excl_scan<kCC, CBar>(sum, sm.sc, Zall);
    }

    // ---- finish the row ---------------------------------------------------------------------
    bool go_minp = false;  // set by the kinds that leave the row to the min_p path
    if (kn.kind == kCGreedy) {
      if (tid == 0) finish_row(am, (j < D && x == am) ? 1 : 0);
    } else if (bad || kn.kind == kCGeneral) {
      general();
    } else if (kn.kind == kCTopP) {
      // the crossing elements resolved exactly; the kept ones join their ranges
      const uint32_t cnt = sm.lcnt;
      const int ghi = sm.gh, gli = sm.gl;
      const int64_t E_ = (int64_t)nst * kCW;
      const int64_t per = (E_ + kCC - 1) / kCC;
      const int64_t e0 = min(E_, (int64_t)tid * per), e1 = min(E_, e0 + per);
      uint64_t mine = 0;
      for (int64_t e = e0; e < e1; ++e) mine += __ldcg(rowslots + e);
      uint64_t Zab;
      (void)sel::excl_scan<kCC, CBar>(mine, sm.sc, Zab);
      // the draft token's weight if it lies above the collected sixteenths
      const bool xabove = xvalid && six_i(vx) > ghi;
      const uint64_t A = Zab + (xabove ? wfn(vx) : 0ull);
      const uint64_t P = sm.ptarget;
      uint64_t lmass = 0;
      for (uint32_t i = tid; i < min(cnt, (uint32_t)kCCap); i += kCC) lmass += wcomp(sm.w.list[i]);
      uint64_t Lt;
      (void)sel::excl_scan<kCC, CBar>(lmass, sm.sc, Lt);
      if (cnt > (uint32_t)kCCap || cnt == 0 || P <= A || P > A + Lt) {
        general();
      } else {
        const uint64_t C = sel::radix_adaptive<kCC, true, CBar>(
            (int)cnt, [&](int i) { return sm.w.list[i]; }, 1ull, P - A, wcomp, lowv, sm.sc);
        if (use_mp && !mp_keep(C)) {  // min_p's bound lies above the nucleus cut: it decides
          go_minp = true;
        } else {
          for (uint32_t i = tid; i < cnt; i += kCC) {
            const uint64_t cc = sm.w.list[i];
            const uint32_t gidx = comp_token(cc);
            if (cc >= C && (int32_t)gidx != x)
              atomicAdd(reinterpret_cast<unsigned long long*>(
                            rowslots + (gidx / N) / (kCVecs * 32)),
                        (unsigned long long)wcomp(cc));
          }
          cbar();
          auto kept = [&](float v, int64_t gidx) -> bool {
            const int gx = six_i(v);
            if (gx > ghi) return true;
            return gx >= gli && comp_key(fkey(v), (uint32_t)gidx) >= C;
          };
          uint64_t wx = 0;
          if (xvalid && kept(vx, x)) wx = wfn(vx);
          mine = 0;
          for (int64_t e = e0; e < e1; ++e) mine += __ldcg(rowslots + e);
          uint64_t Zr;
          const uint64_t ex = sel::excl_scan<kCC, CBar>(mine, sm.sc, Zr);
          const int32_t acc = accept((double)(Zr + wx), (double)wx);
          if (skip_draw) {
            if (tid == 0) finish_row(-1, acc, 3, C, Zr + wx);
          } else if (Zr == 0) {
            if (tid == 0) finish_row((wx > 0) ? x : am, acc, 3, C, Zr + wx);
          } else {
            dr_C = C;
            dr_gh = ghi;
            dr_gl = gli;
            draw_ranges(mine, ex, Zr, e0, e1, acc, 3, C, Zr + wx, dr_wgt);
          }
        }
      }
    } else if (kn.kind == kCTopK && (int)sm.lcnt <= 32 * kCSmallE) {
      // few candidates: every compute thread ranks one of them by counting (composites
      // are distinct, so the ranks are a permutation), then one warp finishes the row
      // (compact loops, so that this code, run once a row, stays small)
      uint64_t* srt = sm.w.list + kCHalf;  // the candidates by rank (value order)
      {
        const int nl = (int)sm.lcnt;
        for (int i = tid; i < nl; i += kCC) {
          const uint64_t ci = sm.w.list[i];
          int r = 0;
          for (int jj = 0; jj < nl; ++jj) r += (sm.w.list[jj] > ci) ? 1 : 0;
          srt[r] = ci;
        }
      }
      cbar();
      if (warp == 0) {
        const int nl = (int)sm.lcnt;
        uint64_t* wid = sm.w.list + kCHalf + 128;  // kept: weight by rank in id order
        uint32_t* kid = reinterpret_cast<uint32_t*>(sm.w.list + kCHalf + 256);  // kept ids
        uint64_t v[kCSmallE], w[kCSmallE], incl[kCSmallE];
#pragma unroll
        for (int e = 0; e < kCSmallE; ++e) {
          const int i = e * 32 + lane;  // rank
          v[e] = (i < nl) ? srt[i] : 0ull;
          w[e] = (i < nl && i < k) ? wcomp(v[e]) : 0ull;
          incl[e] = w[e];
        }
        const uint64_t Zk = warp_scan_incl(incl);
        // top-p within the top k: rank r kept iff r = 0 or the mass before it is below P
        // (P a fraction of the top-k mass, or of the whole row's with the joint order);
        // min_p then keeps the ranks whose value passes its bound
        uint64_t P = Zk;
        if (kn.tp < 1.f) {
          const uint64_t Zref = jrow ? Zall : Zk;
          const double want = ceil((double)kn.tp * (double)Zref);
          P = (want > (double)Zref) ? Zref : (want > 0.0 ? (uint64_t)want : 0ull);
        }
        uint64_t Z = 0, wx = 0;
        bool kept[kCSmallE];
#pragma unroll
        for (int e = 0; e < kCSmallE; ++e) {
          const int i = e * 32 + lane;
          kept[e] = i < nl && i < k && (i == 0 || (incl[e] - w[e] < P && mp_keep(v[e])));
          const uint32_t tk = comp_token(v[e]);
          if (kept[e]) {
            Z += w[e];
            if ((int32_t)tk == x) wx = w[e];
          }
          if (i < 128) kid[i] = kept[e] ? tk : 0xFFFFFFFFu;
        }
        Z = warp_sum_u64(Z);
        wx = warp_sum_u64(wx);
        const int32_t acc = accept((double)Z, (double)wx);
        // the kept set is a prefix of the value order: its smallest composite bounds it
        uint64_t Cmin = ~0ull;
#pragma unroll
        for (int e = 0; e < kCSmallE; ++e)
          if (kept[e] && v[e] < Cmin) Cmin = v[e];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const uint64_t y = __shfl_xor_sync(0xffffffffu, Cmin, o);
          Cmin = y < Cmin ? y : Cmin;
        }
        const uint64_t Zr = skip_draw ? 0ull : Z - wx;
        int32_t tok = skip_draw ? -1 : ((wx > 0) ? x : (int32_t)comp_token(srt[0]));  // srt[0]: the argmax
        if (Zr > 0) {
          uint64_t t = (uint64_t)((double)uD * (double)Zr);
          if (t >= Zr) t = Zr - 1;
          __syncwarp();
          // the kept tokens in id order (their rank among the kept ids), the draft token
          // without weight
#pragma unroll
          for (int e = 0; e < kCSmallE; ++e) {
            const int i = e * 32 + lane;
            if (!kept[e]) continue;
            const uint32_t tk = kid[i];
            int r = 0;
            for (int jj = 0; jj < nl && jj < 128; ++jj) r += (kid[jj] < tk) ? 1 : 0;
            wid[r] = ((int32_t)tk == x) ? 0ull : w[e];
            kid[128 + r] = tk;
          }
          __syncwarp();
          const int nk = __popc(__ballot_sync(0xffffffffu, kept[0])) +
                         __popc(__ballot_sync(0xffffffffu, kept[1])) +
                         __popc(__ballot_sync(0xffffffffu, kept[2])) +
                         __popc(__ballot_sync(0xffffffffu, kept[3]));
          uint64_t cw[kCSmallE], ww[kCSmallE];
#pragma unroll
          for (int e = 0; e < kCSmallE; ++e) {
            const int i = e * 32 + lane;
            ww[e] = (i < nk) ? wid[i] : 0ull;
            cw[e] = ww[e];
          }
          (void)warp_scan_incl(cw);
          // the first token whose inclusive prefix mass exceeds t
          int32_t f = INT32_MAX;
#pragma unroll
          for (int e = 0; e < kCSmallE; ++e) {
            const int i = e * 32 + lane;
            if (i < nk && ww[e] > 0 && cw[e] > t && cw[e] - ww[e] <= t) f = (int32_t)kid[128 + i];
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) f = min(f, __shfl_xor_sync(0xffffffffu, f, o));
          if (f != INT32_MAX) tok = f;
        }
        if (lane == 0) finish_row(tok, acc, 1, Cmin, Z);
      }
    } else if (kn.kind == kCTopK) {
      const int nl = (int)sm.lcnt;
      auto item = [&](int i) { return sm.w.list[i]; };
      const uint64_t Ck = sel::radix_adaptive<kCC, false, CBar>(
          nl, item, 1ull, (uint64_t)k, [](uint64_t) { return (uint64_t)1; }, lowv, sm.sc);
      auto mass_from = [&](uint64_t c0) -> uint64_t {
        uint64_t sum = 0;
        for (int i = tid; i < nl; i += kCC) {
          const uint64_t cc = sm.w.list[i];
          if (cc >= c0) sum += wcomp(cc);
        }
        uint64_t tot;
        (void)sel::excl_scan<kCC, CBar>(sum, sm.sc, tot);
        return tot;
      };
      uint64_t C = Ck, Z = mass_from(Ck);
      if (kn.tp < 1.f) {
        // top-k first: the nucleus of the top-k set; joint: the nucleus of the whole row
        // (its mass Zall), which cuts inside the top k only if P is within their mass
        const uint64_t Zref = jrow ? Zall : Z;
        const double want = ceil((double)kn.tp * (double)Zref);
        const uint64_t P = (want > (double)Zref) ? Zref : (want > 0.0 ? (uint64_t)want : 0ull);
        if (P <= Z) {
          C = sel::radix_adaptive<kCC, true, CBar>(nl, item, Ck, P, wcomp, lowv, sm.sc);
          Z = mass_from(C);
        }
      }
      if (use_mp) {
        // min_p: the smallest kept list value that passes the bound (the argmax does)
        uint32_t kmin = fkey(M);
        for (int i = tid; i < nl; i += kCC) {
          const uint64_t cc = sm.w.list[i];
          if (cc >= C && mp_keep(cc)) kmin = min(kmin, (uint32_t)(cc >> kIdxBits));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
        if (lane == 0) sm.redi[warp] = (int32_t)kmin;
        cbar();
        uint32_t km = 0xFFFFFFFFu;
        for (int w2 = 0; w2 < kCW; ++w2) km = min(km, (uint32_t)sm.redi[w2]);
        cbar();
        const uint64_t Cm = comp_key(km, kIdxMax);
        if (Cm > C) {
          C = Cm;
          Z = mass_from(C);
        }
      }
      uint64_t wx = 0;
      if (xvalid && comp_key(fkey(vx), (uint32_t)x) >= C) wx = wfn(vx);
      const int32_t acc = accept((double)Z, (double)wx);
      const uint64_t Zr = skip_draw ? 0ull : Z - wx;
      int32_t tok = -1;
      if (skip_draw) {
      } else if (Zr == 0) {
        tok = (wx > 0) ? x : am;
      } else {
        uint64_t t = (uint64_t)((double)uD * (double)Zr);
        if (t >= Zr) t = Zr - 1;
        const int idx_sh[3] = {16, 8, 0};
        uint64_t gsel = 0;
        (void)sel::radix<kCC, true, CBar>(
            nl, item, C, t + 1,
            [&](uint64_t cc) { return ((int32_t)comp_token(cc) == x) ? 0ull : wcomp(cc); },
            idx_sh, 3, sm.sc, &gsel);
        tok = (int32_t)comp_token(gsel);
      }
      if (tid == 0) finish_row(tok, acc, 1, C, Z);
    } else if (use_mp) {  // kCPlain with min_p
      go_minp = true;
    } else {  // kCPlain: the warp ranges scaled to the row maximum, in token order
      const int64_t E_ = (int64_t)nst * kCW;
      const int64_t per = (E_ + kCC - 1) / kCC;
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
      const double ex = excl_scan_f64_t<kCW, CBar>(mine, sm.dscan, Zr);
      const double wx = xvalid ? (double)ex2((vx - M) * sl2) : 0.0;
      const int32_t acc = accept(Zr + wx, wx);
      const uint64_t Zfx = (uint64_t)((Zr + wx) * 1099511627776.0);
      if (skip_draw) {
        if (tid == 0) finish_row(-1, acc, 2, 1ull, Zfx);
      } else if (!(Zr > 0.0)) {
        if (tid == 0) finish_row((wx > 0.0) ? x : am, acc, 2, 1ull, Zfx);
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
          // the residual in the range's own weight units (relative to its maximum)
          sm.res_d = (t - rs) / (m > 0.0 ? (double)ex2((em - M) * sl2) : 1.0);
        }
        cbar();
        if (warp == 0) {
          const int64_t es = min((int64_t)(sm.res_u % (uint64_t)e1max), e1max - 1);
          const float em = sm.redf[0][0];
          const int64_t v0 = (es / kCW) * (SE / N) + (es % kCW) * (kCVecs * 32);
          const int32_t tok = walk_range(v0, (float)sm.res_d, [&](float v, int64_t gidx) -> float {
            return (gidx == (int64_t)x || v == -INFINITY) ? 0.f : ex2((v - em) * sl2);
          });
          if (lane == 0) finish_row(tok >= 0 ? tok : am, acc, 2, 1ull, Zfx);
        }
      }
    }
    if constexpr (EXT) {
      if (go_minp) minp_path(0);
    }
    cbar();  // the row's shared state is free for the next row
  }

}


// The chain of every request whose rows have all recorded their results (TokenSpeed
// verify(): the accepted draft prefix, then the row's corrected or bonus token): accepted
// tokens (-1 past the chain), accept index, logprobs and accept_length. A request with a
// row left unrecorded (a stage wait that gave up) keeps accept_length = 0 from the
// planning launch; with draft probabilities the rejected position is left to
// k_chain_resid. One warp a request: lane j takes position j (and j + 32, ...).
template <typename E>
__global__ void __launch_bounds__(256) k_chain_write(SampleArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t req = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (req >= a.nreq) return;
  const CWin win = cwin(a, req);
  if (win.count < 1 || __ldcg(&a.ws.creq[req]) != (uint32_t)win.count) return;
  const int64_t rbase = win.first;
  const int32_t D = win.count - 1;
  const int32_t DP = a.D;
  const int64_t V = a.V;
  const bool qmode = a.q != nullptr;
  // the first rejected position (D if every draft is accepted)
  int32_t js = D;
  for (int32_t j0 = 0; j0 < D; j0 += 32) {
    const int32_t jj = j0 + lane;
    const bool rej = jj < D && !__ldcg(&a.ws.rowres[rbase + jj].acc);
    const unsigned m = __ballot_sync(0xffffffffu, rej);
    if (m) {
      js = j0 + __ffs(m) - 1;
      break;
    }
  }
  // positions of the padded outputs; a ragged window's rows past it read as unused
  for (int32_t jj = lane; jj < a.R; jj += 32) {
    const int64_t oj = req * a.R + jj;
    const int64_t rj = rbase + jj;  // the packed row of position jj (jj <= D)
    int32_t t = -1;
    if (jj < js) t = a.draft_tokens[req * DP + jj];
    else if (jj == js) t = __ldcg(&a.ws.rowres[rj].tok);
    if (qmode && jj == js && js < D) {  // the residual kernel writes this position
      if (a.accept_index) a.accept_index[oj] = (int32_t)rj;
      continue;
    }
    a.accepted_tokens[oj] = t;
    if (a.accept_index) a.accept_index[oj] = (jj <= js) ? (int32_t)rj : -1;
    if (a.logprobs) {
      float lp = 0.f;
      if (jj <= js && t >= 0 && (int64_t)t < V) {
        const E* xj = reinterpret_cast<const E*>(a.x) + rj * a.ld;
        lp = (SVec<E>::at(xj, t) - __ldcg(&a.ws.rowres[rj].M)) -
             logf(__ldcg(&a.ws.rowres[rj].S));
      }
      a.logprobs[oj] = lp;
    }
  }
  if (lane == 0) a.accept_length[req] = js + 1;
}

// With draft probabilities, the residual draw of every request rejected before its last
// row (TensorRT-LLM rejection_sampling_one_model: at the first rejection j*, a token from
// norm(max(p - q, 0))): p''_j* is recomputed from the row's recorded kept set (its
// weights over the recorded kept mass), the residual max(p'' - q, 0) is formed
// elementwise in fp32 and summed in 2^-40 fixed point, and the draw is the smallest token
// id whose inclusive prefix mass exceeds u_D times the total (a zero residual draws from
// p''). One CTA per request; it writes accepted_tokens[b, j*] and its logprob.
// p''_i of a finished row from its record: the kept set (by kind: the argmax; tokens at
// or above the composite C; every token; or the sixteenths above gh plus those in
// gl..gh at or above C) and the weight 2^((v - M) log2(e) / T) in 2^-40 units over the
// kept mass Zk.
struct KeptRow {
  float M, sl2, s16, invZ;
  uint64_t C;
  int32_t am, gh, gl, kind;

  __device__ __forceinline__ void load(const RowRes* rp, float T) {
    M = __ldcg(&rp->M);
    am = __ldcg(&rp->am);
    kind = __ldcg(&rp->kind);
    C = __ldcg(&rp->C);
    const uint64_t Zk = __ldcg(&rp->Zk);
    gh = __ldcg(&rp->gh);
    gl = __ldcg(&rp->gl);
    sl2 = kind != 0 ? __fdiv_rn(kLog2e, T) : 0.f;
    s16 = sl2 * 16.f;
    invZ = (float)(1.0 / (double)(Zk ? Zk : 1ull));
  }
  __device__ __forceinline__ int six_i(float v) const {
    float t = __fmaf_rd(v, s16, 12582912.f);
    t = fminf(fmaxf(t, 8388608.f), 16777216.f);
    return __float_as_int(t) - 0x4B400000;
  }
  __device__ __forceinline__ float prob(float v, int64_t i) const {
    if (kind == 0) return (i == am) ? 1.f : 0.f;
    if (v == -INFINITY) return 0.f;
    bool kept = kind == 2;
    if (kind == 1) kept = comp_key(fkey(v), (uint32_t)i) >= C;
    if (kind == 3) {
      const int g = six_i(v);
      kept = g > gh || (g >= gl && comp_key(fkey(v), (uint32_t)i) >= C);
    }
    if (!kept) return 0.f;
    return __ull2float_rn(fixw(ex2((v - M) * sl2))) * invZ;
  }
};

// Single-step sampling with a probability output: row r's kept distribution p'' to its
// destination row (blockIdx.x the row, blockIdx.y a slice of `per` tokens). Rows the
// chain kernel did not finish are left unwritten.
template <typename E>
__global__ void __launch_bounds__(256) k_chain_probs(SampleArgs a, int64_t per) {
  const int64_t row = blockIdx.x;
  if (__ldcg(&a.accept_length[row]) != 1) return;
  KeptRow kr;
  kr.load(a.ws.rowres + row, cknobs(a, row).T);
  const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;
  float* dst = a.probs_out + (a.probs_row ? a.probs_row[row] : row) * a.ld_probs;
  const int64_t i0 = (int64_t)blockIdx.y * per, i1 = min(a.V, i0 + per);
  for (int64_t i = i0 + threadIdx.x; i < i1; i += 256) dst[i] = kr.prob(SVec<E>::at(xr, i), i);
}

template <typename E>
__global__ void __launch_bounds__(256) k_chain_resid(SampleArgs a) {
  __shared__ uint64_t tot[8];
  __shared__ int32_t s_tok;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t b = blockIdx.x;
  const CWin win = cwin(a, b);
  const int32_t D = win.count - 1, DP = a.D, R = a.R;
  const int32_t L = __ldcg(&a.accept_length[b]);
  if (L < 1 || L > D) return;  // every draft accepted (the bonus is drawn), or unfinished
  const int32_t js = L - 1;
  const int64_t row = win.first + js;  // the rejected row (packed), output position b R + js
  const RowRes* rp = a.ws.rowres + row;
  const float M = __ldcg(&rp->M);
  const int32_t am = __ldcg(&rp->am);
  const int32_t kind = __ldcg(&rp->kind);
  const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;
  int32_t tok = am;
  if (kind != 0) {
    KeptRow kr;
    kr.load(rp, cknobs(a, b).T);
    const float* qr = a.q + (b * DP + js) * a.ld_q;
    const int64_t V = a.V;
    // p''_i, and the residual weight of token i in fixed point
    auto pw = [&](int64_t i) -> float { return kr.prob(SVec<E>::at(xr, i), i); };
    auto rw = [&](int64_t i, bool from_p) -> uint64_t {
      const float p = pw(i);
      const float r = from_p ? p : fmaxf(p - qr[i], 0.f);
      return __float2ull_rz(r * kFx);
    };
    const int64_t Lw = ((V + 8 * 32 - 1) / (8 * 32)) * 32;  // a warp's contiguous block
    const int64_t w0 = min(V, (int64_t)warp * Lw), w1 = min(V, w0 + Lw);
    bool from_p = false;
    uint64_t Zr = 0;
    for (int round = 0; round < 2; ++round) {
      uint64_t wt = 0;
      for (int64_t i = w0 + lane; i < w1; i += 32) wt += rw(i, from_p);
      wt = warp_sum_u64(wt);
      if (lane == 0) tot[warp] = wt;
      __syncthreads();
      Zr = 0;
      for (int w2 = 0; w2 < 8; ++w2) Zr += tot[w2];
      if (Zr > 0 || from_p) break;
      from_p = true;  // a zero residual draws from p''
      __syncthreads();
    }
    if (Zr > 0) {
      const uint64_t seed = a.seed ? (uint64_t)a.seed[b] : 0;
      const uint64_t off = a.offset ? (uint64_t)a.offset[b] : 0;
      const float uD = a.uniforms ? a.uniforms[b * R + D] : verify_coin(seed, off, (uint32_t)D);
      uint64_t t = (uint64_t)((double)uD * (double)Zr);
      if (t >= Zr) t = Zr - 1;
      uint64_t acc = 0;
      int ws = 7;
      for (int w2 = 0; w2 < 8; ++w2) {
        if (t < acc + tot[w2]) {
          ws = w2;
          break;
        }
        acc += tot[w2];
      }
      if (warp == ws) {
        int32_t found = -1;
        for (int64_t s0 = w0; s0 < w1 && found < 0; s0 += 32) {
          const int64_t i = s0 + lane;
          const uint64_t wi = (i < w1) ? rw(i, from_p) : 0ull;
          uint64_t inc = wi;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
          }
          const unsigned hit = __ballot_sync(0xffffffffu, wi > 0 && acc + inc > t);
          if (hit) found = (int32_t)(s0 + __ffs(hit) - 1);
          acc += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (lane == 0) s_tok = found;
      }
      __syncthreads();
      if (s_tok >= 0) tok = s_tok;
    }
  }
  if (tid == 0) {
    const int64_t oj = b * R + js;
    a.accepted_tokens[oj] = tok;
    if (a.logprobs) {
      float lp = 0.f;
      if (tok >= 0 && (int64_t)tok < a.V)
        lp = (SVec<E>::at(xr, tok) - M) - logf(__ldcg(&a.ws.rowres[row].S));
      a.logprobs[oj] = lp;
    }
  }
}

template <typename E>
cudaError_t launch_chain_t(const SampleArgs& a, cudaStream_t s) {
  int dev = 0, nsm = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  k_chain_plan<<<1, 1024, 0, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t want = (int64_t)nsm * 2;  // two CTAs an SM
  const unsigned grid = (unsigned)(a.rows < want ? a.rows : want);
  const size_t dyn = (size_t)kCNSt * kCStageBytes + sizeof(CSmem);
  if (a.min_p || a.joint) {
    e = cudaFuncSetAttribute(k_chain<E, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dyn);
    if (e != cudaSuccess) return e;
    k_chain<E, true><<<grid, kCThreads, dyn, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(k_chain<E, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dyn);
    if (e != cudaSuccess) return e;
    k_chain<E, false><<<grid, kCThreads, dyn, s>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_chain_write<E><<<(unsigned)((a.nreq * 32 + 255) / 256), 256, 0, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.probs_out) {
    const int64_t per = 8192;
    k_chain_probs<E><<<dim3((unsigned)a.rows, (unsigned)((a.V + per - 1) / per)), 256, 0, s>>>(a, per);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || !a.q) return e;
  k_chain_resid<E><<<(unsigned)a.nreq, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chain(const SampleArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  return a.bf16 ? launch_chain_t<uint16_t>(a, s) : launch_chain_t<float>(a, s);
}

cudaError_t chain_read_error(uint32_t* word, int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_chain_err, sizeof(v));
  if (e != cudaSuccess) return e;
  *word = v;
  if (clear && v) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_chain_err, &z, sizeof(z));
  }
  return e;
}

}  // namespace tsv
