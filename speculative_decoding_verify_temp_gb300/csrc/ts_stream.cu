// Streaming row kernels: one pass over each needed row, split across CTAs, combined by
// the last CTA to finish (an atomic arrival counter in the workspace; no waiting).
//
//  k_rowstat<E, GUMBEL>  row argmax (lowest id on ties) and the temperature-1 log-sum-exp,
//                        then per kind: greedy chain verification (TokenSpeed
//                        flashinfer.py verify(): sampling_argmax + verify_chain_greedy),
//                        chosen-token logprobs (gather_token_logprobs_torch), or the
//                        temperature-only Gumbel-max draw (TensorRT-LLM interface.py,
//                        _sample_sharded_temperature).
//  k_softmax_smem        temperature softmax (TokenSpeed flashinfer.py verify():
//                        softmax(logits, temperature)): a cluster of CTAs per row, each
//                        CTA's slice brought into shared memory once by bulk copies, the
//                        row maximum and sum combined through distributed shared memory,
//                        the probabilities written from the staged copy.
//  k_softmax             the same for rows too long to stage: the slices are streamed
//                        twice.
//  k_draw_probs          chain speculative sampling on probability rows (TensorRT-LLM
//                        interface.py, rejection_sampling_one_model): the accept tests,
//                        then one streamed pass over the single row that the final
//                        (residual or bonus) draw needs.
#include <stdint.h>

#include <cooperative_groups.h>

#include "ts_common.cuh"
#include "ts_internal.h"

namespace cg = cooperative_groups;

namespace tsv {

constexpr int kStreamThreads = 256;
constexpr float kGumbelCap = 17.0f;  // > the largest noise -ln(-ln(1 - 2^-24)) = 16.64

template <typename E>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void unpack(const uint4& r, float* x) {
    x[0] = __uint_as_float(r.x);
    x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z);
    x[3] = __uint_as_float(r.w);
  }
  __device__ __forceinline__ static float scalar(const float* p, int64_t i) { return p[i]; }
};
template <>
struct Vec<uint16_t> {
  static constexpr int N = 8;
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
  __device__ __forceinline__ static float scalar(const uint16_t* p, int64_t i) {
    return bf16_bits_to_f32(p[i]);
  }
};

// Block-wide reduction of (argmax, lse) into thread 0; returns true on thread 0.
__device__ __forceinline__ void block_reduce_stat(float& bv, int32_t& bi, float& lm, float& ls) {
  __shared__ float s_v[32], s_m[32], s_s[32];
  __shared__ int32_t s_i[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  warp_argmax(bv, bi);
  warp_lse(lm, ls);
  if (lane == 0) {
    s_v[w] = bv;
    s_i[w] = bi;
    s_m[w] = lm;
    s_s[w] = ls;
  }
  __syncthreads();
  if (w == 0) {
    bv = lane < nw ? s_v[lane] : -INFINITY;
    bi = lane < nw ? s_i[lane] : INT32_MAX;
    lm = lane < nw ? s_m[lane] : -INFINITY;
    ls = lane < nw ? s_s[lane] : 0.f;
    warp_argmax(bv, bi);
    warp_lse(lm, ls);
  }
}

// ---------------------------------------------------------------------------------
// Row statistics: argmax + log-sum-exp, or the Gumbel-max argmax.

template <typename E, bool GUMBEL>
__global__ void __launch_bounds__(kStreamThreads) k_rowstat(RowStatArgs a) {
  constexpr int N = Vec<E>::N;
  const int64_t row = blockIdx.x / a.splits;
  if (!GUMBEL && a.req_temperature && a.req_temperature[row / (a.D + 1)] >= kGreedyT) return;
  const int split = (int)(blockIdx.x % a.splits);
  const int64_t lo = (int64_t)split * a.split_len;
  const int64_t hi = min(a.V, lo + a.split_len);
  const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;

  // Gumbel noise stream of this row
  bool noise = false;
  float invT = 1.f;
  uint32_t k0 = 0, k1 = 0, c1 = 0, c2 = 0, c3 = 0;
  if (GUMBEL) {
    const float T = a.temperature[row];
    noise = (T >= kGreedyT);
    invT = noise ? __frcp_rn(T) : 1.f;
    const int64_t b = row / a.n_per_req;
    const uint64_t seed = (uint64_t)a.seed[b], off = (uint64_t)a.offset[b];
    k0 = (uint32_t)seed;
    k1 = (uint32_t)(seed >> 32);
    c1 = (uint32_t)(row % a.n_per_req);
    c2 = (uint32_t)off;
    c3 = (uint32_t)(off >> 32);
  }

  float bv = -INFINITY;
  int32_t bi = INT32_MAX;
  float lm = -INFINITY, ls = 0.f, lc = 0.f;
  const bool lse = !GUMBEL && a.want_lse;
  // Gumbel: the best score any CTA of the row has published so far (a lower bound of the
  // row's best): an element group whose largest possible score is below it is skipped
  float wbound = -INFINITY;

  // Elements x[0..n) with indices base.. base+n-1, n a multiple of 4 for the vector path.
  auto visit = [&](const float* x, int n, int64_t base) {
    if (GUMBEL && noise) {
      for (int g = 0; g < n; g += 4) {
        const float gm = fmaxf(fmaxf(x[g], x[g + 1]), fmaxf(x[g + 2], x[g + 3]));
        if (gm * invT + kGumbelCap >= fmaxf(bv, wbound)) {
          const uint32_t gi = (uint32_t)((base + g) >> 2);
          const uint4 r = philox4x32_10(make_uint4(gi, c1, c2, c3), k0, k1);
          const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
          const float bound = fmaxf(bv, wbound);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (x[g + k] == -INFINITY) continue;
            const float u = u01(wv[k]);
            const float xs = x[g + k] * invT;
            // -ln(-ln u) <= -ln(1 - u) (1 - u is exact): an element whose bound, with a
            // margin far above the fast log's error, stays below the best cannot win
            if (xs - __logf(1.f - u) + 1e-3f < bound) continue;
            const float e = -logf(u);
            const float s = xs - __logf(e);
            if (s > bv) {
              bv = s;
              bi = (int32_t)(base + g + k);
            }
          }
        }
      }
      return;
    }
    float vm = x[0];
    for (int k = 1; k < n; ++k) vm = fmaxf(vm, x[k]);
    if (vm > bv) {
      for (int k = 0; k < n; ++k)
        if (x[k] == vm) {
          bi = (int32_t)(base + k);
          break;
        }
      bv = vm;
    }
    if (lse && vm > -INFINITY) {
      const float nm = fmaxf(lm, vm);
      const float f = ex2((lm - nm) * kLog2e);
      ls *= f;
      lc *= f;
      lm = nm;
      float vs = 0.f;
      for (int k = 0; k < n; ++k) vs += ex2((x[k] - nm) * kLog2e);
      kahan_add(ls, lc, vs);
    }
  };

  if (a.vec) {
    const int64_t nv = (hi - lo) / N;
    const uint4* vp = reinterpret_cast<const uint4*>(xr + lo);
    constexpr int U = 4;
    // rounds of U vectors a thread (the same count for every thread of the CTA)
    const int64_t rounds = (nv + U * kStreamThreads - 1) / (U * kStreamThreads);
    for (int64_t rd = 0; rd < rounds; ++rd) {
      const int64_t vi = rd * (U * kStreamThreads) + threadIdx.x;
      uint4 r[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (vi + u * kStreamThreads < nv) r[u] = ldg_stream(vp + vi + u * kStreamThreads);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (vi + u * kStreamThreads >= nv) continue;
        float x[N];
        Vec<E>::unpack(r[u], x);
        visit(x, N, lo + (vi + u * kStreamThreads) * N);
      }
      if (GUMBEL && noise) {
        // publish the warp's best score to the row and take the row's best back
        float m = bv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float rb = m;
        if ((threadIdx.x & 31) == 0) {
          const uint32_t old = atomicMax(&a.ws.best[row], m > -INFINITY ? fkey(m) : 0u);
          if (old != 0u) rb = fmaxf(rb, key_to_value(old));
        }
        wbound = __shfl_sync(0xffffffffu, rb, 0);
      }
    }
    // ragged tail: fewer than N elements, padded with -inf to a multiple of 4
    const int64_t t0 = lo + nv * N;
    if (threadIdx.x == 0 && t0 < hi) {
      float x[8];
      int n = (int)(hi - t0);
      for (int k = 0; k < 8; ++k) x[k] = k < n ? Vec<E>::scalar(xr, t0 + k) : -INFINITY;
      visit(x, (n + 3) & ~3, t0);
    }
  } else {
    for (int64_t g = lo + 4 * (int64_t)threadIdx.x; g < hi; g += 4 * kStreamThreads) {
      float x[4];
      for (int k = 0; k < 4; ++k) x[k] = (g + k < hi) ? Vec<E>::scalar(xr, g + k) : -INFINITY;
      visit(x, 4, g);
    }
  }
  ls += lc;  // fold the compensation in before combining

  block_reduce_stat(bv, bi, lm, ls);

  __shared__ int s_last;
  if (threadIdx.x == 0) {
    a.ws.part[row * kMaxSplits + split] = Part{bv, bi, lm, ls};
    __threadfence();
    const uint32_t prev = atomicAdd(&a.ws.rowcnt[row], 1u);
    s_last = (prev == (uint32_t)a.splits - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Last CTA of the row: combine the splits in order.
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float v = -INFINITY, m = -INFINITY, s = 0.f;
    int32_t i = INT32_MAX;
    for (int k = lane; k < a.splits; k += 32) {
      const Part* pp = &a.ws.part[row * kMaxSplits + k];
      const float v2 = __ldcg(&pp->v), m2 = __ldcg(&pp->m), s2 = __ldcg(&pp->s);
      const int32_t i2 = __ldcg(&pp->i);
      argmax_merge(v, i, v2, i2);
      lse_merge(m, s, m2, s2);
    }
    warp_argmax(v, i);
    warp_lse(m, s);
    if (lane == 0) {
      a.ws.rowcnt[row] = 0;
      if (GUMBEL) a.ws.best[row] = 0;
      const int32_t am = (i == INT32_MAX) ? 0 : i;
      if (a.kind == 2) {
        a.tokens_out[row] = am;
      } else if (a.kind == 1) {
        const int32_t t = a.lp_tokens[row];
        float lp = 0.f;
        if (t >= 0 && (int64_t)t < a.V) lp = (Vec<E>::scalar(xr, t) - m) - logf(s);
        a.lp_out[row] = lp;
      } else {
        // greedy chain verification: publish the row, the last row of the request writes
        a.ws.rowres[row] = RowRes{m, am, s, -1, 0, {0, 0, 0}};
        __threadfence();
        const int32_t R = a.D + 1;
        // the request's window of rows [first, first + cnt): a ragged batch finds it by
        // bisection of qo (a window that does not fit is left unverified)
        int64_t b = row / R, first = b * R;
        int32_t cnt = R;
        if (a.qo) {
          int64_t lo = 0, hi = a.nreq - 1;
          while (lo < hi) {
            const int64_t mid = (lo + hi + 1) / 2;
            if ((int64_t)a.qo[mid] <= row) lo = mid;
            else hi = mid - 1;
          }
          b = lo;
          first = a.qo[b];
          const int64_t e = a.qo[b + 1];
          cnt = (first <= row && row < e && e <= a.rows && e - first <= R) ? (int32_t)(e - first)
                                                                             : 0;
        }
        const int32_t Db = cnt - 1;
        const uint32_t prev = cnt > 0 ? atomicAdd(&a.ws.reqcnt[b], 1u) : 0u;
        if (cnt > 0 && prev == (uint32_t)Db) {
          __threadfence();
          a.ws.reqcnt[b] = 0;
          int32_t js = Db;
          for (int32_t j = 0; j < Db; ++j) {
            if (a.draft_tokens[b * a.D + j] != __ldcg(&a.ws.rowres[first + j].am)) {
              js = j;
              break;
            }
          }
          for (int32_t j = 0; j < R; ++j) {
            const int64_t oj = b * R + j;  // the padded output position
            const int64_t rj = first + j;  // its packed row (j <= js)
            int32_t tok = -1;
            if (j < js) tok = a.draft_tokens[b * a.D + j];
            else if (j == js) tok = __ldcg(&a.ws.rowres[rj].am);
            a.accepted_tokens[oj] = tok;
            if (a.accept_index) a.accept_index[oj] = (j <= js) ? (int32_t)rj : -1;
            if (a.logprobs) {
              float lp = 0.f;
              if (j <= js) {
                const E* xj = reinterpret_cast<const E*>(a.x) + rj * a.ld;
                lp = (Vec<E>::scalar(xj, tok) - __ldcg(&a.ws.rowres[rj].M)) -
                     logf(__ldcg(&a.ws.rowres[rj].S));
              }
              a.logprobs[oj] = lp;
            }
          }
          a.accept_length[b] = js + 1;
        }
      }
    }
  }
}

cudaError_t launch_rowstat(const RowStatArgs& a, int bf16, cudaStream_t s) {
  const dim3 grid((unsigned)(a.rows * a.splits));
  if (a.kind == 2) {
    if (bf16) k_rowstat<uint16_t, true><<<grid, kStreamThreads, 0, s>>>(a);
    else k_rowstat<float, true><<<grid, kStreamThreads, 0, s>>>(a);
  } else {
    if (bf16) k_rowstat<uint16_t, false><<<grid, kStreamThreads, 0, s>>>(a);
    else k_rowstat<float, false><<<grid, kStreamThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// Chain speculative sampling on probability rows.

// Inclusive block scan of a float (fixed order: lanes, then warps).
__device__ __forceinline__ float block_incl_scan(float v, float* s_w, float& total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) s_w[w] = v;
  __syncthreads();
  if (w == 0) {
    float t = lane < nw ? s_w[lane] : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < nw) s_w[lane] = t;
  }
  __syncthreads();
  const float excl_w = (w > 0) ? s_w[w - 1] : 0.f;
  total = s_w[nw - 1];
  __syncthreads();
  return v + excl_w;
}

__global__ void __launch_bounds__(kStreamThreads) k_draw_probs(DrawArgs a) {
  const int64_t b = blockIdx.x / a.splits;
  const int split = (int)(blockIdx.x % a.splits);
  const int32_t R = a.D + 1;
  __shared__ int32_t s_js, s_x;
  __shared__ float s_uD;

  // 1. the accept tests (every CTA of the request repeats them: D scalar pairs)
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const uint64_t seed = a.seed ? (uint64_t)a.seed[b] : 0, off = a.offset ? (uint64_t)a.offset[b] : 0;
    int32_t js = a.D;
    for (int32_t j0 = 0; j0 < a.D; j0 += 32) {
      const int32_t j = j0 + lane;
      bool fail = false;
      if (j < a.D) {
        const int32_t x = a.drafts[b * a.D + j];
        const bool valid = x >= 0 && (int64_t)x < a.V;
        const float u = a.uniforms ? a.uniforms[b * R + j] : verify_coin(seed, off, (uint32_t)j);
        const float px = valid ? a.p[(b * R + j) * a.ld + x] : 0.f;
        if (a.q) {
          const float qx = valid ? a.q[(b * a.D + j) * a.ld_q + x] : 0.f;
          fail = !(__fmul_rn(u, qx) < px);
        } else {
          fail = !(u < px);
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, fail);
      if (m) {
        js = j0 + __ffs(m) - 1;
        break;
      }
    }
    if (lane == 0) {
      s_js = js;
      s_x = (js < a.D) ? a.drafts[b * a.D + js] : -1;
      s_uD = a.uniforms ? a.uniforms[b * R + a.D] : verify_coin(seed, off, (uint32_t)a.D);
    }
  }
  __syncthreads();
  const int32_t js = s_js, x = s_x;
  const bool resid_q = (js < a.D) && a.q != nullptr;
  const int64_t r = b * R + js;
  const float* pr = a.p + r * a.ld;
  const float* qr = resid_q ? a.q + (b * a.D + js) * a.ld_q : nullptr;

  // w_i: the residual max(p - q, 0) formed in fp32, or p with the draft removed, or p.
  auto weight = [&](float p, float q, int64_t i) -> float {
    if (resid_q) {
      const float d = __fsub_rn(p, q);
      return d > 0.f ? d : 0.f;
    }
    return (i == (int64_t)x) ? 0.f : p;
  };

  // 2. mass of this split (residual and base)
  const int64_t lo = (int64_t)split * a.split_len;
  const int64_t hi = min(a.V, lo + a.split_len);
  float ws = 0.f, wc = 0.f, bs = 0.f, bc = 0.f;
  if (a.vec) {
    const int64_t nv = (hi - lo) / 4;
    const uint4* pv = reinterpret_cast<const uint4*>(pr + lo);
    const uint4* qv = resid_q ? reinterpret_cast<const uint4*>(qr + lo) : nullptr;
    for (int64_t vi = threadIdx.x; vi < nv; vi += kStreamThreads) {
      float p[4], q[4] = {0.f, 0.f, 0.f, 0.f};
      Vec<float>::unpack(ldg_stream(pv + vi), p);
      if (resid_q) Vec<float>::unpack(ldg_stream(qv + vi), q);
      const int64_t i0 = lo + vi * 4;
      float w4 = 0.f, b4 = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w4 += weight(p[k], q[k], i0 + k);
        b4 += p[k];
      }
      kahan_add(ws, wc, w4);
      kahan_add(bs, bc, b4);
    }
    for (int64_t i = lo + nv * 4 + threadIdx.x; i < hi; i += kStreamThreads) {
      const float p = pr[i], q = resid_q ? qr[i] : 0.f;
      kahan_add(ws, wc, weight(p, q, i));
      kahan_add(bs, bc, p);
    }
  } else {
    for (int64_t i = lo + threadIdx.x; i < hi; i += kStreamThreads) {
      const float p = pr[i], q = resid_q ? qr[i] : 0.f;
      kahan_add(ws, wc, weight(p, q, i));
      kahan_add(bs, bc, p);
    }
  }
  ws += wc;
  bs += bc;
  __shared__ float s_red[2][32];
  {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ws += __shfl_xor_sync(0xffffffffu, ws, o);
      bs += __shfl_xor_sync(0xffffffffu, bs, o);
    }
    if (lane == 0) {
      s_red[0][w] = ws;
      s_red[1][w] = bs;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float t0 = 0.f, t1 = 0.f;
      for (int k = 0; k < (int)(blockDim.x >> 5); ++k) {
        t0 += s_red[0][k];
        t1 += s_red[1][k];
      }
      ws = t0;
      bs = t1;
    }
  }

  __shared__ int s_last;
  if (threadIdx.x == 0) {
    a.ws.dpart[b * kMaxSplits + split] = DrawPart{ws, bs};
    __threadfence();
    const uint32_t prev = atomicAdd(&a.ws.reqcnt[b], 1u);
    s_last = (prev == (uint32_t)a.splits - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // 3. last CTA of the request: locate the split, then the token, in token-id order
  __shared__ int s_split, s_fallback;
  __shared__ float s_t;
  if (threadIdx.x == 0) {
    float Z = 0.f, Zb = 0.f;
    for (int k = 0; k < a.splits; ++k) {
      Z += __ldcg(&a.ws.dpart[b * kMaxSplits + k].w);
      Zb += __ldcg(&a.ws.dpart[b * kMaxSplits + k].b);
    }
    const int fb = !(Z > 0.f);  // zero residual: draw from p itself
    if (fb) Z = Zb;
    float t = __fmul_rn(s_uD, Z);
    int sp = -1, last_nz = 0;
    float acc = 0.f;
    for (int k = 0; k < a.splits; ++k) {
      const float pk = fb ? __ldcg(&a.ws.dpart[b * kMaxSplits + k].b)
                          : __ldcg(&a.ws.dpart[b * kMaxSplits + k].w);
      if (pk > 0.f) last_nz = k;
      if (sp < 0 && acc + pk > t) {
        sp = k;
        t -= acc;
      }
      acc += pk;
    }
    if (sp < 0) {  // rounding put t past the total: take the last token with mass
      sp = last_nz;
      t = INFINITY;
    }
    s_split = sp;
    s_t = t;
    s_fallback = fb;
    a.ws.reqcnt[b] = 0;
  }
  __syncthreads();
  const int fb = s_fallback;
  const int64_t slo = (int64_t)s_split * a.split_len;
  const int64_t shi = min(a.V, slo + a.split_len);
  float t = s_t;
  __shared__ float s_w[32];
  __shared__ int32_t s_tok, s_lastnz;
  if (threadIdx.x == 0) {
    s_tok = -1;
    s_lastnz = -1;
  }
  __syncthreads();
  // tiles of 4 consecutive tokens per thread, scanned in order
  for (int64_t t0 = slo; t0 < shi; t0 += 4 * kStreamThreads) {
    const int64_t i0 = t0 + 4 * (int64_t)threadIdx.x;
    float w[4];
    int32_t my_last = -1;
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t i = i0 + k;
      float wk = 0.f;
      if (i < shi) {
        const float p = pr[i];
        wk = fb ? p : weight(p, resid_q ? qr[i] : 0.f, i);
      }
      w[k] = wk;
      sum += wk;
      if (wk > 0.f) my_last = (int32_t)i;
    }
    float total;
    const float incl = block_incl_scan(sum, s_w, total);
    const float excl = incl - sum;
    if (excl <= t && t < incl) {  // exactly one thread: the prefix is nondecreasing
      float acc = excl;
      int32_t tok = my_last;
      for (int k = 0; k < 4; ++k) {
        if (w[k] > 0.f && acc + w[k] > t) {
          tok = (int32_t)(i0 + k);
          break;
        }
        acc += w[k];
      }
      s_tok = tok;
    }
    if (my_last >= 0) atomicMax(&s_lastnz, my_last);
    __syncthreads();
    if (s_tok >= 0) break;
    t -= total;
    __syncthreads();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t tok = s_tok >= 0 ? s_tok : s_lastnz;
    if (tok < 0) tok = (x >= 0) ? x : 0;  // no mass anywhere in the split (degenerate input)
    for (int32_t j = 0; j < R; ++j) {
      const int64_t rj = b * R + j;
      int32_t tj = -1;
      if (j < js) tj = a.drafts[b * a.D + j];
      else if (j == js) tj = tok;
      a.accepted_tokens[rj] = tj;
      if (a.accept_index) a.accept_index[rj] = (j <= js) ? (int32_t)rj : -1;
      if (a.logprobs) {
        float lp = 0.f;
        if (j <= js && tj >= 0 && (int64_t)tj < a.V) lp = logf(a.p[rj * a.ld + tj]);
        a.logprobs[rj] = lp;
      }
    }
    a.accept_length[b] = js + 1;
  }
}

cudaError_t launch_draw_probs(const DrawArgs& a, cudaStream_t s) {
  const dim3 grid((unsigned)(a.B * a.splits));
  k_draw_probs<<<grid, kStreamThreads, 0, s>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------
// ln p[r, tokens[r]] for probability rows.

__global__ void k_logprobs_probs(const float* p, int64_t ld, int64_t V, int64_t rows,
                                 const int32_t* tokens, float* out) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  const int32_t t = tokens[r];
  out[r] = (t >= 0 && (int64_t)t < V) ? logf(p[r * ld + t]) : 0.f;
}

cudaError_t launch_logprobs_probs(const float* p, int64_t ld, int64_t V, int64_t rows,
                                  const int32_t* tokens, float* out, cudaStream_t s) {
  const int th = 256;
  k_logprobs_probs<<<(unsigned)((rows + th - 1) / th), th, 0, s>>>(p, ld, V, rows, tokens, out);
  return cudaGetLastError();
}


// ---------------------------------------------------------------------------------
// Temperature softmax: probs[r, i] = exp((x_ri - M_r) / T_r) / sum_j exp((x_rj - M_r) / T_r),
// one-hot at the argmax for greedy rows. A cluster of kSoftCL CTAs takes a row; every CTA
// streams its slice once for the maximum, the argmax and the sum (online, per thread,
// Kahan-compensated), the CTAs exchange their partials through distributed shared memory,
// and every CTA streams its slice again to write its probabilities.

constexpr int kSoftCL = 4;

template <typename E>
__global__ void __launch_bounds__(kStreamThreads) k_softmax(const void* x, int64_t ld, int64_t V,
                                                            const float* temperature,
                                                            float* out, int64_t slice) {
  __shared__ float s_part[4];  // this CTA's (max, sum, argmax bits)
  __shared__ float s_v[32], s_m[32], s_s[32];
  __shared__ int32_t s_i[32];
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int64_t row = blockIdx.x / kSoftCL;
  constexpr int N = Vec<E>::N;
  const E* xr = reinterpret_cast<const E*>(x) + row * ld;
  const int64_t lo = (int64_t)crank * slice;
  const int64_t hi = min(V, lo + slice);
  const float T = temperature ? temperature[row] : 1.f;
  const bool greedy = !(T >= kGreedyT);
  const float sl2 = greedy ? 0.f : __fdiv_rn(kLog2e, T);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t nv = (hi > lo) ? (hi - lo) / N : 0;  // whole vectors of the slice
  const uint4* vp = reinterpret_cast<const uint4*>(xr + lo);

  // ---- 1. maximum, argmax, sum of exp((x - m) / T) with a running maximum m -------------
  float bv = -INFINITY, ls = 0.f, lc = 0.f;
  int32_t bi = INT32_MAX;
  auto visit = [&](const float* xv, int n, int64_t base) {
    float vm = xv[0];
    for (int q = 1; q < n; ++q) vm = fmaxf(vm, xv[q]);
    if (vm > bv || bi == INT32_MAX) {
      for (int q = 0; q < n; ++q)
        if (xv[q] == vm) {
          bi = (int32_t)(base + q);
          break;
        }
      if (!greedy && vm > bv && bv > -INFINITY) {
        const float f = ex2((bv - vm) * sl2);
        ls *= f;
        lc *= f;
      }
      bv = fmaxf(bv, vm);
    }
    if (!greedy && bv > -INFINITY) {
      float vs = 0.f;
      for (int q = 0; q < n; ++q) vs += ex2((xv[q] - bv) * sl2);
      kahan_add(ls, lc, vs);
    }
  };
  {
    int64_t vi = tid;
    constexpr int U = 4;
    for (; vi + (U - 1) * kStreamThreads < nv; vi += U * kStreamThreads) {
      uint4 r[U];
#pragma unroll
      for (int u = 0; u < U; ++u) r[u] = ldg_stream(vp + vi + u * kStreamThreads);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float xv[N];
        Vec<E>::unpack(r[u], xv);
        visit(xv, N, lo + (vi + u * kStreamThreads) * N);
      }
    }
    for (; vi < nv; vi += kStreamThreads) {
      float xv[N];
      Vec<E>::unpack(ldg_stream(vp + vi), xv);
      visit(xv, N, lo + vi * N);
    }
    const int64_t t0 = lo + nv * N;
    if (tid == 0 && t0 < hi) {  // the slice's ragged tail
      float xv[N];
      const int n = (int)(hi - t0);
      for (int q = 0; q < N; ++q) xv[q] = q < n ? Vec<E>::scalar(xr, t0 + q) : -INFINITY;
      visit(xv, N, t0);
    }
  }
  ls += lc;
  // merge (max, sum) pairs whose sums are relative to their own maxima
  auto merge = [&](float& m, float& sum, int32_t& i, float m2, float s2, int32_t i2) {
    const float nm = fmaxf(m, m2);
    if (!greedy && nm > -INFINITY)
      sum = ((m > -INFINITY) ? sum * ex2((m - nm) * sl2) : 0.f) +
            ((m2 > -INFINITY) ? s2 * ex2((m2 - nm) * sl2) : 0.f);
    if (m2 > m || (m2 == m && i2 < i)) i = i2;
    m = nm;
  };
  {
    float m = bv, sum = ls;
    int32_t i = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      merge(m, sum, i, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sum, o),
            __shfl_xor_sync(0xffffffffu, i, o));
    if (lane == 0) {
      s_m[w] = m;
      s_s[w] = sum;
      s_i[w] = i;
    }
    __syncthreads();
    if (w == 0) {
      const int nw = kStreamThreads / 32;
      m = lane < nw ? s_m[lane] : -INFINITY;
      sum = lane < nw ? s_s[lane] : 0.f;
      i = lane < nw ? s_i[lane] : INT32_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        merge(m, sum, i, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sum, o),
              __shfl_xor_sync(0xffffffffu, i, o));
      if (lane == 0) {
        s_part[0] = m;
        s_part[1] = sum;
        s_part[2] = __int_as_float(i);
      }
    }
  }
  cluster.sync();  // the CTAs' partials are visible
  if (tid == 0) {
    float m = -INFINITY, sum = 0.f;
    int32_t i = INT32_MAX;
    for (int c = 0; c < kSoftCL; ++c) {  // every CTA merges in the same order
      const float* pp = cluster.map_shared_rank(s_part, c);
      merge(m, sum, i, pp[0], pp[1], __float_as_int(pp[2]));
    }
    s_v[0] = m;
    s_v[1] = (sum > 0.f) ? __frcp_rn(sum) : 0.f;
    s_i[0] = i;
  }
  cluster.sync();  // no CTA leaves while a peer may still read its partial
  const float M = s_v[0], inv = s_v[1];
  const int32_t am = s_i[0];

  // ---- 2. the probabilities of the slice ----------------------------------------------
  float* orow = out + row * V;
  auto prob = [&](float v, int64_t gi) -> float {
    if (greedy) return (gi == (int64_t)am) ? 1.f : 0.f;
    return ex2((v - M) * sl2) * inv;
  };
  const bool vout = ((reinterpret_cast<uintptr_t>(orow + lo) & 15) == 0);
  for (int64_t vi = tid; vi < nv; vi += kStreamThreads) {
    float xv[N];
    Vec<E>::unpack(ldg_stream(vp + vi), xv);
    const int64_t base = lo + vi * N;
    float y[N];
#pragma unroll
    for (int q = 0; q < N; ++q) y[q] = prob(xv[q], base + q);
    if (vout) {
      float4* op = reinterpret_cast<float4*>(orow + base);
#pragma unroll
      for (int h = 0; h < N / 4; ++h) __stcs(op + h, make_float4(y[4 * h], y[4 * h + 1], y[4 * h + 2], y[4 * h + 3]));
    } else {
#pragma unroll
      for (int q = 0; q < N; ++q) orow[base + q] = y[q];
    }
  }
  for (int64_t i = lo + nv * N + tid; i < hi; i += kStreamThreads)
    orow[i] = prob(Vec<E>::scalar(xr, i), i);
}

// The same softmax with each CTA's slice staged once in shared memory: bulk copies bring
// the slice in (16 KB chunks, one mbarrier each, all in flight at once), both passes read
// it from there, so the logits are read from HBM once.
constexpr int kSmChunk = 16384;       // bytes a chunk
constexpr int kSmMaxChunks = 8;       // slices of at most 128 KB
constexpr long long kSmWaitCycles = 1ll << 32;
static __device__ unsigned int g_softmax_err;

template <typename E>
__global__ void __launch_bounds__(kStreamThreads) k_softmax_smem(const void* x, int64_t ld,
                                                                 int64_t V,
                                                                 const float* temperature,
                                                                 float* out, int64_t slice) {
  extern __shared__ __align__(128) unsigned char sbuf[];
  __shared__ uint64_t bars[kSmMaxChunks];
  __shared__ float s_part[4];
  __shared__ float s_v[32], s_m[32], s_s[32];
  __shared__ int32_t s_i[32];
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int CL = (int)cluster.num_blocks();
  const int64_t row = blockIdx.x / CL;
  constexpr int N = Vec<E>::N;
  const E* xr = reinterpret_cast<const E*>(x) + row * ld;
  const int64_t lo = (int64_t)crank * slice;
  const int64_t hi = min(V, lo + slice);
  const float T = temperature ? temperature[row] : 1.f;
  const bool greedy = !(T >= kGreedyT);
  const float sl2 = greedy ? 0.f : __fdiv_rn(kLog2e, T);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t nv = (hi > lo) ? (hi - lo) / N : 0;  // whole vectors of the slice
  const uint32_t bytes = (uint32_t)(nv * 16);      // staged bytes (whole vectors)
  const int nch = (int)((bytes + kSmChunk - 1) / kSmChunk);
  const uint4* sv = reinterpret_cast<const uint4*>(sbuf);

  if (tid == 0) {
    for (int c = 0; c < nch; ++c) mbar_init(&bars[c], 1);
    fence_mbar_init();
    const unsigned char* src = reinterpret_cast<const unsigned char*>(xr + lo);
    for (int c = 0; c < nch; ++c) {
      const uint32_t nb = min((uint32_t)kSmChunk, bytes - (uint32_t)c * kSmChunk);
      mbar_arrive_expect_tx(&bars[c], nb);
      bulk_g2s(sbuf + (size_t)c * kSmChunk, src + (size_t)c * kSmChunk, nb, &bars[c]);
    }
  }
  __syncthreads();

  // ---- 1. maximum, argmax, sum of exp((x - m) / T) with a running maximum m -------------
  float bv = -INFINITY, ls = 0.f, lc = 0.f;
  int32_t bi = INT32_MAX;
  auto visit = [&](const float* xv, int n, int64_t base) {
    float vm = xv[0];
    for (int q = 1; q < n; ++q) vm = fmaxf(vm, xv[q]);
    if (vm > bv || bi == INT32_MAX) {
      for (int q = 0; q < n; ++q)
        if (xv[q] == vm) {
          bi = (int32_t)(base + q);
          break;
        }
      if (!greedy && vm > bv && bv > -INFINITY) {
        const float f = ex2((bv - vm) * sl2);
        ls *= f;
        lc *= f;
      }
      bv = fmaxf(bv, vm);
    }
    if (!greedy && bv > -INFINITY) {
      float vs = 0.f;
      for (int q = 0; q < n; ++q) vs += ex2((xv[q] - bv) * sl2);
      kahan_add(ls, lc, vs);
    }
  };
  constexpr int VPC = kSmChunk / 16;  // vectors a chunk
  for (int c = 0; c < nch; ++c) {
    // wait for chunk c: only the time limit ends the wait, so that the CTA never leaves
    // with a copy in flight while the copies are still landing
    const long long t0 = clock64();
    while (!mbar_try_wait(&bars[c], 0u)) {
      if (clock64() - t0 > kSmWaitCycles) {
        atomicOr(&g_softmax_err, 1u);
        break;
      }
    }
    const int64_t v1 = min(nv, (int64_t)(c + 1) * VPC);
    for (int64_t vi = (int64_t)c * VPC + tid; vi < v1; vi += kStreamThreads) {
      float xv[N];
      Vec<E>::unpack(sv[vi], xv);
      visit(xv, N, lo + vi * N);
    }
  }
  const int64_t t0 = lo + nv * N;
  if (tid == 0 && t0 < hi) {  // the slice's ragged tail, from global memory
    float xv[N];
    const int n = (int)(hi - t0);
    for (int q = 0; q < N; ++q) xv[q] = q < n ? Vec<E>::scalar(xr, t0 + q) : -INFINITY;
    visit(xv, N, t0);
  }
  ls += lc;
  auto merge = [&](float& m, float& sum, int32_t& i, float m2, float s2, int32_t i2) {
    const float nm = fmaxf(m, m2);
    if (!greedy && nm > -INFINITY)
      sum = ((m > -INFINITY) ? sum * ex2((m - nm) * sl2) : 0.f) +
            ((m2 > -INFINITY) ? s2 * ex2((m2 - nm) * sl2) : 0.f);
    if (m2 > m || (m2 == m && i2 < i)) i = i2;
    m = nm;
  };
  {
    float m = bv, sum = ls;
    int32_t i = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      merge(m, sum, i, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sum, o),
            __shfl_xor_sync(0xffffffffu, i, o));
    if (lane == 0) {
      s_m[w] = m;
      s_s[w] = sum;
      s_i[w] = i;
    }
    __syncthreads();
    if (w == 0) {
      const int nw = kStreamThreads / 32;
      m = lane < nw ? s_m[lane] : -INFINITY;
      sum = lane < nw ? s_s[lane] : 0.f;
      i = lane < nw ? s_i[lane] : INT32_MAX;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        merge(m, sum, i, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sum, o),
              __shfl_xor_sync(0xffffffffu, i, o));
      if (lane == 0) {
        s_part[0] = m;
        s_part[1] = sum;
        s_part[2] = __int_as_float(i);
      }
    }
  }
  cluster.sync();  // the CTAs' partials are visible
  if (tid == 0) {
    float m = -INFINITY, sum = 0.f;
    int32_t i = INT32_MAX;
    for (int c = 0; c < CL; ++c) {  // every CTA merges in the same order
      const float* pp = cluster.map_shared_rank(s_part, c);
      merge(m, sum, i, pp[0], pp[1], __float_as_int(pp[2]));
    }
    s_v[0] = m;
    s_v[1] = (sum > 0.f) ? __frcp_rn(sum) : 0.f;
    s_i[0] = i;
  }
  cluster.sync();  // no CTA leaves while a peer may still read its partial
  const float M = s_v[0], inv = s_v[1];
  const int32_t am = s_i[0];

  // ---- 2. the probabilities of the slice, from the staged copy ------------------------
  float* orow = out + row * V;
  auto prob = [&](float v, int64_t gi) -> float {
    if (greedy) return (gi == (int64_t)am) ? 1.f : 0.f;
    return ex2((v - M) * sl2) * inv;
  };
  const bool vout = ((reinterpret_cast<uintptr_t>(orow + lo) & 15) == 0);
  for (int64_t vi = tid; vi < nv; vi += kStreamThreads) {
    float xv[N];
    Vec<E>::unpack(sv[vi], xv);
    const int64_t base = lo + vi * N;
    float y[N];
#pragma unroll
    for (int q = 0; q < N; ++q) y[q] = prob(xv[q], base + q);
    if (vout) {
      float4* op = reinterpret_cast<float4*>(orow + base);
#pragma unroll
      for (int h = 0; h < N / 4; ++h) __stcs(op + h, make_float4(y[4 * h], y[4 * h + 1], y[4 * h + 2], y[4 * h + 3]));
    } else {
#pragma unroll
      for (int q = 0; q < N; ++q) orow[base + q] = y[q];
    }
  }
  for (int64_t i = lo + nv * N + tid; i < hi; i += kStreamThreads)
    orow[i] = prob(Vec<E>::scalar(xr, i), i);
}

cudaError_t softmax_read_error(uint32_t* word, int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_softmax_err, sizeof(v));
  if (e != cudaSuccess) return e;
  if (clear && v) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_softmax_err, &z, sizeof(z));
  }
  *word = v;
  return e;
}

cudaError_t launch_softmax(const void* x, int bf16, int64_t rows, int64_t ld, int64_t V,
                           const float* temperature, float* out, cudaStream_t s) {
  // staged: the smallest cluster (1, 2, 4 or 8 CTAs) whose slices fit 128 KB of shared
  // memory, slices of whole 16-byte vectors (a multiple of 8 elements). (Smaller slices,
  // 3 or 4 CTAs an SM, measured slower on the 201088-token bf16 rows.)
  const int64_t esize = bf16 ? 2 : 4;
  for (int cl = 1; cl <= 8; cl *= 2) {
    const int64_t slice = (((V + cl - 1) / cl) + 7) & ~(int64_t)7;
    if (slice * esize > (int64_t)kSmChunk * kSmMaxChunks) continue;
    const size_t dyn = (size_t)((slice * esize + 15) & ~(int64_t)15);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(rows * cl));
    cfg.blockDim = dim3(kStreamThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (bf16) {
      e = cudaFuncSetAttribute(k_softmax_smem<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
      if (e != cudaSuccess) return e;
      return cudaLaunchKernelEx(&cfg, k_softmax_smem<uint16_t>, x, ld, V, temperature, out, slice);
    }
    e = cudaFuncSetAttribute(k_softmax_smem<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, k_softmax_smem<float>, x, ld, V, temperature, out, slice);
  }
  // larger rows: the streaming kernel (each slice read twice)
  // slices of whole 16-byte vectors: a multiple of 8 elements
  const int64_t slice = (((V + kSoftCL - 1) / kSoftCL) + 7) & ~(int64_t)7;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(rows * kSoftCL));
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)kSoftCL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (bf16) return cudaLaunchKernelEx(&cfg, k_softmax<uint16_t>, x, ld, V, temperature, out, slice);
  return cudaLaunchKernelEx(&cfg, k_softmax<float>, x, ld, V, temperature, out, slice);
}

}  // namespace tsv
