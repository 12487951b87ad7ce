// Gumbel-max sampling from logits (TensorRT-LLM interface.py,
// _sample_sharded_temperature): the token of a row is argmax_i (l_i / T + G_i) with
// G_i = -ln(-ln u_i), u_i drawn from the request's Philox stream, or the plain argmax
// (lowest id on ties) when T is below the greedy threshold.
//
// k_gumbel is a persistent kernel whose warps work independently: each claims chunks
// (a contiguous run of 16-byte vectors of one row) one at a time from a counter in row
// order, so the cost of a row, which depends on its temperature, does not set the length
// of a wave, and no warp waits for another. A warp streams a chunk in rounds of 4 vectors
// a lane with the next round's loads in flight (across chunk ends too: the next claim is
// made a chunk ahead), and keeps a bound: the best score it knows of, its own or one
// published to the row by another warp (an atomic max of the score's order key). Each
// chunk's best goes to the workspace; the warp that finishes a row's last chunk merges
// them and writes the token.
//
// The exact score of an element costs a Philox block (shared by a group of 4 elements)
// and two logarithms. It is skipped when an upper bound shows the element cannot beat a
// score already computed:
//   - a group whose max(l) / T + 17 is below the bound is not drawn at all (17 exceeds
//     the largest noise an element can get, -ln(-ln(1 - 2^-24)) = 16.64);
//   - a drawn group whose max(l) / T - ln(1 - u_max) is below it is dropped
//     (-ln(-ln u) <= -ln(1 - u) for u in (0, 1), and G is increasing in u);
//   - so is an element whose l / T - ln(1 - u) is below it.
// The last two use the fast logarithm with a margin of 1e-3, far above its error, so a
// skipped element's computed score is always below a computed score. The groups a warp
// must draw are first compacted into a queue in shared memory and then drawn two a lane,
// so that the cost follows the number of such groups, not the number of rounds in which
// any lane has one. When a warp starts a round with no bound at all, one lane first scores
// the group holding the round's largest logit and that score serves as the bound. The
// skips change which scores are computed, never a computed score, and equal scores go to
// the lower id, so the token is the argmax of the scores a full pass computes.
#include <stdint.h>

#include "ts_common.cuh"
#include "ts_internal.h"
#include "ts_rowutil.cuh"

namespace tsv {
namespace {

constexpr int kGThreads = 256;
constexpr int kGWarps = kGThreads / 32;
constexpr int kGU = 4;            // vectors a lane loads per round
constexpr float kGCap = 17.0f;    // above every noise value the kernel computes
constexpr float kGSlack = 1e-3f;  // margin of the fast-log upper bounds

// A row's Philox stream (key and counter words) and 1 / T.
struct GumbelRow {
  uint32_t k0, k1, c1, c2, c3;
  float invT;
};

// The 4 logits of a group, kept as raw words in the queue.
template <typename E>
struct GroupBits;
template <>
struct GroupBits<uint16_t> {
  using T = uint2;
  __device__ __forceinline__ static T take(const uint4& r, int q) {
    return q == 0 ? make_uint2(r.x, r.y) : make_uint2(r.z, r.w);
  }
  __device__ __forceinline__ static void unpack(const T& b, float* x) {
    x[0] = __uint_as_float(b.x << 16);
    x[1] = __uint_as_float(b.x & 0xFFFF0000u);
    x[2] = __uint_as_float(b.y << 16);
    x[3] = __uint_as_float(b.y & 0xFFFF0000u);
  }
  __device__ __forceinline__ static float gmax(const uint4& r, int q) {
    const uint32_t m = q == 0 ? SVec<uint16_t>::bmax2(r.x, r.y) : SVec<uint16_t>::bmax2(r.z, r.w);
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
};
template <>
struct GroupBits<float> {
  using T = uint4;
  __device__ __forceinline__ static T take(const uint4& r, int) { return r; }
  __device__ __forceinline__ static void unpack(const T& b, float* x) { SVec<float>::unpack(b, x); }
  __device__ __forceinline__ static float gmax(const uint4& r, int) { return SVec<float>::vmax(r); }
};

// Score the elements of a drawn group (logits x, ids 4 * gi ..; w its Philox block) that
// can beat `bound`; the best (bv, bi) takes the higher score, the lower id on equal ones.
__device__ __forceinline__ void gumbel_scores(const GumbelRow& g, const uint4& w, const float* x,
                                              uint32_t gi, float& bound, float& bv, int32_t& bi) {
  const float gm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  const uint32_t um = max(max(w.x, w.y), max(w.z, w.w));
  if (gm * g.invT - __logf(1.f - u01(um)) + kGSlack < bound) return;
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (x[k] == -INFINITY) continue;
    const float u = u01(wv[k]);
    const float xs = x[k] * g.invT;
    if (xs - __logf(1.f - u) + kGSlack < bound) continue;
    const float e = -logf(u);
    const float s = xs - __logf(e);
    const int32_t id = (int32_t)(4 * gi + k);
    if (s > bv || (s == bv && id < bi)) {
      bv = s;
      bi = id;
      bound = fmaxf(bound, s);
    }
  }
}

__device__ __forceinline__ uint4 group_ctr(const GumbelRow& g, uint32_t gi) {
  return make_uint4(gi, g.c1, g.c2, g.c3);
}

template <typename E>
__global__ void __launch_bounds__(kGThreads, 3) k_gumbel(GumbelArgs a) {
  using SV = SVec<E>;
  using GB = GroupBits<E>;
  using QB = typename GB::T;
  constexpr int N = SV::N;          // elements per vector
  constexpr int G = N / 4;          // groups per vector
  constexpr int kQ = 32 * kGU * G;  // queue entries a warp (a round at most)
  constexpr int64_t kRound = 32 * kGU;  // vectors a warp round
  __shared__ QB s_qx[kGWarps][kQ];
  __shared__ uint32_t s_qg[kGWarps][kQ];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt = (1u << lane) - 1u;
  const int64_t nv = a.V / N;  // whole vectors of a row
  const uint4 neg = make_uint4(SV::kNegInfWord, SV::kNegInfWord, SV::kNegInfWord,
                               SV::kNegInfWord);
  QB* qx = s_qx[warp];
  uint32_t* qg = s_qg[warp];

  auto claim = [&]() {
    uint32_t c = 0;
    if (lane == 0) c = atomicAdd(&a.ws.work[0], 1u);
    return __shfl_sync(0xffffffffu, c, 0);
  };
  struct Chunk {  // row, chunk of the row, and its vectors [v0, v1) (32 bits: < 2^31 each)
    int32_t row, chunk, v0, v1;
  };
  auto geom = [&](uint32_t c) {
    Chunk k;
    k.row = (int32_t)(c / (uint32_t)a.cpr);
    k.chunk = (int32_t)(c % (uint32_t)a.cpr);
    k.v0 = k.chunk * (int32_t)a.chunk_vecs;
    k.v1 = (int32_t)min(nv, (int64_t)k.v0 + a.chunk_vecs);
    return k;
  };
  auto nrounds = [&](const Chunk& k) { return (int)((max(k.v1 - k.v0, 0) + kRound - 1) / kRound); };
  uint4 rn[kGU];  // the loads of the next round
  auto load = [&](const Chunk& k, int rd) {
    const uint4* vp =
        reinterpret_cast<const uint4*>(reinterpret_cast<const E*>(a.x) + (int64_t)k.row * a.ld);
    const int32_t vb = k.v0 + rd * (int32_t)kRound + lane;
#pragma unroll
    for (int u = 0; u < kGU; ++u) rn[u] = (vb + u * 32 < k.v1) ? ldg_stream(vp + vb + u * 32) : neg;
  };

  uint32_t cur = claim();
  if (cur >= a.total_chunks) return;
  uint32_t nxt = claim();
  Chunk ck = geom(cur);
  load(ck, 0);
  for (;;) {
    const bool has_next = nxt < a.total_chunks;
    const Chunk cn = geom(has_next ? nxt : cur);
    const int rounds = nrounds(ck);
    auto advance = [&](int rd) {  // issue the loads that follow round rd
      if (rd + 1 < rounds) load(ck, rd + 1);
      else if (has_next) load(cn, 0);
    };
    const int64_t row = ck.row;
    const E* xr = reinterpret_cast<const E*>(a.x) + row * a.ld;
    const bool last_chunk = ck.chunk == a.cpr - 1;
    const float T = a.temperature[row];
    float bv = -INFINITY;
    int32_t bi = INT32_MAX;
    if (rounds == 0) advance(-1);

    if (T < kGreedyT) {
      for (int rd = 0; rd < rounds; ++rd) {
        uint4 r[kGU];
#pragma unroll
        for (int u = 0; u < kGU; ++u) r[u] = rn[u];
        advance(rd);
        const int64_t vb = (int64_t)ck.v0 + rd * kRound + lane;
#pragma unroll
        for (int u = 0; u < kGU; ++u) {
          const float vm = SV::vmax(r[u]);
          if (vm > bv) {
            float x[N];
            SV::unpack(r[u], x);
            int k = N - 1;
#pragma unroll
            for (int j = N - 2; j >= 0; --j)
              if (x[j] == vm) k = j;
            bv = vm;
            bi = (int32_t)((vb + u * 32) * N + k);
          }
        }
      }
      if (last_chunk && lane == 0) {
        for (int64_t i = nv * N; i < a.V; ++i) {
          const float v = SV::at(xr, i);
          if (v > bv) {
            bv = v;
            bi = (int32_t)i;
          }
        }
      }
    } else {
      GumbelRow g;
      const int64_t b = row / a.n_per_req;
      const uint64_t seed = (uint64_t)a.seed[b], off = (uint64_t)a.offset[b];
      g.k0 = (uint32_t)seed;
      g.k1 = (uint32_t)(seed >> 32);
      g.c1 = (uint32_t)(row % a.n_per_req);
      g.c2 = (uint32_t)off;
      g.c3 = (uint32_t)(off >> 32);
      g.invT = __frcp_rn(T);
      uint32_t* best = &a.ws.best[row];
      // wb: the warp's bound, the same in every lane and >= every lane's bv at a round's start
      float wb;
      {
        uint32_t k0 = 0;
        if (lane == 0) k0 = __ldcg(best);
        k0 = __shfl_sync(0xffffffffu, k0, 0);
        wb = k0 ? key_to_value(k0) : -INFINITY;
      }
      uint32_t fut = 0;  // lane 0: the row's best key returned by the last publish
      for (int rd = 0; rd < rounds; ++rd) {
        uint4 r[kGU];
#pragma unroll
        for (int u = 0; u < kGU; ++u) r[u] = rn[u];
        advance(rd);
        if (rd > 0) {  // the previous round's publish, awaited behind the loads
          const uint32_t k0 = __shfl_sync(0xffffffffu, fut, 0);
          if (k0) wb = fmaxf(wb, key_to_value(k0));
        }
        const int64_t vb = (int64_t)ck.v0 + rd * kRound + lane;
        float gm[kGU * G];
        float lmx = -INFINITY;
#pragma unroll
        for (int u = 0; u < kGU; ++u)
#pragma unroll
          for (int q = 0; q < G; ++q) {
            gm[u * G + q] = GB::gmax(r[u], q);
            lmx = fmaxf(lmx, gm[u * G + q]);
          }
        const float wmx = warp_max(lmx);
        if (wmx == -INFINITY || wmx * g.invT + kGCap < wb) continue;  // warp-uniform
        if (wb == -INFINITY) {
          // no bound yet: score the group holding the warp's largest logit first
          const int pl = __ffs(__ballot_sync(0xffffffffu, lmx == wmx)) - 1;
          float ps = -INFINITY;
          if (lane == pl) {
            QB pb{};
            uint32_t pgi = 0;
            bool found = false;
#pragma unroll
            for (int u = 0; u < kGU; ++u)
#pragma unroll
              for (int q = 0; q < G; ++q)
                if (!found && gm[u * G + q] == wmx) {
                  found = true;
                  pb = GB::take(r[u], q);
                  pgi = (uint32_t)((vb + u * 32) * G + q);
                }
            float px[4];
            GB::unpack(pb, px);
            float pbound = -INFINITY;
            int32_t pi = INT32_MAX;
            gumbel_scores(g, philox4x32_10(group_ctr(g, pgi), g.k0, g.k1), px, pgi, pbound, ps,
                          pi);
          }
          wb = __shfl_sync(0xffffffffu, ps, pl);
        }
        // compact the groups this warp must draw
        int n = 0;
#pragma unroll
        for (int u = 0; u < kGU; ++u)
#pragma unroll
          for (int q = 0; q < G; ++q) {
            const float m = gm[u * G + q];
            const bool f = m != -INFINITY && m * g.invT + kGCap >= wb;
            const uint32_t bal = __ballot_sync(0xffffffffu, f);
            if (f) {
              const int pos = n + __popc(bal & lt);
              qx[pos] = GB::take(r[u], q);
              qg[pos] = (uint32_t)((vb + u * 32) * G + q);
            }
            n += __popc(bal);
          }
        __syncwarp();
        // draw them, two a lane at a time
        float bound = fmaxf(bv, wb);
        for (int i0 = 0; i0 < n; i0 += 64) {
          const int ia = i0 + lane, ib = ia + 32;
          const bool va = ia < n, vbb = ib < n;
          const uint32_t ga = va ? qg[ia] : 0u, gb = vbb ? qg[ib] : 0u;
          const QB xa = va ? qx[ia] : QB{}, xb = vbb ? qx[ib] : QB{};
          uint4 wa = group_ctr(g, ga), wb2 = group_ctr(g, gb);
          philox4x32_10_x2(wa, wb2, g.k0, g.k1);
          float x[4];
          if (va) {
            GB::unpack(xa, x);
            gumbel_scores(g, wa, x, ga, bound, bv, bi);
          }
          if (vbb) {
            GB::unpack(xb, x);
            gumbel_scores(g, wb2, x, gb, bound, bv, bi);
          }
        }
        __syncwarp();
        // publish the warp's best to the row; the reply is read next round
        const float m = warp_max(bv);
        if (m > wb) {
          wb = m;
          if (lane == 0) fut = atomicMax(best, fkey(m));
        } else if (lane == 0) {
          fut = __ldcg(best);
        }
      }
      // the ragged tail (fewer than N elements), padded with -inf to whole groups
      if (last_chunk && lane == 0 && nv * N < a.V) {
        const int64_t t0 = nv * N;
        const int n = (int)(a.V - t0);
        float x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = k < n ? SV::at(xr, t0 + k) : -INFINITY;
        float bound = fmaxf(bv, wb);
        for (int q = 0; q < (n + 3) / 4; ++q) {
          const uint32_t gi = (uint32_t)((t0 >> 2) + q);
          gumbel_scores(g, philox4x32_10(group_ctr(g, gi), g.k0, g.k1), x + 4 * q, gi, bound, bv,
                        bi);
        }
      }
    }

    // the chunk's best (lowest id on equal scores), then the row's if this was its last
    warp_argmax(bv, bi);
    uint32_t prev = 0;
    if (lane == 0) {
      a.ws.part[row * kMaxSplits + ck.chunk] = Part{bv, bi, 0.f, 0.f};
      __threadfence();
      prev = atomicAdd(&a.ws.rowcnt[row], 1u);
    }
    if (__shfl_sync(0xffffffffu, prev, 0) == (uint32_t)a.cpr - 1) {
      __threadfence();
      float v = -INFINITY;
      int32_t i = INT32_MAX;
      for (int k = lane; k < a.cpr; k += 32) {
        const Part* pp = &a.ws.part[row * kMaxSplits + k];
        argmax_merge(v, i, __ldcg(&pp->v), __ldcg(&pp->i));
      }
      warp_argmax(v, i);
      if (lane == 0) {
        a.tokens_out[row] = (i == INT32_MAX) ? 0 : i;
        a.ws.rowcnt[row] = 0;
        a.ws.best[row] = 0;
      }
    }
    if (!has_next) break;
    ck = cn;
    nxt = claim();
  }
}

}  // namespace

cudaError_t launch_gumbel(const GumbelArgs& a, int bf16, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(a.ws.work, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  if (bf16) k_gumbel<uint16_t><<<a.grid, kGThreads, 0, s>>>(a);
  else k_gumbel<float><<<a.grid, kGThreads, 0, s>>>(a);
  return cudaGetLastError();
}

int gumbel_ctas_per_sm(int bf16) {
  int n = 0;
  if (bf16) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gumbel<uint16_t>, kGThreads, 0);
  else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_gumbel<float>, kGThreads, 0);
  return n < 1 ? 1 : n;
}

}  // namespace tsv
