// Device helpers shared by the verify-and-sample kernels (sm_103a).
//
// Nothing here is shared with the CPU oracle: the Philox block function, the uniform
// mapping and the ordering keys are written again from their definitions.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <cooperative_groups.h>

namespace tsv {

namespace cg = cooperative_groups;

constexpr float kGreedyT = 1e-5f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Fixed-point scale of a softmax weight e in (0, 1]: w = floor(e * 2^40).
constexpr float kFx = 1099511627776.0f;
constexpr uint32_t kIdxBits = 24;  // composite keys hold (2^24 - 1 - token id)
constexpr uint32_t kIdxMax = (1u << kIdxBits) - 1u;

// ---------------------------------------------------------------------------------
// Values and ordering keys

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// Monotone map float -> uint32: a > b (as floats) iff key(a) > key(b); -0 and +0 share
// the key of +0, so equal floats have equal keys. NaN is outside the contract.
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t b = __float_as_uint(x);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The float of an order key from fkey (the key of -0 gives +0).
__device__ __forceinline__ float key_to_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Composite order key: value descending, then token id ascending, is composite
// descending. Token ids must be below 2^24.
__device__ __forceinline__ uint64_t comp_key(uint32_t key, uint32_t idx) {
  return ((uint64_t)key << kIdxBits) | (uint64_t)(kIdxMax - idx);
}

// Fast 2^x (MUFU), denormal results flushed to zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// floor(e * 2^40) for e in [0, 1]; exact (power-of-two scale, truncating conversion).
__device__ __forceinline__ uint64_t fixw(float e) { return __float2ull_rz(e * kFx); }

// ---------------------------------------------------------------------------------
// Philox4x32-10 (Salmon et al., SC'11): ten rounds of the two-multiplier round
// function with a Weyl-bumped 2x32 key.

// The ten round keys of one stream: the key bumped by the two Weyl constants each round.
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};

__device__ __forceinline__ PhiloxKeys philox_keys(uint32_t k0, uint32_t k1) {
  PhiloxKeys k;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = k0;
    k.k1[r] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return k;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const PhiloxKeys& k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
    const uint32_t h0 = __umulhi(m0, c.x), l0 = m0 * c.x;
    const uint32_t h1 = __umulhi(m1, c.z), l1 = m1 * c.z;
    c = make_uint4(h1 ^ c.y ^ k.k0[r], l1, h0 ^ c.w ^ k.k1[r], l0);
  }
  return c;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
  return philox4x32_10(c, philox_keys(k0, k1));
}

// Two blocks of one stream computed side by side (the same rounds as above, written so
// that the two dependency chains interleave).
__device__ __forceinline__ void philox4x32_10_x2(uint4& a, uint4& b, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
    const uint64_t pa0 = (uint64_t)m0 * a.x, pa1 = (uint64_t)m1 * a.z;
    const uint64_t pb0 = (uint64_t)m0 * b.x, pb1 = (uint64_t)m1 * b.z;
    a = make_uint4((uint32_t)(pa1 >> 32) ^ a.y ^ k0, (uint32_t)pa1,
                   (uint32_t)(pa0 >> 32) ^ a.w ^ k1, (uint32_t)pa0);
    b = make_uint4((uint32_t)(pb1 >> 32) ^ b.y ^ k0, (uint32_t)pb1,
                   (uint32_t)(pb0 >> 32) ^ b.w ^ k1, (uint32_t)pb0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

// A 32-bit word to (2*(w >> 9) + 1) * 2^-24: exact in fp32, inside (0, 1).
__device__ __forceinline__ float u01(uint32_t w) {
  return __uint2float_rn(((w >> 9) << 1) | 1u) * 5.9604644775390625e-8f;
}

// Verify coin j of a request: counter (j, 0xFFFFFFFF, lo(offset), hi(offset)), word 0.
__device__ __forceinline__ float verify_coin(uint64_t seed, uint64_t offset, uint32_t j) {
  uint4 r = philox4x32_10(make_uint4(j, 0xFFFFFFFFu, (uint32_t)offset, (uint32_t)(offset >> 32)),
                          (uint32_t)seed, (uint32_t)(seed >> 32));
  return u01(r.x);
}

// ---------------------------------------------------------------------------------
// Warp helpers

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (value, index) argmax with the lowest index among equal values.
__device__ __forceinline__ void argmax_merge(float& v, int32_t& i, float v2, int32_t i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void warp_argmax(float& v, int32_t& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    int32_t i2 = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_merge(v, i, v2, i2);
  }
}

// Online log-sum-exp state: the sum is s * exp(m), m in the units of the input. The
// exponent is formed as (x - m) * log2(e) so that the terms that dominate the sum,
// those with x near m, see a small, accurately rounded argument.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  float nm = fmaxf(m, m2);
  if (nm == -INFINITY) return;
  s = s * ex2((m - nm) * kLog2e) + s2 * ex2((m2 - nm) * kLog2e);
  m = nm;
}

__device__ __forceinline__ void warp_lse(float& m, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
}

// Kahan-compensated accumulation.
__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  float y = x - c;
  float t = s + y;
  c = (t - s) - y;
  s = t;
}

// ---------------------------------------------------------------------------------
// Global loads that bypass L1 (each byte is read once per pass).

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---------------------------------------------------------------------------------
// mbarrier + bulk copy (TMA, 1-D) into shared memory

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Copies `bytes` (a multiple of 16; both addresses 16-byte aligned) from global to this
// CTA's shared memory; completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, "
      "1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// One arrival on a barrier (no transaction bytes).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

}  // namespace tsv
