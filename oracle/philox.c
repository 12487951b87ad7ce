/*
 * Oracle: Philox4x32-10 and the uniform streams drawn from it.
 * TEST INFRASTRUCTURE ONLY (see orc.h).
 *
 * Block function: Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3"
 * (SC'11), section 3 (Philox): a 4x32-bit counter, a 2x32-bit key, ten rounds.
 * One round multiplies counter words 0 and 2 by two fixed odd constants,
 * keeps both halves of each 64-bit product, and permutes/xors them with the
 * other two counter words and the key; between rounds the key is bumped by
 * two Weyl constants (golden ratio and sqrt(3)-1, as 32-bit fractions).
 *
 * Stream layout (the pages name "Philox keyed by seed with an offset" but do
 * not give a layout; this is the reading chosen and documented):
 *   key                   = (low 32 bits of seed, high 32 bits of seed)
 *   verify coin j         : counter (j, 0xFFFFFFFF, lo(offset), hi(offset)), word 0
 *   Gumbel element v, row n: counter (v >> 2, n, lo(offset), hi(offset)), word v & 3
 * Row indices n are below 0xFFFFFFFF, so the two streams never share a counter.
 */
#include "orc.h"

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c[0];
    uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c[1] ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c[3] ^ k1;
    uint32_t n3 = lo0;
    c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
  }
  out[0] = c[0]; out[1] = c[1]; out[2] = c[2]; out[3] = c[3];
}

/* A 32-bit word to a uniform in the open interval (0, 1): keep the top 23
 * bits m and return (2m + 1) / 2^24. Every value is exact in fp32 and lies in
 * [2^-24, 1 - 2^-24], so neither 0 nor 1 is ever drawn. */
float orc_u01(uint32_t x) {
  uint32_t m = x >> 9;
  double u = (2.0 * (double)m + 1.0) / 16777216.0;
  return (float)u; /* exact: 24 significant bits at most */
}

static void key_of(uint64_t seed, uint32_t key[2]) {
  key[0] = (uint32_t)(seed & 0xFFFFFFFFu);
  key[1] = (uint32_t)(seed >> 32);
}

float orc_verify_coin(uint64_t seed, uint64_t offset, uint32_t j) {
  uint32_t key[2], ctr[4], out[4];
  key_of(seed, key);
  ctr[0] = j;
  ctr[1] = 0xFFFFFFFFu;
  ctr[2] = (uint32_t)(offset & 0xFFFFFFFFu);
  ctr[3] = (uint32_t)(offset >> 32);
  orc_philox4x32_10(ctr, key, out);
  return orc_u01(out[0]);
}

float orc_gumbel_u01(uint64_t seed, uint64_t offset, uint32_t n, uint32_t v) {
  uint32_t key[2], ctr[4], out[4];
  key_of(seed, key);
  ctr[0] = v >> 2;
  ctr[1] = n;
  ctr[2] = (uint32_t)(offset & 0xFFFFFFFFu);
  ctr[3] = (uint32_t)(offset >> 32);
  orc_philox4x32_10(ctr, key, out);
  return orc_u01(out[v & 3u]);
}
