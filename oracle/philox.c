/*
 * philox.c -- oracle: Philox4x32-10 counter-based generator.  Test
 * infrastructure only (see fp4_oracle.h).
 *
 * Written from Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3" (SC'11), section 4 (Philox): each round multiplies counter
 * words 0 and 2 by the two round multipliers, keeps the 32-bit high and low
 * halves, XORs the high halves with the other two counter words and the key,
 * and permutes; the key is bumped by the two Weyl constants between rounds.
 */
#include "fp4_oracle.h"

static const uint32_t kMul0 = 0xD2511F53u;
static const uint32_t kMul1 = 0xCD9E8D57u;
static const uint32_t kWeyl0 = 0x9E3779B9u;  /* golden ratio */
static const uint32_t kWeyl1 = 0xBB67AE85u;  /* sqrt(3) - 1 */

void ora_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)kMul0 * c0;
    uint64_t p1 = (uint64_t)kMul1 * c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += kWeyl0;
    k1 += kWeyl1;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

uint32_t ora_rng_word(uint64_t seed, uint64_t step, uint64_t g) {
  /* eight elements per Philox call: element g takes the 16-bit half g & 1 of
   * word (g >> 1) & 3 of the block at counter g >> 3 */
  uint64_t oct = g >> 3;
  uint32_t ctr[4] = {(uint32_t)oct, (uint32_t)(oct >> 32), (uint32_t)step,
                     (uint32_t)(step >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  ora_philox4x32_10(ctr, key, out);
  uint32_t h = (out[(g >> 1) & 3] >> (16 * (g & 1))) & 0xFFFFu;
  return h << 16;
}
