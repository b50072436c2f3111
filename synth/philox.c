/*
 * Seeded synthetic inputs: the Philox4x32-10 counter-based generator
 * (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
 * SC'11), written from the paper's definition, plus the plain derived draws
 * the workloads use (uniforms, Box-Muller normals, bounded integers) and
 * round-to-nearest-even conversion to bfloat16.
 *
 * This file holds no arithmetic of the speculative-decoding method. Both the
 * oracle and the CUDA path receive the arrays it fills.
 *
 * Stream layout: key = (seed_lo, seed_hi); counter = (block_lo, block_hi,
 * stream, 0) where `stream` names the tensor being drawn and `block` is the
 * index of the 4-word output block. Word j of block b is element 4*b + j.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static inline void mulhilo(uint32_t a, uint32_t b, uint32_t* hi, uint32_t* lo) {
  uint64_t p = (uint64_t)a * (uint64_t)b;
  *hi = (uint32_t)(p >> 32);
  *lo = (uint32_t)p;
}

/* Ten rounds; the key is bumped by the Weyl constants between rounds. */
void synth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += PHILOX_W0; k1 += PHILOX_W1; }
    uint32_t hi0, lo0, hi1, lo1;
    mulhilo(PHILOX_M0, c0, &hi0, &lo0);
    mulhilo(PHILOX_M1, c2, &hi1, &lo1);
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static inline void block_words(uint64_t seed, uint32_t stream, uint64_t block, uint32_t w[4]) {
  uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), stream, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  synth_philox4x32_10(ctr, key, w);
}

/* Raw 32-bit words: element i of (seed, stream). */
void synth_u32(uint64_t seed, uint32_t stream, uint64_t n, uint32_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (int64_t)((n + 3) / 4); ++b) {
    uint32_t w[4];
    block_words(seed, stream, (uint64_t)b, w);
    for (int j = 0; j < 4; ++j) {
      uint64_t i = (uint64_t)b * 4 + j;
      if (i < n) out[i] = w[j];
    }
  }
}

/* Uniforms in [0,1): u = (x >> 8) * 2^-24, exact in fp32. */
void synth_uniform(uint64_t seed, uint32_t stream, uint64_t n, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (int64_t)((n + 3) / 4); ++b) {
    uint32_t w[4];
    block_words(seed, stream, (uint64_t)b, w);
    for (int j = 0; j < 4; ++j) {
      uint64_t i = (uint64_t)b * 4 + j;
      if (i < n) out[i] = (float)(w[j] >> 8) * (1.0f / 16777216.0f);
    }
  }
}

/* Integers uniform in [0, bound): floor(x * bound / 2^32). */
void synth_randint(uint64_t seed, uint32_t stream, uint64_t n, uint32_t bound, int32_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (int64_t)((n + 3) / 4); ++b) {
    uint32_t w[4];
    block_words(seed, stream, (uint64_t)b, w);
    for (int j = 0; j < 4; ++j) {
      uint64_t i = (uint64_t)b * 4 + j;
      if (i < n) out[i] = (int32_t)(((uint64_t)w[j] * (uint64_t)bound) >> 32);
    }
  }
}

/* Box-Muller in double: words (w0,w1) -> two normals, (w2,w3) -> two more.
 * u1 = ((w >> 8) + 1) * 2^-24 lies in (0,1] so the log is finite. */
static inline void normals4(uint64_t seed, uint32_t stream, uint64_t block, double z[4]) {
  uint32_t w[4];
  block_words(seed, stream, block, w);
  const double two_pi = 6.283185307179586476925286766559;
  for (int p = 0; p < 2; ++p) {
    double u1 = ((double)(w[2 * p] >> 8) + 1.0) * (1.0 / 16777216.0);
    double u2 = (double)(w[2 * p + 1] >> 8) * (1.0 / 16777216.0);
    double r = sqrt(-2.0 * log(u1));
    z[2 * p] = r * cos(two_pi * u2);
    z[2 * p + 1] = r * sin(two_pi * u2);
  }
}

void synth_normal_f32(uint64_t seed, uint32_t stream, uint64_t n, double mean, double std, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (int64_t)((n + 3) / 4); ++b) {
    double z[4];
    normals4(seed, stream, (uint64_t)b, z);
    for (int j = 0; j < 4; ++j) {
      uint64_t i = (uint64_t)b * 4 + j;
      if (i < n) out[i] = (float)(mean + std * z[j]);
    }
  }
}

/* fp32 -> bf16 bits, round to nearest even (inputs here are finite). */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

void synth_normal_bf16(uint64_t seed, uint32_t stream, uint64_t n, double mean, double std, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < (int64_t)((n + 3) / 4); ++b) {
    double z[4];
    normals4(seed, stream, (uint64_t)b, z);
    for (int j = 0; j < 4; ++j) {
      uint64_t i = (uint64_t)b * 4 + j;
      if (i < n) out[i] = f32_to_bf16_rne((float)(mean + std * z[j]));
    }
  }
}

void synth_f32_to_bf16(const float* in, uint64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}
