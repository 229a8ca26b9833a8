/*
 * Seeded synthetic inputs shared by the GPU path's tests/bench and the oracle.
 *
 * This file holds no arithmetic of the model: only counter-based random
 * streams (splitmix64, Steele/Lea/Flood 2014, as published by S. Vigna),
 * the Box-Muller transform for normal deviates, fp32 -> bfloat16
 * round-to-nearest-even, uniform integers and a Fisher-Yates permutation.
 *
 * Every value depends only on (seed, stream, element index), so any slice of
 * any tensor can be regenerated independently, in any order, on any thread.
 * Built with -ffp-contract=off so x86-64 and aarch64 hosts give identical bits
 * (apart from libm's last-ulp behaviour, which bf16 rounding absorbs).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* i-th output (0-based) of a splitmix64 generator whose state starts at s0. */
uint64_t synth_splitmix64_at(uint64_t s0, uint64_t i) {
  return sm64_mix(s0 + (i + 1) * GOLDEN_GAMMA);
}

/* Initial state of the stream `stream` under `seed`. */
uint64_t synth_stream_state(uint64_t seed, uint64_t stream) {
  return synth_splitmix64_at(synth_splitmix64_at(seed, 0) ^ stream, stream);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Standard normal pair (2p, 2p+1) of the stream (Box-Muller, fp64). */
static inline void normal_pair(uint64_t s0, uint64_t p, double* z0, double* z1) {
  uint64_t a = synth_splitmix64_at(s0, 2 * p);
  uint64_t b = synth_splitmix64_at(s0, 2 * p + 1);
  double u1 = (double)((a >> 11) + 1) * 0x1.0p-53; /* (0, 1] */
  double u2 = (double)(b >> 11) * 0x1.0p-53;       /* [0, 1) */
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  *z0 = r * cos(t);
  *z1 = r * sin(t);
}

/* Runs BODY for every k < n with z = N_{offset+k}; each pair shares one transform. */
#define FOR_EACH_NORMAL(s0, offset, n, BODY)                                  \
  do {                                                                        \
    uint64_t p_lo = (offset) >> 1, p_hi = ((offset) + (n) + 1) >> 1;          \
    int64_t np_ = (int64_t)(p_hi - p_lo);                                     \
    _Pragma("omp parallel for schedule(static)")                              \
    for (int64_t q = 0; q < np_; ++q) {                                       \
      double zz[2];                                                           \
      uint64_t p = p_lo + (uint64_t)q;                                        \
      normal_pair(s0, p, &zz[0], &zz[1]);                                     \
      for (int h = 0; h < 2; ++h) {                                           \
        uint64_t i = 2 * p + (uint64_t)h;                                     \
        if (i < (offset) || i >= (offset) + (n)) continue;                    \
        uint64_t k = i - (offset);                                            \
        double z = zz[h];                                                     \
        BODY;                                                                 \
      }                                                                       \
    }                                                                         \
  } while (0)

/* out[k] = bf16(float(mean + std * N_{offset+k})), k < n. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, double mean,
                       double std, uint16_t* out) {
  uint64_t s0 = synth_stream_state(seed, stream);
  FOR_EACH_NORMAL(s0, offset, n, out[k] = f32_to_bf16_rne((float)(mean + std * z)));
}

/* out[k] = float(mean + std * N_{offset+k}). */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, double mean,
                      double std, float* out) {
  uint64_t s0 = synth_stream_state(seed, stream);
  FOR_EACH_NORMAL(s0, offset, n, out[k] = (float)(mean + std * z));
}

/* out[k] uniform in [lo, hi] (inclusive); requires hi - lo + 1 <= 2^32. */
void synth_uniform_int(uint64_t seed, uint64_t stream, uint64_t n, int64_t lo, int64_t hi,
                       int32_t* out) {
  uint64_t s0 = synth_stream_state(seed, stream);
  uint64_t span = (uint64_t)(hi - lo + 1);
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < nn; ++k) {
    uint64_t a = synth_splitmix64_at(s0, (uint64_t)k);
    out[k] = (int32_t)(lo + (int64_t)(((a >> 32) * span) >> 32));
  }
}

/* Fisher-Yates shuffle of 0..n-1 driven by the stream. */
void synth_permutation(uint64_t seed, uint64_t stream, int32_t n, int32_t* out) {
  uint64_t s0 = synth_stream_state(seed, stream);
  for (int32_t i = 0; i < n; ++i) out[i] = i;
  for (int32_t i = n - 1; i > 0; --i) {
    uint64_t a = synth_splitmix64_at(s0, (uint64_t)i);
    int32_t j = (int32_t)(((a >> 32) * (uint64_t)(i + 1)) >> 32);
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}

/* bf16 bit patterns -> float32 values (exact widening). */
void synth_bf16_to_f32(const uint16_t* in, uint64_t n, float* out) {
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < nn; ++k) {
    uint32_t u = (uint32_t)in[k] << 16;
    memcpy(&out[k], &u, 4);
  }
}
