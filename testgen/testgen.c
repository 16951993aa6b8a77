/*
 * Seeded, counter-based synthetic input generator.
 *
 * This file produces INPUTS only (activations, weights, biases) for the MoE
 * layer; it holds none of the layer's arithmetic.  Both the CPU oracle and the
 * CUDA path are fed from it, so that the two sides see identical bits.
 *
 * Definition (fixed, so any implementation can reproduce it):
 *   gamma     = 0x9E3779B97F4A7C15
 *   mix64(z)  = SplitMix64 finaliser:  z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                                      z ^= z>>27; z *= 0x94D049BB133111EB;
 *                                      z ^= z>>31
 *   key(seed, tensor_id) = mix64(seed * gamma + mix64((tensor_id + 1) * gamma))
 *   word(k)   = mix64(key + (k + 1) * gamma)            (the k-th SplitMix64 output)
 *   element i of a tensor: u1 = ((word(2i) >> 11) + 1) * 2^-53   in (0, 1]
 *                          u2 =  (word(2i+1) >> 11)    * 2^-53   in [0, 1)
 *                          z  = sqrt(-2 ln u1) * cos(2 pi u2)    (Box-Muller, cosine branch)
 *   value = (float)(std * z)   rounded fp64 -> fp32 to nearest-even,
 *   and for bf16 tensors the fp32 value is rounded once more to bf16, nearest-even.
 *
 * Every element depends only on (seed, tensor_id, i), so any thread count and
 * any chunking give the same array.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define TG_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t tg_mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t tg_key(uint64_t seed, uint64_t tensor_id) {
  return tg_mix64(seed * TG_GAMMA + tg_mix64((tensor_id + 1ULL) * TG_GAMMA));
}

static inline double tg_normal_keyed(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t w1 = tg_mix64(key + (2ULL * i + 1ULL) * TG_GAMMA);
  uint64_t w2 = tg_mix64(key + (2ULL * i + 2ULL) * TG_GAMMA);
  double u1 = (double)((w1 >> 11) + 1ULL) * 0x1.0p-53;
  double u2 = (double)(w2 >> 11) * 0x1.0p-53;
  return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

static inline uint16_t tg_f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* One standard-normal draw, element i of tensor `tensor_id`. */
double testgen_normal_at(uint64_t seed, uint64_t tensor_id, uint64_t i) {
  return tg_normal_keyed(tg_key(seed, tensor_id), i);
}

/* out[j] = (float)(std * z(offset + j)), j in [0, n). */
void testgen_fill_f32(uint64_t seed, uint64_t tensor_id, uint64_t offset, uint64_t n, double std, float* out) {
  const uint64_t key = tg_key(seed, tensor_id);
  long long nn = (long long)n;
#pragma omp parallel for schedule(static)
  for (long long j = 0; j < nn; ++j) out[j] = (float)(std * tg_normal_keyed(key, offset + (uint64_t)j));
}

/* Same values as testgen_fill_f32, rounded once more to bf16 (bit patterns). */
void testgen_fill_bf16(uint64_t seed, uint64_t tensor_id, uint64_t offset, uint64_t n, double std, uint16_t* out) {
  const uint64_t key = tg_key(seed, tensor_id);
  long long nn = (long long)n;
#pragma omp parallel for schedule(static)
  for (long long j = 0; j < nn; ++j)
    out[j] = tg_f32_to_bf16_rne((float)(std * tg_normal_keyed(key, offset + (uint64_t)j)));
}

void testgen_f32_to_bf16(const float* in, uint16_t* out, uint64_t n) {
  long long nn = (long long)n;
#pragma omp parallel for schedule(static)
  for (long long j = 0; j < nn; ++j) out[j] = tg_f32_to_bf16_rne(in[j]);
}

void testgen_bf16_to_f32(const uint16_t* in, float* out, uint64_t n) {
  long long nn = (long long)n;
#pragma omp parallel for schedule(static)
  for (long long j = 0; j < nn; ++j) {
    uint32_t u = (uint32_t)in[j] << 16;
    memcpy(&out[j], &u, 4);
  }
}
