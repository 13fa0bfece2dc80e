/*
 * synth.c -- seeded synthetic inputs for the frame step (host side).
 *
 * This module draws the random inputs that both the CUDA library and the
 * CPU oracle consume: weights, activations, positions and the raw fp32
 * values of a prefilled K/V history.  It holds none of the decode step's
 * arithmetic (no norm, projection, rotation, quantisation or attention);
 * turning raw K/V values into FP8 codes is left to each side's own
 * quantiser.
 *
 * Generator (one definition, implemented again bit for bit in synth_gpu.cu):
 *   mix(z)      the SplitMix64 output function (Steele, Lea, Flood 2014):
 *               z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *               z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31.
 *   key(seed, stream) = mix(seed * 0xD1B54A32D192ED03 + (stream + 1) * G),
 *               G = 0x9E3779B97F4A7C15 (the SplitMix64 increment).
 *   word(key, n)      = mix(key + (n + 1) * G)          (counter-based).
 *   normal(key, i)    = (sum of twelve 20-bit fields of words 4i..4i+3,
 *                        three per word at bits 0, 20 and 40) - 6 * 2^20,
 *                       times 2^-20.  Irwin-Hall(12) - 6: mean 0, variance 1,
 *                       support (-6, 6); every value is exact in fp32.
 *   uniform_int(key, i, lo, hi) = lo + (word(key, i) >> 32) % (hi - lo).
 *   bf16(x)     round-to-nearest-even of an fp32 value to bfloat16.
 */
#include <stdint.h>
#include <string.h>

#define SYNTH_G 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * 0xD1B54A32D192ED03ULL + (stream + 1) * SYNTH_G);
}

static inline uint64_t word_at(uint64_t key, uint64_t n) {
  return mix64(key + (n + 1) * SYNTH_G);
}

static inline float normal_at(uint64_t key, uint64_t i) {
  uint32_t sum = 0;
  for (int j = 0; j < 4; ++j) {
    uint64_t w = word_at(key, 4 * i + (uint64_t)j);
    sum += (uint32_t)(w & 0xFFFFF) + (uint32_t)((w >> 20) & 0xFFFFF) +
           (uint32_t)((w >> 40) & 0xFFFFF);
  }
  return (float)((int32_t)sum - 6 * 1048576) * (1.0f / 1048576.0f);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) /* inf / nan: keep, quiet nan */
    return (uint16_t)((u >> 16) | ((u & 0x007FFFFFu) ? 0x40u : 0u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

uint64_t synth_word(uint64_t seed, uint64_t stream, uint64_t n) {
  return word_at(synth_key(seed, stream), n);
}

/* out[j] = normal(key(seed, stream), start + j), j < count. */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t start,
                      int64_t count, float* out) {
  uint64_t key = synth_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < count; ++j) out[j] = normal_at(key, start + (uint64_t)j);
}

/* out[j] = bf16(normal(key, start + j) * scale), the product in fp32. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t start,
                       int64_t count, float scale, uint16_t* out) {
  uint64_t key = synth_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < count; ++j) {
    float v = normal_at(key, start + (uint64_t)j) * scale;
    out[j] = f32_to_bf16_rne(v);
  }
}

/* out[j] = lo + (word(key, start + j) >> 32) % (hi - lo). */
void synth_uniform_int(uint64_t seed, uint64_t stream, uint64_t start,
                       int64_t count, int32_t lo, int32_t hi, int32_t* out) {
  uint64_t key = synth_key(seed, stream);
  uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo);
  for (int64_t j = 0; j < count; ++j)
    out[j] = (int32_t)((int64_t)lo + (int64_t)((word_at(key, start + (uint64_t)j) >> 32) % span));
}

/* Fill out[j] = bf16(value) for a constant (used for RMSNorm gains). */
void synth_fill_bf16(int64_t count, float value, uint16_t* out) {
  uint16_t b = f32_to_bf16_rne(value);
  for (int64_t j = 0; j < count; ++j) out[j] = b;
}

/*
 * Raw K/V history values for sessions [s0, s0+ns), one (layer, K|V) slab.
 * Stream = kv_stream_base + 2*layer + which; element index of
 * (s, h, t, i) = ((s*H + h)*T_ref + t)*D + i, which does not depend on how
 * many sessions a buffer holds, so a smaller batch is a prefix of a larger.
 * Writes out[((s-s0)*H + h)*T_max + t][i] for t < t_count (t_count <= T_ref).
 */
void synth_kv_slab_f32(uint64_t seed, uint64_t stream, int s0, int ns, int H,
                       int T_ref, int t_count, int D, int64_t out_T, float* out) {
  uint64_t key = synth_key(seed, stream);
  int64_t rows = (int64_t)ns * H;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    int64_t s = s0 + r / H, h = r % H;
    for (int t = 0; t < t_count; ++t) {
      uint64_t base = (uint64_t)(((s * H + h) * T_ref + t) * D);
      float* o = out + (r * out_T + t) * D;
      for (int i = 0; i < D; ++i) o[i] = normal_at(key, base + (uint64_t)i);
    }
  }
}
