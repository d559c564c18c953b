/*
 * Counter-based seeded input generator: the definition shared by the host
 * (synth_host.c) and device (synth_cuda.cu) fillers.
 *
 * This module produces test and benchmark inputs only. It holds none of the
 * fused GEMM + epilogue arithmetic; both the CPU oracle and the CUDA path read
 * their inputs from it.
 *
 * Hash: SplitMix64's output mix (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), applied to a counter:
 *   key  = mix(seed + tensor_id * GOLDEN)
 *   h(i) = mix(key + (i + 1) * GOLDEN)           (all arithmetic mod 2^64)
 * so any element of any tensor can be regenerated alone.
 *
 * Normal draws: the scaled Irwin-Hall sum of eight 16-bit uniforms (the four
 * 16-bit fields of h(2e) and of h(2e+1) for element e). With S their integer
 * sum, c = 2*S - 524280 is an integer with mean 0 and standard deviation
 * sqrt((8/3)*(65536^2 - 1)); the value is (float)c * scale, one correctly
 * rounded fp32 multiply, then rounded to nearest even into fp16 or bf16.
 * Every step is integer or a single IEEE-rounded operation, so host and
 * device produce identical bits.
 */
#ifndef SYNTH_HASH_H
#define SYNTH_HASH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_FN __host__ __device__ static inline
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL

/* dtype codes shared by the fillers: 0 = fp16, 1 = bf16, 2 = fp32 */
#define SYNTH_F16 0
#define SYNTH_BF16 1
#define SYNTH_F32 2

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SYNTH_FN uint64_t synth_key(uint64_t seed, uint32_t tensor_id) {
  return synth_mix64(seed + (uint64_t)tensor_id * SYNTH_GOLDEN);
}

SYNTH_FN uint64_t synth_at(uint64_t key, uint64_t index) {
  return synth_mix64(key + (index + 1ULL) * SYNTH_GOLDEN);
}

/* centred Irwin-Hall integer c in [-524280, 524280] for element e */
SYNTH_FN int32_t synth_irwin_hall8(uint64_t key, uint64_t e) {
  uint64_t h1 = synth_at(key, 2ULL * e);
  uint64_t h2 = synth_at(key, 2ULL * e + 1ULL);
  uint32_t s = (uint32_t)(h1 & 0xFFFF) + (uint32_t)((h1 >> 16) & 0xFFFF) +
               (uint32_t)((h1 >> 32) & 0xFFFF) + (uint32_t)(h1 >> 48) +
               (uint32_t)(h2 & 0xFFFF) + (uint32_t)((h2 >> 16) & 0xFFFF) +
               (uint32_t)((h2 >> 32) & 0xFFFF) + (uint32_t)(h2 >> 48);
  return 2 * (int32_t)s - 524280;
}

/* fp32 -> fp16 bits, round to nearest even (input generation only) */
SYNTH_FN uint16_t synth_f32_to_f16_bits(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t x = v.u;
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t exp = (x >> 23) & 0xFFu;
  uint32_t man = x & 0x7FFFFFu;
  if (exp == 0xFFu) return (uint16_t)(sign | 0x7C00u | (man ? 0x200u : 0u));
  int32_t e = (int32_t)exp - 127 + 15;
  if (e >= 31) return (uint16_t)(sign | 0x7C00u);
  if (e <= 0) {
    if (e < -10) return sign;
    man |= 0x800000u;
    uint32_t shift = (uint32_t)(14 - e);
    uint32_t q = man >> shift;
    uint32_t rem = man & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (q & 1u))) q++;
    return (uint16_t)(sign | q);
  }
  uint32_t q = ((uint32_t)e << 10) | (man >> 13);
  uint32_t rem = man & 0x1FFFu;
  if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q++;
  return (uint16_t)(sign | q);
}

/* fp32 -> bf16 bits, round to nearest even (input generation only) */
SYNTH_FN uint16_t synth_f32_to_bf16_bits(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t x = v.u;
  if ((x & 0x7F800000u) == 0x7F800000u && (x & 0x7FFFFFu))
    return (uint16_t)((x >> 16) | 0x40u);
  uint32_t lsb = (x >> 16) & 1u;
  return (uint16_t)((x + 0x7FFFu + lsb) >> 16);
}

#endif
