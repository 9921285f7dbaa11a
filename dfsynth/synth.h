/* Seeded synthetic-input generator shared by the GPU side and the CPU oracle side.
 *
 * This header holds no arithmetic of the Dual-Flow method; it only defines how
 * every synthetic tensor element is drawn, so that a CUDA fill on the device and
 * a C fill on the host produce the same bits for the same (seed, tensor id, index).
 *
 *   key(seed, tid)  = mix(mix(seed + G) ^ mix(tid))
 *   word(key, c)    = mix(key + (c + 1) * G)        -- the (c+1)-th splitmix64 output
 *                                                      of a generator whose state is key
 *   mix             = the splitmix64 output finaliser (Steele, Lea & Flood, OOPSLA 2014;
 *                     constants as published by Vigna for SplitMix64), G = 0x9E3779B97F4A7C15
 *
 * Normal draws are Irwin-Hall: twelve 16-bit uniforms k_j (four per 64-bit word, three
 * words per element) give n = sum(k_j) - 393210, an integer in [-393210, 393210] with mean 0
 * and variance (65536^2 - 1); x = float(n) * float(sigma / 65536) is one IEEE fp32 multiply
 * (exact integer-to-float conversion first), so host and device agree bit for bit.
 * Storage rounding to bf16 is round-to-nearest-even on the fp32 bit pattern.
 */
#ifndef DFSYNTH_SYNTH_H
#define DFSYNTH_SYNTH_H
#include <stdint.h>

#if defined(__CUDACC__)
#define DFS_FN static __host__ __device__ __forceinline__
#else
#define DFS_FN static inline
#endif

#define DFS_GOLDEN 0x9E3779B97F4A7C15ULL
#define DFS_IH_CENTER 393210 /* 12 * 32767.5 */

DFS_FN uint64_t dfs_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

DFS_FN uint64_t dfs_key(uint64_t seed, uint64_t tid) {
  return dfs_mix64(dfs_mix64(seed + DFS_GOLDEN) ^ dfs_mix64(tid));
}

DFS_FN uint64_t dfs_word(uint64_t key, uint64_t c) { return dfs_mix64(key + (c + 1ULL) * DFS_GOLDEN); }

DFS_FN int32_t dfs_irwin_hall(uint64_t key, uint64_t i) {
  int32_t s = 0;
  for (int j = 0; j < 3; ++j) {
    uint64_t w = dfs_word(key, 3ULL * i + (uint64_t)j);
    s += (int32_t)(w & 0xFFFFu) + (int32_t)((w >> 16) & 0xFFFFu) + (int32_t)((w >> 32) & 0xFFFFu) +
         (int32_t)((w >> 48) & 0xFFFFu);
  }
  return s - DFS_IH_CENTER;
}

DFS_FN float dfs_normal_f32(uint64_t key, uint64_t i, float scale) {
  float n = (float)dfs_irwin_hall(key, i); /* |n| < 2^19: exact */
#if defined(__CUDA_ARCH__)
  return __fmul_rn(n, scale);
#else
  return n * scale;
#endif
}

DFS_FN uint16_t dfs_f32_to_bf16_rne(float f) {
  union {
    float f;
    uint32_t u;
  } v;
  v.f = f;
  uint32_t u = v.u;
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

DFS_FN int32_t dfs_uniform_int(uint64_t key, uint64_t i, int32_t lo, int32_t hi) {
  uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
  return (int32_t)((int64_t)lo + (int64_t)(dfs_word(key, i) % span));
}

#endif
