/* Host (CPU) fills for the seeded synthetic inputs; see synth.h for the definitions. */
#include <stddef.h>
#include "synth.h"

void dfs_fill_normal_bf16(uint16_t* out, uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n, float scale) {
  const uint64_t key = dfs_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = dfs_f32_to_bf16_rne(dfs_normal_f32(key, offset + (uint64_t)i, scale));
}

void dfs_fill_normal_f32(float* out, uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n, float scale) {
  const uint64_t key = dfs_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = dfs_normal_f32(key, offset + (uint64_t)i, scale);
}

void dfs_fill_uniform_i32(int32_t* out, uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n, int32_t lo,
                          int32_t hi) {
  const uint64_t key = dfs_key(seed, tid);
  for (uint64_t i = 0; i < n; ++i) out[i] = dfs_uniform_int(key, offset + i, lo, hi);
}

/* Fisher-Yates shuffle of 0..n-1 driven by the counter hash: step i (from n-1 down to 1)
 * swaps a[i] with a[word(key, i) mod (i + 1)]. */
void dfs_permutation_i32(int32_t* out, uint64_t seed, uint64_t tid, uint64_t n) {
  const uint64_t key = dfs_key(seed, tid);
  for (uint64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (uint64_t i = n; i-- > 1;) {
    uint64_t j = dfs_word(key, i) % (i + 1);
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}
