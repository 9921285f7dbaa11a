// Device fills for the seeded synthetic inputs (same definitions as synth_host.c, see synth.h).
// Used to generate gigabyte-scale inputs in place on the GPU; not part of any timed path.
#include <cuda_runtime.h>
#include "synth.h"

namespace {

__global__ void fill_normal_bf16_kernel(uint16_t* out, uint64_t key, uint64_t offset, uint64_t n, float scale) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = dfs_f32_to_bf16_rne(dfs_normal_f32(key, offset + i, scale));
}

__global__ void fill_normal_f32_kernel(float* out, uint64_t key, uint64_t offset, uint64_t n, float scale) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = dfs_normal_f32(key, offset + i, scale);
}

int grid_for(uint64_t n) {
  uint64_t blocks = (n + 255) / 256;
  if (blocks > 148ull * 64ull) blocks = 148ull * 64ull;
  if (blocks == 0) blocks = 1;
  return (int)blocks;
}

}  // namespace

extern "C" int dfs_cuda_fill_normal_bf16(void* out, uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n,
                                         float scale, void* stream) {
  if (n == 0) return 0;
  fill_normal_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((uint16_t*)out, dfs_key(seed, tid), offset,
                                                                         n, scale);
  return (int)cudaGetLastError();
}

extern "C" int dfs_cuda_fill_normal_f32(void* out, uint64_t seed, uint64_t tid, uint64_t offset, uint64_t n,
                                        float scale, void* stream) {
  if (n == 0) return 0;
  fill_normal_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>((float*)out, dfs_key(seed, tid), offset, n,
                                                                        scale);
  return (int)cudaGetLastError();
}
