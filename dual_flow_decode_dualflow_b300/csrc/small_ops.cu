// Row-wise kernels of the decode step and the fp32 (CUDA-core, no TF32) path.
//
//  - embedding gather of both flows (separate embeddings E1, E2: "Arquitetura Central") fused with
//    the first pre-norm; RMSNorm with the shared gain (LLaMA family named under "Contribuicoes
//    Principais"; shared because embeddings and couplings are the only extra parameters, "Custos
//    de Inferencia vs. Treinamento"); the primary query's RoPE for attention-only calls.
//  - fp32 storage configurations run every step with these plain kernels: projections, query
//    coupling + RoPE + primary-only KV append, shared-KV attention (explicit two-pass softmax),
//    SwiGLU with b coupling, c coupling with residual update.
#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

__device__ __forceinline__ void set_status(int32_t* st, int code) { atomicCAS(st, 0, code); }

// Sum over the block (blockDim.x a multiple of 32, <= 1024).
__device__ float block_sum(float v, float* red) {
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < nw; ++i) s += red[i];
  return s;
}

__device__ float block_max(float v, float* red) {
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float s = -INFINITY;
  for (int i = 0; i < nw; ++i) s = fmaxf(s, red[i]);
  return s;
}

// Four consecutive storage-dtype elements <-> float4.
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// One warp per row n = f * B + b. With E1/E2 given, the row is first gathered from the flow's
// embedding (h_n = E_f[token_b], written to the fp32 residual); then x_n = h_n / rms(h_n) * g in
// the storage dtype. d must be a multiple of 4.
template <typename T>
__global__ void rmsnorm_rows_kernel(float* h, const T* E1, const T* E2, const int32_t* tokens, const T* g, T* x,
                                    int rows, int B, int d, int V, float eps, int32_t* status) {
  const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (n >= rows) return;
  const T* src = nullptr;
  if (E1 != nullptr) {
    int tok = tokens[n % B];
    if (tok < 0 || tok >= V) {
      if (lane == 0) set_status(status, DF_ERR_DEVICE_BOUNDS);
      tok = 0;
    }
    src = (n / B ? E2 : E1) + (size_t)tok * d;
  }
  float* hr = h + (size_t)n * d;
  float ss = 0.f;
#pragma unroll 4
  for (int q = lane * 4; q < d; q += 128) {
    const float4 v = src ? ld4(src + q) : ld4(hr + q);
    if (src) st4(hr + q, v);
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float r = 1.0f / sqrtf(ss / (float)d + eps);
  T* xr = x + (size_t)n * d;
#pragma unroll 4
  for (int q = lane * 4; q < d; q += 128) {
    const float4 v = src ? ld4(src + q) : ld4(hr + q);
    const float4 gg = ld4(g + q);
    st4(xr + q, make_float4(v.x * r * gg.x, v.y * r * gg.y, v.z * r * gg.z, v.w * r * gg.w));
  }
}

// Input of a norm-fed bf16 projection (one warp per row n = f * B + b): x_n = bf16(h_n (*) g) and
// ss[n] = sum h_n^2; the projection scales its fp32 product by 1 / sqrt(ss / d + eps). With E1/E2
// given (first kernel of the decode step) the row is first gathered, h_n = E_f[token_b], and
// written to the fp32 residual. d must be a multiple of 4.
__global__ void norm_prep_kernel(float* h, const __nv_bfloat16* E1, const __nv_bfloat16* E2, const int32_t* tokens,
                                 const __nv_bfloat16* g, __nv_bfloat16* x, float* ss, int ss_ld, int rows, int B, int d,
                                 int V, int32_t* status, unsigned long long* t_start, unsigned long long* t_end) {
  griddep_launch_dependents();
  const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  // in-graph timing (nullable): the step's start and this launch's end
  if (t_start != nullptr && threadIdx.x == 0) atomicMin(t_start, (unsigned long long)globaltimer());
  if (n >= rows) return;
  const __nv_bfloat16* src = nullptr;
  if (E1 != nullptr) {
    int tok = tokens[n % B];
    if (tok < 0 || tok >= V) {
      if (lane == 0) set_status(status, DF_ERR_DEVICE_BOUNDS);
      tok = 0;
    }
    src = (n / B ? E2 : E1) + (size_t)tok * d;
  }
  float* hr = h + (size_t)n * d;
  __nv_bfloat16* xr = x + (size_t)n * d;
  float s = 0.f;
  // the row in chunks of 16 vectors per lane (2048 features per warp): every load of a chunk is
  // issued before its stores, so a chunk costs one round trip
  for (int q0 = lane * 4; q0 < d; q0 += 16 * 128) {
    float4 v[16], gg[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int q = q0 + 128 * j;
      if (q < d) {
        v[j] = src ? ld4(src + q) : ld4(hr + q);
        gg[j] = ld4(g + q);
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int q = q0 + 128 * j;
      if (q < d) {
        if (src) st4(hr + q, v[j]);
        st4(xr + q, make_float4(v[j].x * gg[j].x, v[j].y * gg[j].y, v[j].z * gg[j].z, v[j].w * gg[j].w));
        s += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
      }
    }
  }
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) ss[(size_t)n * ss_ld] = s;
  if (t_end != nullptr && lane == 0) atomicMax(t_end, (unsigned long long)globaltimer());
}

// Attention-only call without the auxiliary flow: q[0, b, h] = RoPE(q1[b, h]) at position seq_len[b].
__global__ void rope_q1_bf16_kernel(const __nv_bfloat16* q1, __nv_bfloat16* q, const int32_t* seq_len,
                                    const float2* rope, int Hq, int max_ctx, int32_t* status) {
  const int b = blockIdx.x / Hq, h = blockIdx.x % Hq, f = threadIdx.x;  // 128 threads
  const int pos = seq_len[b];
  if (pos < 0 || pos > max_ctx) {
    if (f == 0) set_status(status, DF_ERR_DEVICE_BOUNDS);
    return;
  }
  const size_t base = ((size_t)b * Hq + h) * kHeadDim;
  const float2 cs = rope[(size_t)pos * 64 + (f & 63)];
  const float x = __bfloat162float(q1[base + f]), xp = __bfloat162float(q1[base + (f ^ 64)]);
  q[base + f] = __float2bfloat16_rn(f < 64 ? x * cs.x - xp * cs.y : x * cs.x + xp * cs.y);
}

// ---------------------------------- fp32 path ----------------------------------

// y[m, n] (+)= sum_k x[m, k] W[n, k]; one warp per output feature n.
__global__ void linear_f32_kernel(const float* x, int M, const float* W, int N, int K, float* y, int accumulate) {
  const int n = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (n >= N) return;
  const float* w = W + (size_t)n * K;
  for (int m = 0; m < M; ++m) {
    const float* xm = x + (size_t)m * K;
    float s = 0.f;
    for (int k = lane; k < K; k += 32) s += xm[k] * w[k];
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) {
      if (accumulate) y[(size_t)m * N + n] += s;
      else y[(size_t)m * N + n] = s;
    }
  }
}

struct CacheGeom {
  int paged, page_size, max_ctx, max_pages, pages_per_seq, n_kv_heads, head_dim;
  const int32_t* page_table;
};

__device__ __forceinline__ long long cache_off(const CacheGeom& g, int b, int hk, int pos) {
  if (pos < 0 || pos >= g.max_ctx) return -1;
  if (!g.paged) return ((long long)(b * g.n_kv_heads + hk) * g.max_ctx + pos) * g.head_dim;
  const int lp = pos / g.page_size;
  if (lp >= g.pages_per_seq) return -1;
  const int pid = g.page_table[(size_t)b * g.pages_per_seq + lp];
  if (pid < 0 || pid >= g.max_pages) return -1;
  return (((long long)pid * g.n_kv_heads + hk) * g.page_size + pos % g.page_size) * g.head_dim;
}

// raw: [M, (Hq + 2 Hkv) D] projections (rows flow-major). Query coupling (before RoPE), RoPE of
// q1, q2, k1 at position seq_len[b], q stored fp32 [2, B, Hq, D], k1/v1 appended (primary only).
__global__ void qkv_post_f32_kernel(const float* raw, int B, int aux_on, int Hq, const float* a, float* kc, float* vc,
                                    CacheGeom geo, const int32_t* seq_len, const float2* rope, float* q,
                                    int32_t* status) {
  const int D = geo.head_dim, half = D / 2, Hkv = geo.n_kv_heads;
  const int b = blockIdx.x, hs = blockIdx.y, i = threadIdx.x;
  if (i >= half) return;
  const int ncol = (Hq + 2 * Hkv) * D;
  const int pos = seq_len[b];
  if (pos < 0 || pos > geo.max_ctx) {
    if (i == 0) set_status(status, DF_ERR_DEVICE_BOUNDS);
    return;
  }
  const float2 cs = rope[(size_t)pos * half + i];
  const float* r1 = raw + (size_t)b * ncol;
  if (hs < Hq) {
    const int c = hs * D + i;
    const float x = r1[c], xp = r1[c + half];
    q[(((size_t)0 * B + b) * Hq + hs) * D + i] = x * cs.x - xp * cs.y;
    q[(((size_t)0 * B + b) * Hq + hs) * D + i + half] = xp * cs.x + x * cs.y;
    if (aux_on) {
      const float* r2 = raw + (size_t)(B + b) * ncol;
      const float y = r2[c] + a[c] * x, yp = r2[c + half] + a[c + half] * xp;
      q[(((size_t)1 * B + b) * Hq + hs) * D + i] = y * cs.x - yp * cs.y;
      q[(((size_t)1 * B + b) * Hq + hs) * D + i + half] = yp * cs.x + y * cs.y;
    }
  } else {
    const bool is_k = hs < Hq + Hkv;
    const int hk = is_k ? hs - Hq : hs - Hq - Hkv;
    const int c = (Hq + (is_k ? 0 : Hkv) + hk) * D + i;
    const long long off = cache_off(geo, b, hk, pos);
    if (off < 0) {
      if (i == 0) set_status(status, DF_ERR_DEVICE_BOUNDS);
      return;
    }
    float v0 = r1[c], v1 = r1[c + half];
    if (is_k) {
      const float t0 = v0 * cs.x - v1 * cs.y, t1 = v1 * cs.x + v0 * cs.y;
      v0 = t0;
      v1 = t1;
    }
    float* dst = is_k ? kc : vc;
    dst[off + i] = v0;
    dst[off + i + half] = v1;
  }
}

// Attention-only fp32: raw = Wq . h2 [B, Hq D]; q[0] = RoPE(q1), q[1] = RoPE(raw + a (*) q1).
__global__ void q2_post_f32_kernel(const float* raw, const float* q1, int B, int aux_on, int Hq, int D,
                                   const float* a, const int32_t* seq_len, const float2* rope, int max_ctx, float* q,
                                   int32_t* status) {
  const int b = blockIdx.x, h = blockIdx.y, i = threadIdx.x, half = D / 2;
  if (i >= half) return;
  const int pos = seq_len[b];
  if (pos < 0 || pos > max_ctx) {
    if (i == 0) set_status(status, DF_ERR_DEVICE_BOUNDS);
    return;
  }
  const float2 cs = rope[(size_t)pos * half + i];
  const size_t c = ((size_t)b * Hq + h) * D + i;
  const float x = q1[c], xp = q1[c + half];
  q[(((size_t)0 * B + b) * Hq + h) * D + i] = x * cs.x - xp * cs.y;
  q[(((size_t)0 * B + b) * Hq + h) * D + i + half] = xp * cs.x + x * cs.y;
  if (aux_on) {
    const size_t cr = (size_t)b * Hq * D + h * D + i;
    const float y = raw[cr] + a[h * D + i] * x, yp = raw[cr + half] + a[h * D + i + half] * xp;
    q[(((size_t)1 * B + b) * Hq + h) * D + i] = y * cs.x - yp * cs.y;
    q[(((size_t)1 * B + b) * Hq + h) * D + i + half] = yp * cs.x + y * cs.y;
  }
}

// One CTA per (query head, sequence, flow): explicit softmax over every attended key.
__global__ void attention_f32_kernel(const float* q, float* o, const float* kc, const float* vc, CacheGeom geo,
                                     const int32_t* seq_len, int B, int Hq, int extra, int32_t* status) {
  extern __shared__ float sm[];
  __shared__ float red[32];
  const int h = blockIdx.x, b = blockIdx.y, f = blockIdx.z;
  const int D = geo.head_dim, G = Hq / geo.n_kv_heads, g = h / G;
  const int L = seq_len[b] + extra;
  float* qs = sm;
  float* sc = sm + D;
  const size_t qo = (((size_t)f * B + b) * Hq + h) * D;
  if (L <= 0 || L > geo.max_ctx) {
    if (L != 0 && threadIdx.x == 0) set_status(status, DF_ERR_DEVICE_BOUNDS);
    for (int d = threadIdx.x; d < D; d += blockDim.x) o[qo + d] = 0.f;
    return;
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x) qs[d] = q[qo + d];
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)D);
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < L; j += blockDim.x) {
    const long long off = cache_off(geo, b, g, j);
    float s = -INFINITY;
    if (off >= 0) {
      s = 0.f;
      for (int d = 0; d < D; ++d) s += qs[d] * kc[off + d];
      s *= scale;
    } else {
      set_status(status, DF_ERR_DEVICE_BOUNDS);
    }
    sc[j] = s;
    mx = fmaxf(mx, s);
  }
  mx = block_max(mx, red);
  float sum = 0.f;
  for (int j = threadIdx.x; j < L; j += blockDim.x) {
    const float p = expf(sc[j] - mx);
    sc[j] = p;
    sum += p;
  }
  sum = block_sum(sum, red);
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < L; ++j) {
      const long long off = cache_off(geo, b, g, j);
      if (off >= 0) acc += sc[j] * vc[off + d];
    }
    o[qo + d] = acc / sum;
  }
}

// raw [M, 2F] (gate | up): u1 = silu(g1) up1; u2 = silu(g2) up2 + b (*) u1.
__global__ void swiglu_f32_kernel(const float* raw, int B, int aux_on, int F, const float* bc, float* u) {
  const int b = blockIdx.y;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < F; j += gridDim.x * blockDim.x) {
    const float g1 = raw[(size_t)b * 2 * F + j], p1 = raw[(size_t)b * 2 * F + F + j];
    const float u1 = g1 / (1.0f + expf(-g1)) * p1;
    u[(size_t)b * F + j] = u1;
    if (aux_on) {
      const float g2 = raw[(size_t)(B + b) * 2 * F + j], p2 = raw[(size_t)(B + b) * 2 * F + F + j];
      u[(size_t)(B + b) * F + j] = g2 / (1.0f + expf(-g2)) * p2 + bc[j] * u1;
    }
  }
}

// h1 += y1; h2 += y2 + c (*) y1 (c == nullptr: plain residual add).
__global__ void couple_add_f32_kernel(const float* raw, int B, int aux_on, int n, const float* c, float* h) {
  const int b = blockIdx.y;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    const float y1 = raw[(size_t)b * n + i];
    h[(size_t)b * n + i] += y1;
    if (aux_on) h[(size_t)(B + b) * n + i] += raw[(size_t)(B + b) * n + i] + (c ? c[i] * y1 : 0.f);
  }
}

CacheGeom geom(const dualflow_ctx* ctx, const int32_t* table) {
  const dualflow_config& c = ctx->cfg;
  CacheGeom g;
  g.paged = c.paged;
  g.page_size = c.paged ? c.page_size : 1;
  g.max_ctx = c.max_ctx;
  g.max_pages = c.max_pages;
  g.pages_per_seq = c.paged ? (c.max_ctx + c.page_size - 1) / c.page_size : 0;
  g.n_kv_heads = c.n_kv_heads;
  g.head_dim = c.head_dim;
  g.page_table = table;
  return g;
}

int ok_launch() { return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA; }

}  // namespace

int launch_embed_rmsnorm(dualflow_ctx* ctx, const void* E1, const void* E2, const int32_t* tokens, const void* g,
                         int batch, int aux_on, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  const int rows = aux_on ? 2 * batch : batch;
  const int blocks = (rows + 3) / 4;
  if (c.dtype == DF_DTYPE_BF16)
    rmsnorm_rows_kernel<__nv_bfloat16><<<blocks, 128, 0, s>>>(
        ctx->h, (const __nv_bfloat16*)E1, (const __nv_bfloat16*)E2, tokens, (const __nv_bfloat16*)g,
        (__nv_bfloat16*)ctx->x, rows, batch, c.d_model, c.vocab, c.rms_eps, ctx->status);
  else
    rmsnorm_rows_kernel<float><<<blocks, 128, 0, s>>>(ctx->h, (const float*)E1, (const float*)E2, tokens,
                                                      (const float*)g, (float*)ctx->x, rows, batch, c.d_model,
                                                      c.vocab, c.rms_eps, ctx->status);
  return ok_launch();
}

int launch_embed_prep(dualflow_ctx* ctx, const void* E1, const void* E2, const int32_t* tokens, const void* g,
                      int batch, int aux_on, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  const int rows = aux_on ? 2 * batch : batch;
  norm_prep_kernel<<<(rows + 3) / 4, 128, 0, s>>>(ctx->h, (const __nv_bfloat16*)E1, (const __nv_bfloat16*)E2, tokens,
                                                  (const __nv_bfloat16*)g, (__nv_bfloat16*)ctx->x, ctx->ss, ctx->ss_ld,
                                                  rows, batch, c.d_model, c.vocab, ctx->status,
                                                  ctx->cur_stamp ? ctx->stamps : nullptr, ctx->cur_stamp);
  return ok_launch();
}

int launch_norm_prep(dualflow_ctx* ctx, float* h, const void* g, int batch, int aux_on, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  const int rows = aux_on ? 2 * batch : batch;
  norm_prep_kernel<<<(rows + 3) / 4, 128, 0, s>>>(h, nullptr, nullptr, nullptr, (const __nv_bfloat16*)g,
                                                  (__nv_bfloat16*)ctx->x, ctx->ss, ctx->ss_ld, rows, batch,
                                                  c.d_model, 0, ctx->status, nullptr, ctx->cur_stamp);
  return ok_launch();
}

int launch_rmsnorm(dualflow_ctx* ctx, const float* h, const void* g, void* x, int batch, int aux_on, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  const int rows = aux_on ? 2 * batch : batch;
  const int blocks = (rows + 3) / 4;
  if (c.dtype == DF_DTYPE_BF16)
    rmsnorm_rows_kernel<__nv_bfloat16><<<blocks, 128, 0, s>>>(const_cast<float*>(h), nullptr, nullptr, nullptr,
                                                              (const __nv_bfloat16*)g, (__nv_bfloat16*)x, rows, batch,
                                                              c.d_model, 0, c.rms_eps, ctx->status);
  else
    rmsnorm_rows_kernel<float><<<blocks, 128, 0, s>>>(const_cast<float*>(h), nullptr, nullptr, nullptr,
                                                      (const float*)g, (float*)x, rows, batch, c.d_model, 0,
                                                      c.rms_eps, ctx->status);
  return ok_launch();
}

int launch_rope_q1(dualflow_ctx* ctx, const void* q1, void* q, const int32_t* seq_len, int batch, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  rope_q1_bf16_kernel<<<batch * c.n_q_heads, kHeadDim, 0, s>>>((const __nv_bfloat16*)q1, (__nv_bfloat16*)q, seq_len,
                                                                ctx->rope, c.n_q_heads, c.max_ctx, ctx->status);
  return ok_launch();
}

int launch_linear_f32(dualflow_ctx*, const float* x, int m, const float* W, int n, int k, float* y, int accumulate,
                      cudaStream_t s) {
  if (m <= 0) return DF_OK;
  linear_f32_kernel<<<(n + 7) / 8, 256, 0, s>>>(x, m, W, n, k, y, accumulate);
  return ok_launch();
}

int launch_qkv_post_f32(dualflow_ctx* ctx, const float* raw, int batch, int aux_on, const float* a, void* k_cache,
                        void* v_cache, const int32_t* page_table, const int32_t* seq_len, float* q, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  dim3 grid(batch, c.n_q_heads + 2 * c.n_kv_heads);
  const int threads = ((c.head_dim / 2 + 31) / 32) * 32;
  qkv_post_f32_kernel<<<grid, threads, 0, s>>>(raw, batch, aux_on, c.n_q_heads, a, (float*)k_cache, (float*)v_cache,
                                               geom(ctx, page_table), seq_len, ctx->rope, q, ctx->status);
  return ok_launch();
}

int launch_q2_post_f32(dualflow_ctx* ctx, const float* raw, const float* q1, int batch, int aux_on, const float* a,
                       const int32_t* seq_len, float* q, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  dim3 grid(batch, c.n_q_heads);
  const int threads = ((c.head_dim / 2 + 31) / 32) * 32;
  q2_post_f32_kernel<<<grid, threads, 0, s>>>(raw, q1, batch, aux_on, c.n_q_heads, c.head_dim, a, seq_len, ctx->rope,
                                              c.max_ctx, q, ctx->status);
  return ok_launch();
}

int launch_attention_f32(dualflow_ctx* ctx, const float* q, float* o, const void* k_cache, const void* v_cache,
                         const int32_t* page_table, const int32_t* seq_len, int batch, int extra, int aux_on,
                         cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  dim3 grid(c.n_q_heads, batch, aux_on ? 2 : 1);
  const size_t smem = (size_t)(c.head_dim + c.max_ctx + 1) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(attention_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return DF_ERR_CUDA;
  attention_f32_kernel<<<grid, 128, smem, s>>>(q, o, (const float*)k_cache, (const float*)v_cache,
                                               geom(ctx, page_table), seq_len, batch, c.n_q_heads, extra, ctx->status);
  return ok_launch();
}

int launch_swiglu_f32(dualflow_ctx* ctx, const float* raw, int batch, int aux_on, const float* b, float* u,
                      cudaStream_t s) {
  const int F = ctx->cfg.ffn_hidden;
  dim3 grid((F + 255) / 256, batch);
  swiglu_f32_kernel<<<grid, 256, 0, s>>>(raw, batch, aux_on, F, b, u);
  return ok_launch();
}

int launch_couple_add_f32(dualflow_ctx*, const float* raw, int batch, int aux_on, int n, const float* c, float* h,
                          cudaStream_t s) {
  dim3 grid((n + 255) / 256, batch);
  couple_add_f32_kernel<<<grid, 256, 0, s>>>(raw, batch, aux_on, n, c, h);
  return ok_launch();
}

}  // namespace df
