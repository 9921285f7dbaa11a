// Mixture-of-experts MLP of the dual-flow decode step with router replay ("Replay de Roteador",
// gist.science technical summary, "Mecanismos Chave"): the auxiliary flow reuses the experts the
// primary router selects, with its own mixing weights; the two flows' expert fan-outs are set
// independently ("Contribuicoes Principais", item 3). The reading implemented here: the primary takes the
// top-k1 experts of its router logits r1 with softmax(r1) weights over them; the auxiliary flow takes
// the top-k2 experts of the PRIMARY logits r1 (so its set contains the primary's when k2 >= k1) with
// softmax weights from its own logits r2 over that set. Ties go to the lower expert index.
//
// Kernels here: the routing decision (one warp per sequence) and the combine of the experts'
// outputs (fixed summation order, output coupling c, residual, and the next RMSNorm's operand).
// The router and the expert projections themselves run on the tcgen05 stacked linear kernel.
#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

// Rank of lane e's logit among the E logits of lanes 0..E-1: the number of experts ordered before it
// (larger logit, or equal logit and lower index). The experts of rank < k are the top-k, in rank
// order. Every lane of the warp executes the shuffles; lanes >= E get rank >= E.
__device__ __forceinline__ int rank_of(float v, int e, int E) {
  int r = 0;
  for (int j = 0; j < E; ++j) {
    const float u = __shfl_sync(0xffffffffu, v, j);
    if (j != e && (u > v || (u == v && j < e))) ++r;
  }
  return e < E ? r : E + e;
}

// Softmax weight of lane e over the lanes with sel set (fp32, max-subtracted).
__device__ __forceinline__ float masked_softmax(float v, bool sel) {
  float mx = sel ? v : -INFINITY;
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const float p = sel ? expf(v - mx) : 0.f;
  float s = p;
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return sel ? p / s : 0.f;
}

// One warp per sequence b; lane e < E is expert e. rlog: [rows][E] fp32 router logits (primary rows
// 0..B-1, auxiliary rows B..2B-1). Writes sel_pos[row][e] (position of e in the row's ordered set,
// -1 if not selected), sel_w[row][e] (mixing weight), ids[f][b][kmax] (experts in set order, -1
// padded; nullable).
__global__ void moe_route_kernel(const float* rlog, int B, int E, int k1, int k2, int aux_on, int32_t* sel_pos,
                                 float* sel_w, int32_t* ids, int kmax, unsigned long long* stamp) {
  griddep_launch_dependents();
  griddep_wait();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), e = threadIdx.x & 31;
  // in-graph timing (nullable): raised by every warp as it finishes
  if (stamp != nullptr && e == 0 && b >= B) atomicMax(stamp, (unsigned long long)globaltimer());
  if (b >= B) return;
  const bool live = e < E;
  const float r1 = live ? rlog[(size_t)b * E + e] : -INFINITY;
  // the auxiliary row's logits are requested with the primary's (one round trip)
  const float r2 = (live && aux_on) ? rlog[(size_t)(B + b) * E + e] : -INFINITY;
  const int rank = rank_of(r1, e, E);
  const bool in1 = live && rank < k1;
  const float w1 = masked_softmax(r1, in1);
  if (live) {
    sel_pos[(size_t)b * E + e] = in1 ? rank : -1;
    sel_w[(size_t)b * E + e] = w1;
  }
  if (ids && e < kmax) ids[(size_t)b * kmax + e] = -1;
  __syncwarp();
  if (ids && in1) ids[(size_t)b * kmax + rank] = e;
  if (!aux_on) {
    if (ids && e < kmax) ids[((size_t)B + b) * kmax + e] = -1;
    if (stamp != nullptr && e == 0) atomicMax(stamp, (unsigned long long)globaltimer());
    return;
  }
  // auxiliary flow: the primary logits choose the set (replay), its own logits weight it
  const bool in2 = live && rank < k2;
  const float w2 = masked_softmax(r2, in2);
  if (live) {
    sel_pos[(size_t)(B + b) * E + e] = in2 ? rank : -1;
    sel_w[(size_t)(B + b) * E + e] = w2;
  }
  if (ids && e < kmax) ids[((size_t)B + b) * kmax + e] = -1;
  __syncwarp();
  if (ids && in2) ids[((size_t)B + b) * kmax + rank] = e;
  if (stamp != nullptr && e == 0) atomicMax(stamp, (unsigned long long)globaltimer());
}

// grid (B, ceil(d / 512)), 128 threads, 4 features each. For sequence b and both flows:
// y_f = sum over the row's experts, in set order, of w * Y[e][row]; y2 += c (*) y1; h_f += y_f.
// With g_next: x_next = bf16(h (*) g_next) and ss[row * ss_ld + chunk] = sum of h^2 over the chunk.
__global__ void moe_combine_kernel(const float* Y, int mrows, int d, int B, int E, int aux_on, const int32_t* sel_pos,
                                   const float* sel_w, const __nv_bfloat16* c, float* h, const __nv_bfloat16* g_next,
                                   __nv_bfloat16* x_next, float* ss, int ss_ld, int32_t* status,
                                   unsigned long long* stamp) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ int order[2][32];
  __shared__ float wts[2][32];
  __shared__ int nsel[2];
  __shared__ float red[2][4];
  const int b = blockIdx.x, chunk = blockIdx.y, t = threadIdx.x;
  const int nf = aux_on ? 2 : 1;
  if (t < 64) {
    const int f = t >> 5, e = t & 31;
    if (f < nf) {
      const int row = f * B + b;
      if (e == 0) nsel[f] = 0;
      __syncwarp();
      if (e < E) {
        const int pos = sel_pos[(size_t)row * E + e];
        if (pos >= 0 && pos < 32) {
          order[f][pos] = e;
          wts[f][pos] = sel_w[(size_t)row * E + e];
          atomicAdd(&nsel[f], 1);
        }
      }
    }
  }
  __syncthreads();
  const int i = chunk * 512 + 4 * t;
  const bool live = i < d;  // d is a multiple of 4
  float4 y[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  // the residual rows, then the expert rows in chunks of kCombineLoads, each chunk's loads issued
  // before its sums (which keep the set order)
  constexpr int kCombineLoads = 8;
  float4 hres[2];
  if (live)
    for (int f = 0; f < nf; ++f) hres[f] = *reinterpret_cast<const float4*>(h + (size_t)(f * B + b) * d + i);
  if (live) {
    for (int f = 0; f < nf; ++f) {
      const int row = f * B + b;
      for (int j0 = 0; j0 < nsel[f]; j0 += kCombineLoads) {
        float4 v[kCombineLoads];
#pragma unroll
        for (int j = 0; j < kCombineLoads; ++j)
          if (j0 + j < nsel[f]) v[j] = *reinterpret_cast<const float4*>(Y + ((size_t)order[f][j0 + j] * mrows + row) * d + i);
#pragma unroll
        for (int j = 0; j < kCombineLoads; ++j)
          if (j0 + j < nsel[f]) {
            const float w = wts[f][j0 + j];
            y[f] = make_float4(__fmaf_rn(w, v[j].x, y[f].x), __fmaf_rn(w, v[j].y, y[f].y),
                               __fmaf_rn(w, v[j].z, y[f].z), __fmaf_rn(w, v[j].w, y[f].w));
          }
      }
    }
  }
  float s[2] = {0.f, 0.f};
  if (live) {
    if (aux_on) {  // output coupling, one way: y2 += c (*) y1
      const uint2 cu = *reinterpret_cast<const uint2*>(c + i);
      const float2 c01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cu.x));
      const float2 c23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&cu.y));
      y[1] = make_float4(__fmaf_rn(c01.x, y[0].x, y[1].x), __fmaf_rn(c01.y, y[0].y, y[1].y),
                         __fmaf_rn(c23.x, y[0].z, y[1].z), __fmaf_rn(c23.y, y[0].w, y[1].w));
    }
    float2 g01 = make_float2(0.f, 0.f), g23 = g01;
    if (g_next) {
      const uint2 gu = *reinterpret_cast<const uint2*>(g_next + i);
      g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gu.x));
      g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gu.y));
    }
    for (int f = 0; f < nf; ++f) {
      const int row = f * B + b;
      float4* hp = reinterpret_cast<float4*>(h + (size_t)row * d + i);
      float4 hv = hres[f];
      hv = make_float4(__fadd_rn(hv.x, y[f].x), __fadd_rn(hv.y, y[f].y), __fadd_rn(hv.z, y[f].z),
                       __fadd_rn(hv.w, y[f].w));
      *hp = hv;
      if (g_next) {
        __nv_bfloat162 a = __floats2bfloat162_rn(__fmul_rn(hv.x, g01.x), __fmul_rn(hv.y, g01.y));
        __nv_bfloat162 bb = __floats2bfloat162_rn(__fmul_rn(hv.z, g23.x), __fmul_rn(hv.w, g23.y));
        uint2 u;
        u.x = *reinterpret_cast<uint32_t*>(&a);
        u.y = *reinterpret_cast<uint32_t*>(&bb);
        *reinterpret_cast<uint2*>(x_next + (size_t)row * d + i) = u;
        s[f] = __fmaf_rn(hv.w, hv.w, __fmaf_rn(hv.z, hv.z, __fmaf_rn(hv.y, hv.y, __fmul_rn(hv.x, hv.x))));
      }
    }
  }
  if (g_next) {
    const int w = t >> 5, lane = t & 31;
    for (int f = 0; f < 2; ++f)
      for (int off = 16; off > 0; off >>= 1) s[f] += __shfl_xor_sync(0xffffffffu, s[f], off);
    if (lane == 0) {
      red[0][w] = s[0];
      red[1][w] = s[1];
    }
    __syncthreads();
    if (t < nf) {
      const float v = ((red[t][0] + red[t][1]) + red[t][2]) + red[t][3];
      ss[(size_t)(t * B + b) * ss_ld + chunk] = v;
    }
  }
  if (stamp != nullptr) {  // in-graph timing: this launch's end
    __syncthreads();
    if (t == 0) atomicMax(stamp, (unsigned long long)globaltimer());
  }
  (void)status;
}

// ---- prefill (primary flow only, many rows): the rows each expert serves, gathered contiguously --

// One CTA per expert e (1024 threads). Counts every expert's rows, then lays the experts' row lists
// end to end in expert order (rows in row order within an expert): perm[q] = source row of gathered
// row q, pos[r * k + j] = gathered row of row r's j-th expert; expert e's rows are cut into blocks
// of 256 for the expert GEMMs, blk[g] = (expert, first gathered row, rows), n_blk = number of blocks.
__global__ void __launch_bounds__(1024) moe_plan_kernel(int R, int E, int k, const int32_t* sel_pos, int32_t* perm,
                                                        int32_t* pos, int4* blk, int32_t* n_blk, int32_t* status) {
  __shared__ int cnt[32];
  __shared__ int wsum[32];
  __shared__ int off_s, base_s, chunk_s;
  const int e = blockIdx.x, t = threadIdx.x, lane = t & 31, wid = t >> 5;
  if (t < 32) cnt[t] = 0;
  __syncthreads();
  for (int r0 = 0; r0 < R; r0 += 1024) {
    const int r = r0 + t;
    for (int j = 0; j < E; ++j) {
      const bool f = r < R && sel_pos[(size_t)r * E + j] >= 0;
      const unsigned bal = __ballot_sync(0xffffffffu, f);
      if (lane == 0 && bal) atomicAdd(&cnt[j], __popc(bal));
    }
  }
  __syncthreads();
  if (t == 0) {
    int off = 0, b0 = 0;
    for (int j = 0; j < e; ++j) {
      off += cnt[j];
      b0 += (cnt[j] + 255) / 256;
    }
    const int nb = (cnt[e] + 255) / 256, cap_blk = (R * k + 255) / 256 + E;
    for (int i = 0; i < nb; ++i)
      if (b0 + i < cap_blk) blk[b0 + i] = make_int4(e, off + 256 * i, min(256, cnt[e] - 256 * i), 0);
    if (e == E - 1) *n_blk = min(b0 + nb, cap_blk);
    if (off + cnt[e] > R * k) atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);  // more selections than k per row
    off_s = off;
    base_s = 0;
  }
  __syncthreads();
  for (int r0 = 0; r0 < R; r0 += 1024) {
    const int r = r0 + t;
    const int sp = r < R ? sel_pos[(size_t)r * E + e] : -1;
    const bool f = sp >= 0;
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) wsum[wid] = __popc(bal);
    __syncthreads();
    if (t < 32) {  // exclusive prefix of the warps' counts
      const int v = wsum[t];
      int incl = v;
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (t >= o) incl += u;
      }
      wsum[t] = incl - v;
      if (t == 31) chunk_s = incl;
    }
    __syncthreads();
    if (f) {
      const int q = off_s + base_s + wsum[wid] + __popc(bal & ((1u << lane) - 1u));
      if (q < R * k && sp < k) {
        perm[q] = r;
        pos[(size_t)r * k + sp] = q;
      } else {
        atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
      }
    }
    __syncthreads();
    if (t == 0) base_s += chunk_s;
    __syncthreads();
  }
}

// One warp per gathered row q: the source row's norm operand (bf16, d) and its sums of squares.
__global__ void moe_gather_kernel(int rows, int R, int d, const __nv_bfloat16* x, const float* ss, int ss_ld,
                                  const int32_t* perm, __nv_bfloat16* xg, float* ssg, int32_t* status) {
  const int q = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (q >= rows) return;
  const int r = perm[q];
  uint4* dst = reinterpret_cast<uint4*>(xg + (size_t)q * d);
  if (r < 0 || r >= R) {  // a row list that does not cover every gathered row: zeros, and the error
    for (int i = lane; i < d / 8; i += 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)r * d);
  for (int i = lane; i < d / 8; i += 32) dst[i] = src[i];
  for (int i = lane; i < ss_ld; i += 32) ssg[(size_t)q * ss_ld + i] = ss[(size_t)r * ss_ld + i];
}

// grid (R, ceil(d / 512)), 128 threads, 4 features each: row r's experts' outputs (gathered rows
// pos[r][j]) mixed in set order, y = sum_j w_j Y[pos[r][j]], h[r] += y; with g_next the next norm's
// operand x_next = bf16(h (*) g_next) and ss[r * ss_ld + chunk] = sum of h^2 over the chunk. The
// same arithmetic, in the same order, as the decode step's combine for the primary flow.
__global__ void moe_combine_rows_kernel(const float* yg, int R, int d, int E, int k, const int32_t* sel_pos,
                                        const float* sel_w, const int32_t* pos, float* h,
                                        const __nv_bfloat16* g_next, __nv_bfloat16* x_next, float* ss, int ss_ld,
                                        int32_t* status) {
  __shared__ int qrow[32];
  __shared__ float wts[32];
  __shared__ int nsel;
  __shared__ float red[4];
  const int r = blockIdx.x, chunk = blockIdx.y, t = threadIdx.x;
  if (t < 32) {
    if (t == 0) nsel = 0;
    __syncwarp();
    if (t < E) {
      const int p = sel_pos[(size_t)r * E + t];
      if (p >= 0 && p < k) {
        const int q = pos[(size_t)r * k + p];
        if (q < 0 || q >= R * k) {
          atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
        } else {
          qrow[p] = q;
          wts[p] = sel_w[(size_t)r * E + t];
          atomicAdd(&nsel, 1);
        }
      }
    }
  }
  __syncthreads();
  const int i = chunk * 512 + 4 * t;
  const bool live = i < d;  // d is a multiple of 4
  float s = 0.f;
  if (live) {
    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < nsel; ++j) {
      const float w = wts[j];
      const float4 v = *reinterpret_cast<const float4*>(yg + (size_t)qrow[j] * d + i);
      y = make_float4(__fmaf_rn(w, v.x, y.x), __fmaf_rn(w, v.y, y.y), __fmaf_rn(w, v.z, y.z), __fmaf_rn(w, v.w, y.w));
    }
    float4* hp = reinterpret_cast<float4*>(h + (size_t)r * d + i);
    float4 hv = *hp;
    hv = make_float4(__fadd_rn(hv.x, y.x), __fadd_rn(hv.y, y.y), __fadd_rn(hv.z, y.z), __fadd_rn(hv.w, y.w));
    *hp = hv;
    if (g_next) {
      const uint2 gu = *reinterpret_cast<const uint2*>(g_next + i);
      const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gu.x));
      const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gu.y));
      __nv_bfloat162 a = __floats2bfloat162_rn(__fmul_rn(hv.x, g01.x), __fmul_rn(hv.y, g01.y));
      __nv_bfloat162 bb = __floats2bfloat162_rn(__fmul_rn(hv.z, g23.x), __fmul_rn(hv.w, g23.y));
      uint2 u;
      u.x = *reinterpret_cast<uint32_t*>(&a);
      u.y = *reinterpret_cast<uint32_t*>(&bb);
      *reinterpret_cast<uint2*>(x_next + (size_t)r * d + i) = u;
      s = __fmaf_rn(hv.w, hv.w, __fmaf_rn(hv.z, hv.z, __fmaf_rn(hv.y, hv.y, __fmul_rn(hv.x, hv.x))));
    }
  }
  if (g_next) {
    const int w = t >> 5, lane = t & 31;
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) red[w] = s;
    __syncthreads();
    if (t == 0) ss[(size_t)r * ss_ld + chunk] = ((red[0] + red[1]) + red[2]) + red[3];
  }
}

}  // namespace

int launch_moe_route_rows(const dualflow_config& c, const float* rlog, int R, int32_t* sel_pos, float* sel_w,
                          cudaStream_t s) {
  const int kmax = c.topk_primary > c.topk_aux ? c.topk_primary : c.topk_aux;
  moe_route_kernel<<<(R + 3) / 4, 128, 0, s>>>(rlog, R, c.n_experts, c.topk_primary, c.topk_aux, 0, sel_pos, sel_w,
                                               nullptr, kmax, nullptr);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_moe_plan(const dualflow_config& c, int R, const int32_t* sel_pos, int32_t* perm, int32_t* pos, int4* blk,
                    int32_t* n_blk, int32_t* status, cudaStream_t s) {
  if (c.n_experts > 32) return DF_ERR_UNSUPPORTED;
  moe_plan_kernel<<<c.n_experts, 1024, 0, s>>>(R, c.n_experts, c.topk_primary, sel_pos, perm, pos, blk, n_blk,
                                               status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_moe_gather(int rows, int R, int d, const void* x, const float* ss, int ss_ld, const int32_t* perm, void* xg,
                      float* ssg, int32_t* status, cudaStream_t s) {
  if (d % 8 != 0) return DF_ERR_SHAPE;
  moe_gather_kernel<<<(rows + 3) / 4, 128, 0, s>>>(rows, R, d, static_cast<const __nv_bfloat16*>(x), ss, ss_ld, perm,
                                                   static_cast<__nv_bfloat16*>(xg), ssg, status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_moe_combine_rows(const dualflow_config& c, int R, const float* yg, const int32_t* sel_pos,
                            const float* sel_w, const int32_t* pos, float* h, const void* g_next, void* x_next,
                            float* ss, int ss_ld, int32_t* status, cudaStream_t s) {
  moe_combine_rows_kernel<<<dim3(R, (c.d_model + 511) / 512, 1), 128, 0, s>>>(
      yg, R, c.d_model, c.n_experts, c.topk_primary, sel_pos, sel_w, pos, h,
      static_cast<const __nv_bfloat16*>(g_next), static_cast<__nv_bfloat16*>(x_next), ss, ss_ld, status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_moe_route(dualflow_ctx* ctx, const float* rlog, int batch, int aux_on, int32_t* ids, cudaStream_t s,
                     int pdl) {
  const dualflow_config& c = ctx->cfg;
  const int kmax = c.topk_primary > c.topk_aux ? c.topk_primary : c.topk_aux;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((batch + 3) / 4, 1, 1);
  lc.blockDim = dim3(128, 1, 1);
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, moe_route_kernel, rlog, batch, c.n_experts, c.topk_primary, c.topk_aux, aux_on,
                            ctx->sel_pos, ctx->sel_w, ids, kmax, ctx->cur_stamp) == cudaSuccess
             ? DF_OK
             : DF_ERR_CUDA;
}

int launch_moe_combine(dualflow_ctx* ctx, float* h, int batch, int aux_on, const void* c_vec, const void* g_next,
                       cudaStream_t s, int pdl) {
  const dualflow_config& c = ctx->cfg;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(batch, (c.d_model + 511) / 512, 1);
  lc.blockDim = dim3(128, 1, 1);
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, moe_combine_kernel, (const float*)ctx->moe_y, 2 * c.max_batch, c.d_model, batch,
                            c.n_experts, aux_on, (const int32_t*)ctx->sel_pos, (const float*)ctx->sel_w,
                            (const __nv_bfloat16*)c_vec, h, (const __nv_bfloat16*)g_next, (__nv_bfloat16*)ctx->x,
                            ctx->ss, ctx->ss_ld, ctx->status, ctx->cur_stamp) == cudaSuccess
             ? DF_OK
             : DF_ERR_CUDA;
}

}  // namespace df
