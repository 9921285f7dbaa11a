// Mixture-of-experts MLP of the dual-flow decode step with router replay ("Replay de Roteador",
// gist.science technical summary, "Mecanismos Chave"): the auxiliary flow reuses the experts the
// primary router selects, with its own mixing weights; the two flows' expert fan-outs are set
// independently ("Contribuicoes Principais", item 3). This build's reading: the primary takes the
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
                                 float* sel_w, int32_t* ids, int kmax) {
  griddep_launch_dependents();
  griddep_wait();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), e = threadIdx.x & 31;
  if (b >= B) return;
  const bool live = e < E;
  const float r1 = live ? rlog[(size_t)b * E + e] : -INFINITY;
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
    return;
  }
  // auxiliary flow: the primary logits choose the set (replay), its own logits weight it
  const float r2 = live ? rlog[(size_t)(B + b) * E + e] : -INFINITY;
  const bool in2 = live && rank < k2;
  const float w2 = masked_softmax(r2, in2);
  if (live) {
    sel_pos[(size_t)(B + b) * E + e] = in2 ? rank : -1;
    sel_w[(size_t)(B + b) * E + e] = w2;
  }
  if (ids && e < kmax) ids[((size_t)B + b) * kmax + e] = -1;
  __syncwarp();
  if (ids && in2) ids[((size_t)B + b) * kmax + rank] = e;
}

// grid (B, ceil(d / 512)), 128 threads, 4 features each. For sequence b and both flows:
// y_f = sum over the row's experts, in set order, of w * Y[e][row]; y2 += c (*) y1; h_f += y_f.
// With g_next: x_next = bf16(h (*) g_next) and ss[row * ss_ld + chunk] = sum of h^2 over the chunk.
__global__ void moe_combine_kernel(const float* Y, int mrows, int d, int B, int E, int aux_on, const int32_t* sel_pos,
                                   const float* sel_w, const __nv_bfloat16* c, float* h, const __nv_bfloat16* g_next,
                                   __nv_bfloat16* x_next, float* ss, int ss_ld, int32_t* status) {
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
  if (live) {
    for (int f = 0; f < nf; ++f) {
      const int row = f * B + b;
      for (int j = 0; j < nsel[f]; ++j) {
        const int e = order[f][j];
        const float w = wts[f][j];
        const float4 v = *reinterpret_cast<const float4*>(Y + ((size_t)e * mrows + row) * d + i);
        y[f] = make_float4(__fmaf_rn(w, v.x, y[f].x), __fmaf_rn(w, v.y, y[f].y), __fmaf_rn(w, v.z, y[f].z),
                           __fmaf_rn(w, v.w, y[f].w));
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
      float4 hv = *hp;
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
  (void)status;
}

}  // namespace

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
                            ctx->sel_pos, ctx->sel_w, ids, kmax) == cudaSuccess
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
                            ctx->ss, ctx->ss_ld, ctx->status) == cudaSuccess
             ? DF_OK
             : DF_ERR_CUDA;
}

}  // namespace df
