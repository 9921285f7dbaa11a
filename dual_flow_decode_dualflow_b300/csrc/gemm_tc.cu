// Stacked-activation linear layers on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// One CTA computes a 128-output-feature tile of y = x . W^T for ALL activation rows of both flows
// (primary rows then auxiliary rows, <= 256): the weight tile is the M = 128 operand, the stacked
// activations are the N operand, so every weight byte is streamed from HBM once and serves both
// flows ("Custos de Inferencia vs. Treinamento": grouping keeps the unique weights read unchanged).
// Weight and activation tiles are staged by TMA (128-byte swizzle) through a 4-stage mbarrier
// pipeline; one elected thread issues tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in TMEM).
// When the output has too few tiles to fill the GPU the reduction dimension is split across the S
// CTAs of a thread-block cluster (S <= 8). Each CTA parks its fp32 partial tile in shared memory;
// after a cluster barrier every CTA sums, over distributed shared memory and in rank order (so the
// result is deterministic and independent of which flows are present), its own 1/S slice of the
// tile's features -- feature i and its RoPE / gate-up partner i + 64 travel together -- and runs
// the epilogue on that slice:
//   EPI_QKV      q1 = Wq.x1, q2 = Wq.x2 + a (*) q1 (before RoPE), RoPE(q1, q2, k1) at position
//                seq_len[b], q stored bf16, primary k1/v1 appended to the cache at slot seq_len[b]
//                ("Atencao de KV Compartilhada Assimetrica": the auxiliary flow writes no K/V)
//   EPI_Q2       attention-only call: q2 = Wq.h2 + a (*) q1, RoPE(q1), RoPE(q2)
//   EPI_SWIGLU   u = silu(gate) (*) up for both flows, then u2 += b (*) u1 ("Acoplamento Leve")
//   EPI_COUPLE_ADD  y2 += c (*) y1, then h += y (MLP output coupling and residual)
//   EPI_ADD_F32 / EPI_STORE_F32 / EPI_STORE_BF16  residual update, logits, plain stores
#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 128;
constexpr int kABytes = kGemmTileN * kGemmTileK * 2;  // 16 KB weight tile per stage

struct GemmParams {
  GemmArgs a;
  int n_pad;     // activation rows padded to a multiple of 16 (the MMA's N)
  int splits;    // CTAs of the cluster sharing one tile's reduction (1, 2, 4 or 8)
  int kb_total;  // k / 64
  int n_tiles;
  int32_t* status;
};

__device__ __forceinline__ void set_status(int32_t* st, int code) { atomicCAS(st, 0, code); }

__device__ __forceinline__ float bf2f(const void* p, size_t i) {
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ size_t cache_slot(const GemmArgs& a, int b, int hk, int pos, int32_t* status, bool* ok) {
  *ok = true;
  if (pos < 0 || pos >= a.max_ctx) {
    set_status(status, DF_ERR_DEVICE_BOUNDS);
    *ok = false;
    return 0;
  }
  if (!a.paged) return ((size_t)(b * a.n_kv_heads + hk) * a.max_ctx + pos) * kHeadDim;
  const int lp = pos / a.page_size;
  const int pid = (lp < a.pages_per_seq) ? a.page_table[(size_t)b * a.pages_per_seq + lp] : -1;
  if (pid < 0 || pid >= a.max_pages) {
    set_status(status, DF_ERR_DEVICE_BOUNDS);
    *ok = false;
    return 0;
  }
  return (((size_t)pid * a.n_kv_heads + hk) * a.page_size + (pos % a.page_size)) * kHeadDim;
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                   const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int b_bytes = p.n_pad * 128;
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * b_bytes);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] error
  float* acc_s = reinterpret_cast<float*>(smem);       // [n_pad][128], reuses the pipeline after the mainloop

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int kb0 = (int)((long long)split * p.kb_total / p.splits);
  const int kb1 = (int)((long long)(split + 1) * p.kb_total / p.splits);
  const int nkb = kb1 - kb0;
  uint32_t ncols = 32;
  while ((int)ncols < p.n_pad) ncols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    flags[0] = 0;
    fence_mbar_init();
    tma_prefetch_map(&map_w);
    tma_prefetch_map(&map_x);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  int row0, row1;
  if (EPI == EPI_SWIGLU) {
    row0 = 64 * tile;                 // gate rows of hidden units [64 tile, 64 tile + 64)
    row1 = p.a.n_out + 64 * tile;     // up rows of the same units
  } else {
    row0 = kGemmTileN * tile;
    row1 = row0 + 64;
  }

  if (warp == 0 && lane == 0) {
    // TMA producer: weights are streamed once (evict-first), activations stay L2-resident.
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    for (int i = 0; i < nkb; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
      if (!mbar_wait(&empty[s], ph ^ 1u)) {
        flags[0] = 1;
        set_status(p.status, DF_ERR_TIMEOUT);
        break;
      }
      mbar_arrive_expect_tx(&full[s], (uint32_t)(kABytes + b_bytes));
      const int kc = (kb0 + i) * kGemmTileK;
      tma_load_2d_hint(sA + s * kABytes, &map_w, &full[s], kc, row0, pol_w);
      tma_load_2d_hint(sA + s * kABytes + kABytes / 2, &map_w, &full[s], kc, row1, pol_w);
      tma_load_2d_hint(sB + s * b_bytes, &map_x, &full[s], kc, 0, pol_x);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: 4 x (M=128, N=n_pad, K=16) per stage, accumulate in TMEM.
    const uint32_t idesc = idesc_bf16_f32(kGemmTileN, p.n_pad);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (uint32_t)(i / kStages) & 1u;
      if (!mbar_wait(&full[s], ph)) {
        flags[0] = 1;
        set_status(p.status, DF_ERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint64_t da = sdesc_kmajor_sw128(smem_u32(sA + s * kABytes));
      const uint64_t db = sdesc_kmajor_sw128(smem_u32(sB + s * b_bytes));
#pragma unroll
      for (int j = 0; j < kGemmTileK / 16; ++j)
        umma_bf16(tmem, da + 2ull * j, db + 2ull * j, idesc, (uint32_t)((i | j) != 0));
      umma_commit(&empty[s]);
    }
    umma_commit(done);
  }
  __syncwarp();

  // ---- accumulator: TMEM -> registers -> this CTA's fp32 partial tile acc_s[n][128] ----
  const bool acc_ok = mbar_wait(done, 0);
  tc_fence_after();
  if (!acc_ok) set_status(p.status, DF_ERR_TIMEOUT);
  {
    const int f = threadIdx.x;  // TMEM lane == output feature within the tile
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    for (int c0 = 0; c0 < p.n_pad; c0 += 16) {
      float v[16];
      tmem_ld16(lane_base + (uint32_t)c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) acc_s[(c0 + j) * kGemmTileN + f] = v[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, ncols);

  // ---- split reduction over distributed shared memory: this CTA owns features
  //      [lo0, lo0 + nl) and [64 + lo0, 64 + lo0 + nl) of the tile ----
  const int S = p.splits;
  const int nl = 64 / S, lo0 = split * nl, nf = 2 * nl;
  float* red = acc_s + p.n_pad * kGemmTileN;  // [n_pad][nf] (S > 1)
  if (S > 1) {
    cluster_sync();
    const int quads = nf / 4;
    const uint32_t base = smem_u32(acc_s);
    for (int it = threadIdx.x; it < p.n_pad * quads; it += kThreads) {
      const int n = it / quads, qd = it % quads;
      const int fl = qd * 4;
      const int f = fl < nl ? lo0 + fl : 64 + lo0 + (fl - nl);
      const uint32_t off = base + (uint32_t)((n * kGemmTileN + f) * 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int r = 0; r < S; ++r) {
        const float4 v = ld_dsmem_f4(mapa_shared(off, (uint32_t)r));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      *reinterpret_cast<float4*>(red + n * nf + fl) = acc;
    }
    __syncthreads();
  }
  // reduced value of activation row n, tile feature f (f in this CTA's slice)
  auto acc = [&](int n, int f) -> float {
    if (S == 1) return acc_s[n * kGemmTileN + f];
    return red[n * nf + (f < 64 ? f - lo0 : nl + f - 64 - lo0)];
  };

  // ---- epilogues: unit (i, b) covers features i and i + 64 of rows b (and m_p + b) ----
  const GemmArgs& a = p.a;
  const int m = a.m_p + a.m_a;
  if (EPI == EPI_STORE_F32 || EPI == EPI_STORE_BF16 || EPI == EPI_ADD_F32) {
    for (int it = threadIdx.x; it < nl * m; it += kThreads) {
      const int i = lo0 + it % nl, n = it / nl;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int f = i + 64 * hh, fg = tile * kGemmTileN + f;
        if (fg >= a.n_out) continue;
        const float v = acc(n, f);
        if (EPI == EPI_STORE_F32) reinterpret_cast<float*>(a.y)[(size_t)n * a.ldy + fg] = v;
        if (EPI == EPI_ADD_F32) reinterpret_cast<float*>(a.y)[(size_t)n * a.ldy + fg] += v;
        if (EPI == EPI_STORE_BF16)
          reinterpret_cast<__nv_bfloat16*>(a.y)[(size_t)n * a.ldy + fg] = __float2bfloat16_rn(v);
      }
    }
  } else if (EPI == EPI_COUPLE_ADD) {
    float* y = reinterpret_cast<float*>(a.y);
    for (int it = threadIdx.x; it < nl * a.m_p; it += kThreads) {
      const int i = lo0 + it % nl, b = it / nl;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int f = i + 64 * hh, fg = tile * kGemmTileN + f;
        if (fg >= a.n_out) continue;
        const float z1 = acc(b, f);
        y[(size_t)b * a.ldy + fg] += z1;
        if (a.m_a > 0) y[(size_t)(a.m_p + b) * a.ldy + fg] += acc(a.m_p + b, f) + bf2f(a.vec, fg) * z1;
      }
    }
  } else if (EPI == EPI_SWIGLU) {
    __nv_bfloat16* u = reinterpret_cast<__nv_bfloat16*>(a.y);
    for (int it = threadIdx.x; it < nl * a.m_p; it += kThreads) {
      const int i = lo0 + it % nl, b = it / nl;
      const int j = tile * 64 + i;  // hidden unit: gate at tile feature i, up at i + 64
      const float u1 = silu(acc(b, i)) * acc(b, i + 64);
      u[(size_t)b * a.ldy + j] = __float2bfloat16_rn(u1);
      if (a.m_a > 0) {
        const int r = a.m_p + b;
        u[(size_t)r * a.ldy + j] = __float2bfloat16_rn(silu(acc(r, i)) * acc(r, i + 64) + bf2f(a.vec, j) * u1);
      }
    }
  } else if (EPI == EPI_QKV) {
    const int Hq = a.n_q_heads, Hkv = a.n_kv_heads, B = a.m_p;
    __nv_bfloat16* qo = reinterpret_cast<__nv_bfloat16*>(a.q_out);
    for (int it = threadIdx.x; it < nl * B; it += kThreads) {
      const int i = lo0 + it % nl, b = it / nl;
      const int pos = a.seq_len[b];
      if (pos < 0 || pos > a.max_ctx) {
        set_status(p.status, DF_ERR_DEVICE_BOUNDS);
        continue;
      }
      const float2 cs = a.rope[(size_t)pos * 64 + i];
      if (tile < Hq) {
        const int h = tile;
        const float x1 = acc(b, i), x1p = acc(b, i + 64);
        const size_t o1 = (((size_t)0 * B + b) * Hq + h) * kHeadDim;
        qo[o1 + i] = __float2bfloat16_rn(x1 * cs.x - x1p * cs.y);
        qo[o1 + i + 64] = __float2bfloat16_rn(x1p * cs.x + x1 * cs.y);
        if (a.m_a > 0) {
          const float x2 = acc(B + b, i) + bf2f(a.vec, h * kHeadDim + i) * x1;
          const float x2p = acc(B + b, i + 64) + bf2f(a.vec, h * kHeadDim + i + 64) * x1p;
          const size_t o2 = (((size_t)1 * B + b) * Hq + h) * kHeadDim;
          qo[o2 + i] = __float2bfloat16_rn(x2 * cs.x - x2p * cs.y);
          qo[o2 + i + 64] = __float2bfloat16_rn(x2p * cs.x + x2 * cs.y);
        }
      } else {
        const bool is_k = tile < Hq + Hkv;
        const int hk = is_k ? tile - Hq : tile - Hq - Hkv;
        bool ok;
        const size_t off = cache_slot(a, b, hk, pos, p.status, &ok);
        if (!ok) continue;
        __nv_bfloat16* cache = reinterpret_cast<__nv_bfloat16*>(is_k ? a.k_cache : a.v_cache);
        float v0 = acc(b, i), v1 = acc(b, i + 64);
        if (is_k) {
          const float t0 = v0 * cs.x - v1 * cs.y, t1 = v1 * cs.x + v0 * cs.y;
          v0 = t0;
          v1 = t1;
        }
        cache[off + i] = __float2bfloat16_rn(v0);
        cache[off + i + 64] = __float2bfloat16_rn(v1);
      }
    }
  } else if (EPI == EPI_Q2) {
    const int Hq = a.n_q_heads, B = a.m_a, h = tile;
    __nv_bfloat16* qo = reinterpret_cast<__nv_bfloat16*>(a.q_out);
    for (int it = threadIdx.x; it < nl * B; it += kThreads) {
      const int i = lo0 + it % nl, b = it / nl;
      const int pos = a.seq_len[b];
      if (pos < 0 || pos > a.max_ctx) {
        set_status(p.status, DF_ERR_DEVICE_BOUNDS);
        continue;
      }
      const float2 cs = a.rope[(size_t)pos * 64 + i];
      const size_t qi = ((size_t)b * Hq + h) * kHeadDim;
      const float x1 = bf2f(a.q1_in, qi + i), x1p = bf2f(a.q1_in, qi + i + 64);
      const size_t o1 = (((size_t)0 * B + b) * Hq + h) * kHeadDim;
      qo[o1 + i] = __float2bfloat16_rn(x1 * cs.x - x1p * cs.y);
      qo[o1 + i + 64] = __float2bfloat16_rn(x1p * cs.x + x1 * cs.y);
      const float x2 = acc(b, i) + bf2f(a.vec, h * kHeadDim + i) * x1;
      const float x2p = acc(b, i + 64) + bf2f(a.vec, h * kHeadDim + i + 64) * x1p;
      const size_t o2 = (((size_t)1 * B + b) * Hq + h) * kHeadDim;
      qo[o2 + i] = __float2bfloat16_rn(x2 * cs.x - x2p * cs.y);
      qo[o2 + i + 64] = __float2bfloat16_rn(x2p * cs.x + x2 * cs.y);
    }
  }
  // no CTA may leave while a peer can still read its partial tile
  if (S > 1) cluster_sync();
}

template <int EPI>
int launch_epi(const CUtensorMap& mw, const CUtensorMap& mx, const GemmParams& p, size_t smem, cudaStream_t s) {
  auto kern = gemm_tc_kernel<EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return DF_ERR_CUDA;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return DF_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_tiles, p.splits, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)p.splits;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mw, mx, p) == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace

int gemm_tiles(int n_out, int epi) { return epi == EPI_SWIGLU ? n_out / 64 : (n_out + kGemmTileN - 1) / kGemmTileN; }

// Reduction splits (cluster size): the smallest power of two, at most 8, that gives every SM a
// tile slice, with at least 2 k-blocks per CTA. Depends only on the weight shape, never on which
// flows are present.
int gemm_splits(const dualflow_ctx* ctx, int n_out, int k, int epi) {
  const int tiles = gemm_tiles(n_out, epi);
  const int kb = k / kGemmTileK;
  int s = 1;
  while (s < 8 && tiles * s < ctx->num_sms && 2 * (2 * s) <= kb) s *= 2;
  return s;
}

int launch_gemm_tc(dualflow_ctx* ctx, const GemmArgs& a, cudaStream_t s) {
  const int m = a.m_p + a.m_a;
  if (m <= 0) return DF_OK;
  if (m > kGemmMaxAct || a.k % kGemmTileK != 0 || a.k <= 0) return DF_ERR_SHAPE;
  if (a.epi == EPI_SWIGLU && a.n_out % 64 != 0) return DF_ERR_SHAPE;
  GemmParams p;
  p.a = a;
  p.n_pad = ((m + 15) / 16) * 16;
  p.kb_total = a.k / kGemmTileK;
  p.n_tiles = gemm_tiles(a.n_out, a.epi);
  p.splits = gemm_splits(ctx, a.n_out, a.k, a.epi);
  p.status = ctx->status;
  const uint64_t w_rows = (a.epi == EPI_SWIGLU) ? 2ull * a.n_out : (uint64_t)a.n_out;
  CUtensorMap mw, mx;
  int rc = encode_map_2d_bf16(&mw, a.W, (uint64_t)a.k, w_rows, (uint64_t)a.k * 2, kGemmTileK, 64);
  if (rc != DF_OK) return rc;
  rc = encode_map_2d_bf16(&mx, a.x, (uint64_t)a.k, (uint64_t)m, (uint64_t)a.k * 2, kGemmTileK, (uint32_t)p.n_pad);
  if (rc != DF_OK) return rc;
  // pipeline stages; after the main loop the same bytes hold the partial tile (512 B per row) and
  // the reduced slice (512 / S B per row): 65536 + 512 n_pad >= 768 n_pad for n_pad <= 256
  const size_t smem = 1024 + (size_t)kStages * (kABytes + p.n_pad * 128) + 256;
  switch (a.epi) {
    case EPI_STORE_F32: return launch_epi<EPI_STORE_F32>(mw, mx, p, smem, s);
    case EPI_STORE_BF16: return launch_epi<EPI_STORE_BF16>(mw, mx, p, smem, s);
    case EPI_ADD_F32: return launch_epi<EPI_ADD_F32>(mw, mx, p, smem, s);
    case EPI_COUPLE_ADD: return launch_epi<EPI_COUPLE_ADD>(mw, mx, p, smem, s);
    case EPI_QKV: return launch_epi<EPI_QKV>(mw, mx, p, smem, s);
    case EPI_Q2: return launch_epi<EPI_Q2>(mw, mx, p, smem, s);
    case EPI_SWIGLU: return launch_epi<EPI_SWIGLU>(mw, mx, p, smem, s);
    default: return DF_ERR_ARG;
  }
}

}  // namespace df
