// Stacked-activation linear layers on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// One CTA computes a 128-output-feature tile of y = x . W^T for ALL activation rows of both flows
// (primary rows then auxiliary rows, <= 256): the weight tile is the M = 128 operand, the stacked
// activations are the N operand, so every weight byte is streamed from HBM once and serves both
// flows ("Custos de Inferencia vs. Treinamento": grouping keeps the unique weights read unchanged).
// Weight and activation tiles are staged by TMA (128-byte swizzle) through a 4-stage mbarrier
// pipeline; one elected thread issues tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in TMEM).
// When the output has too few tiles to fill the GPU the reduction dimension is split across CTAs;
// the last CTA to finish a tile sums the fp32 partials in split order (deterministic, independent
// of which flows are present) and runs the epilogue:
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
  int splits;
  int kb_total;  // k / 64
  int n_tiles;
  float* part;   // [splits][n_tiles][n_pad][128] fp32 partials (splits > 1)
  int32_t* cnt;  // [n_tiles] arrival counters, left at zero
  int32_t* status;
};

__device__ __forceinline__ void set_status(int32_t* st, int code) { atomicCAS(st, 0, code); }

__device__ __forceinline__ float bf2f(const void* p, size_t i) {
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// RoPE of the pair (x at feature f, xp at the partner f ^ 64) for D = 128 (rotate-half).
__device__ __forceinline__ float rope_rot(float x, float xp, int f, float2 cs) {
  return (f < 64) ? (x * cs.x - xp * cs.y) : (x * cs.x + xp * cs.y);
}

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
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] error, [1] last arriver
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
    flags[1] = 0;
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

  // ---- accumulator: TMEM -> registers -> (smem tile | global split partial) ----
  const bool acc_ok = mbar_wait(done, 0);
  tc_fence_after();
  if (!acc_ok) set_status(p.status, DF_ERR_TIMEOUT);
  const int f = threadIdx.x;  // output feature within the tile == TMEM lane
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  float* my_part = (p.splits > 1) ? p.part + ((size_t)split * p.n_tiles + tile) * p.n_pad * kGemmTileN : nullptr;
  for (int c0 = 0; c0 < p.n_pad; c0 += 16) {
    float v[16];
    tmem_ld16(lane_base + (uint32_t)c0, v);
    if (p.splits == 1) {
#pragma unroll
      for (int j = 0; j < 16; ++j) acc_s[(c0 + j) * kGemmTileN + f] = v[j];
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) my_part[(size_t)(c0 + j) * kGemmTileN + f] = v[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, ncols);

  if (p.splits > 1) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const int prev = atomicAdd(&p.cnt[tile], 1);
      flags[1] = (prev == p.splits - 1);
    }
    __syncthreads();
    if (!flags[1]) return;
    __threadfence();
    for (int n = 0; n < p.n_pad; ++n) {
      float s = 0.f;
      for (int sp = 0; sp < p.splits; ++sp)
        s += __ldcg(p.part + (((size_t)sp * p.n_tiles + tile) * p.n_pad + n) * kGemmTileN + f);
      acc_s[n * kGemmTileN + f] = s;
    }
    if (threadIdx.x == 0) p.cnt[tile] = 0;
    __syncthreads();
  }

  // ---- epilogues (thread f owns output feature tile*128 + f; acc_s[n][f] = row n) ----
  const GemmArgs& a = p.a;
  const int m = a.m_p + a.m_a;
  if (EPI == EPI_STORE_F32 || EPI == EPI_STORE_BF16 || EPI == EPI_ADD_F32) {
    const int fg = tile * kGemmTileN + f;
    if (fg < a.n_out) {
      for (int n = 0; n < m; ++n) {
        const float v = acc_s[n * kGemmTileN + f];
        if (EPI == EPI_STORE_F32) reinterpret_cast<float*>(a.y)[(size_t)n * a.ldy + fg] = v;
        if (EPI == EPI_ADD_F32) reinterpret_cast<float*>(a.y)[(size_t)n * a.ldy + fg] += v;
        if (EPI == EPI_STORE_BF16) reinterpret_cast<__nv_bfloat16*>(a.y)[(size_t)n * a.ldy + fg] = __float2bfloat16_rn(v);
      }
    }
  } else if (EPI == EPI_COUPLE_ADD) {
    const int fg = tile * kGemmTileN + f;
    if (fg < a.n_out) {
      float* y = reinterpret_cast<float*>(a.y);
      const float c = bf2f(a.vec, fg);
      for (int b = 0; b < a.m_p; ++b) {
        const float z1 = acc_s[b * kGemmTileN + f];
        y[(size_t)b * a.ldy + fg] += z1;
        if (a.m_a > 0) {
          const float z2 = acc_s[(a.m_p + b) * kGemmTileN + f] + c * z1;
          y[(size_t)(a.m_p + b) * a.ldy + fg] += z2;
        }
      }
    }
  } else if (EPI == EPI_SWIGLU) {
    if (f < 64) {
      const int j = tile * 64 + f;  // hidden unit
      __nv_bfloat16* u = reinterpret_cast<__nv_bfloat16*>(a.y);
      const float bc = bf2f(a.vec, j);
      for (int b = 0; b < a.m_p; ++b) {
        const float u1 = silu(acc_s[b * kGemmTileN + f]) * acc_s[b * kGemmTileN + f + 64];
        u[(size_t)b * a.ldy + j] = __float2bfloat16_rn(u1);
        if (a.m_a > 0) {
          const int r = a.m_p + b;
          const float u2 = silu(acc_s[r * kGemmTileN + f]) * acc_s[r * kGemmTileN + f + 64] + bc * u1;
          u[(size_t)r * a.ldy + j] = __float2bfloat16_rn(u2);
        }
      }
    }
  } else if (EPI == EPI_QKV) {
    const int Hq = a.n_q_heads, Hkv = a.n_kv_heads, B = a.m_p;
    const int fp = f ^ 64;
    __nv_bfloat16* qo = reinterpret_cast<__nv_bfloat16*>(a.q_out);
    if (tile < Hq) {
      const int h = tile;
      const float af = bf2f(a.vec, h * kHeadDim + f), afp = bf2f(a.vec, h * kHeadDim + fp);
      for (int b = 0; b < B; ++b) {
        const int pos = a.seq_len[b];
        if (pos < 0 || pos > a.max_ctx) {
          set_status(p.status, DF_ERR_DEVICE_BOUNDS);
          continue;
        }
        const float2 cs = a.rope[(size_t)pos * 64 + (f & 63)];
        const float x1 = acc_s[b * kGemmTileN + f], x1p = acc_s[b * kGemmTileN + fp];
        qo[(((size_t)0 * B + b) * Hq + h) * kHeadDim + f] = __float2bfloat16_rn(rope_rot(x1, x1p, f, cs));
        if (a.m_a > 0) {
          const float x2 = acc_s[(B + b) * kGemmTileN + f] + af * x1;
          const float x2p = acc_s[(B + b) * kGemmTileN + fp] + afp * x1p;
          qo[(((size_t)1 * B + b) * Hq + h) * kHeadDim + f] = __float2bfloat16_rn(rope_rot(x2, x2p, f, cs));
        }
      }
    } else {
      const bool is_k = tile < Hq + Hkv;
      const int hk = is_k ? tile - Hq : tile - Hq - Hkv;
      __nv_bfloat16* cache = reinterpret_cast<__nv_bfloat16*>(is_k ? a.k_cache : a.v_cache);
      for (int b = 0; b < B; ++b) {
        const int pos = a.seq_len[b];
        bool ok;
        const size_t off = cache_slot(a, b, hk, pos, p.status, &ok);
        if (!ok) continue;
        float v = acc_s[b * kGemmTileN + f];
        if (is_k) v = rope_rot(v, acc_s[b * kGemmTileN + fp], f, a.rope[(size_t)pos * 64 + (f & 63)]);
        cache[off + f] = __float2bfloat16_rn(v);
      }
    }
  } else if (EPI == EPI_Q2) {
    const int Hq = a.n_q_heads, B = a.m_a;
    const int h = tile, fp = f ^ 64;
    __nv_bfloat16* qo = reinterpret_cast<__nv_bfloat16*>(a.q_out);
    const float af = bf2f(a.vec, h * kHeadDim + f), afp = bf2f(a.vec, h * kHeadDim + fp);
    for (int b = 0; b < B; ++b) {
      const int pos = a.seq_len[b];
      if (pos < 0 || pos > a.max_ctx) {
        set_status(p.status, DF_ERR_DEVICE_BOUNDS);
        continue;
      }
      const float2 cs = a.rope[(size_t)pos * 64 + (f & 63)];
      const size_t qi = ((size_t)b * Hq + h) * kHeadDim;
      const float x1 = bf2f(a.q1_in, qi + f), x1p = bf2f(a.q1_in, qi + fp);
      qo[(((size_t)0 * B + b) * Hq + h) * kHeadDim + f] = __float2bfloat16_rn(rope_rot(x1, x1p, f, cs));
      const float x2 = acc_s[b * kGemmTileN + f] + af * x1;
      const float x2p = acc_s[b * kGemmTileN + fp] + afp * x1p;
      qo[(((size_t)1 * B + b) * Hq + h) * kHeadDim + f] = __float2bfloat16_rn(rope_rot(x2, x2p, f, cs));
    }
  }
}

template <int EPI>
int launch_epi(const CUtensorMap& mw, const CUtensorMap& mx, const GemmParams& p, size_t smem, cudaStream_t s) {
  auto kern = gemm_tc_kernel<EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return DF_ERR_CUDA;
  dim3 grid(p.n_tiles, p.splits);
  kern<<<grid, kThreads, smem, s>>>(mw, mx, p);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace

int gemm_tiles(int n_out, int epi) { return epi == EPI_SWIGLU ? n_out / 64 : (n_out + kGemmTileN - 1) / kGemmTileN; }

// Reduction splits: enough CTAs to cover every SM once, never fewer than 2 k-blocks per split.
// Depends only on the weight shape, never on which flows are present.
int gemm_splits(const dualflow_ctx* ctx, int n_out, int k, int epi) {
  const int tiles = gemm_tiles(n_out, epi);
  const int kb = k / kGemmTileK;
  if (tiles >= ctx->num_sms) return 1;
  int s = (ctx->num_sms + tiles - 1) / tiles;
  if (s > kb / 2) s = kb / 2;
  return s < 1 ? 1 : s;
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
  p.part = ctx->gemm_part;
  p.cnt = ctx->gemm_cnt;
  if (p.splits > 1) {
    const size_t need = (size_t)p.splits * p.n_tiles * p.n_pad * kGemmTileN;
    if (need > ctx->gemm_part_floats || p.n_tiles > ctx->gemm_cnt_n) return DF_ERR_SHAPE;
  }
  const uint64_t w_rows = (a.epi == EPI_SWIGLU) ? 2ull * a.n_out : (uint64_t)a.n_out;
  CUtensorMap mw, mx;
  int rc = encode_map_2d_bf16(&mw, a.W, (uint64_t)a.k, w_rows, (uint64_t)a.k * 2, kGemmTileK, 64);
  if (rc != DF_OK) return rc;
  rc = encode_map_2d_bf16(&mx, a.x, (uint64_t)a.k, (uint64_t)m, (uint64_t)a.k * 2, kGemmTileK, (uint32_t)p.n_pad);
  if (rc != DF_OK) return rc;
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
