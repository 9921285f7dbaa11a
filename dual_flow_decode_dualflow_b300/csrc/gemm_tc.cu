// Stacked-activation linear layers on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// One CTA computes a 128-output-feature tile of y = x . W^T for ALL activation rows of both flows
// (primary rows then auxiliary rows, <= 256): the weight tile is the M = 128 operand, the stacked
// activations are the N operand, so every weight byte is streamed from HBM once and serves both
// flows ("Custos de Inferencia vs. Treinamento": grouping keeps the unique weights read unchanged).
// Weight and activation tiles are staged by TMA (128-byte swizzle) through a mbarrier pipeline of
// up to 4 stages (as many as fit 96 KB, so that two CTAs share an SM); one elected thread issues
// tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in TMEM). Under programmatic dependent launch
// the weight tiles of the first stages are requested before the kernel waits for its predecessor
// (weights never depend on it, activations do), and the producer warms L2 with the first k-blocks
// of the NEXT projection's weights once its own loads are issued.
//
// When the output has too few tiles to fill the GPU the reduction dimension is split across the S
// CTAs of a thread-block cluster (S <= 8). Every CTA owns a 1/S slice of the tile's features --
// feature i and its RoPE / gate-up partner i + 64 travel together, four at a time. Each CTA writes
// its fp32 partial tile from TMEM to a small exchange area that stays in L2, already cut into the S
// owners' slices; after a cluster barrier (release / acquire, which orders those global stores
// for the cluster) the owner of a slice reads its S partials back from L2 with every rank's load
// in flight at once, sums them in rank order (deterministic, and independent of which flows are
// present) and runs the epilogue on its slice:
//   EPI_QKV      q1 = Wq.x1, q2 = Wq.x2 + a (*) q1 (before RoPE), RoPE(q1, q2, k1) at position
//                seq_len[b], q stored bf16, primary k1/v1 appended to the cache at slot seq_len[b]
//                ("Atencao de KV Compartilhada Assimetrica": the auxiliary flow writes no K/V)
//   EPI_Q2       attention-only call: q2 = Wq.h2 + a (*) q1, RoPE(q1), RoPE(q2)
//   EPI_SWIGLU   u = silu(gate) (*) up for both flows, then u2 += b (*) u1 ("Acoplamento Leve")
//   EPI_COUPLE_ADD  y2 += c (*) y1, then h += y (MLP output coupling and residual)
//   EPI_ADD_F32 / EPI_STORE_F32 / EPI_STORE_BF16  residual update, logits, plain stores
//   EPI_MOE_GATEUP / EPI_MOE_DOWN  one expert per grid.z: SWIGLU (with b where both flows chose the
//                expert) or a plain fp32 store, for the rows whose routing selected that expert
//                (the epilogue walks a compact list of those rows)
// The epilogue operands that do not depend on the accumulator (residual rows, the next norm's gain,
// coupling vectors, rotary angles) are loaded while the MMAs run, one or two units per thread.
//
// RMSNorm across kernels (decode step). RMSNorm(h) . W^T = (1/rms(h)) ((h (*) g) . W^T): a residual
// epilogue that has just produced h also writes x_next = bf16(h (*) g_next) and, per row, the sum
// of h^2 over its 128-feature tile; the kernel that consumes x_next multiplies each accumulated
// row by 1 / sqrt(sum / d + eps). No separate normalisation pass over h is needed.
#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

constexpr int kStages = 6;                 // most pipeline stages (barrier arrays are sized for it)
constexpr int kStageBudget = 96 * 1024;    // stage bytes that still let two CTAs share an SM
constexpr int kSharedStages = 4;           // most stages of a launch that shares SMs (two or more CTAs)
constexpr int kQkvSplits = 4;              // most split-K ranks of the QKV projection
constexpr int kQkvStages = 6;              // its pipeline stages (one CTA per SM)
constexpr int kStageBudget3 = 68 * 1024;   // ... three CTAs
constexpr int kRowGroup = 8;               // row blocks per L2-resident group (row-blocked launches)
constexpr int kThreads = 128;
constexpr int kABytes = kGemmTileN * kGemmTileK * 2;  // 16 KB weight tile per stage
constexpr int kSplitMaxRows = 208;                    // most padded activation rows of a split launch

struct GemmParams {
  GemmArgs a;
  int n_pad;     // activation rows padded to a multiple of 16 (the MMA's N)
  int splits;    // CTAs of the cluster sharing one tile's reduction (1, 2, 4 or 8)
  int kb_total;  // k / 64
  int n_tiles;
  int vec_ok;    // y / u rows allow 16-byte (fp32) or 8-byte (bf16) vector access
  int stages;    // pipeline stages in use (2..kStages)
  int region;    // bytes of the data region (pipeline stages, later the partial tiles)
  int row_blocks;  // > 1: grid y runs over blocks of 256 activation rows (splits == 1)
  float* part;     // S > 1: the split-K exchange area, [CTA of the launch][S slices][n_pad][2 nl]
  int chunk;       // S == 1: accumulator rows drained to shared memory per epilogue pass
  int32_t* status;
  unsigned long long wait_ns;  // limit of the pipeline's bounded waits
};

__device__ __forceinline__ void set_status(int32_t* st, int code) { atomicCAS(st, 0, code); }

// silu with the fast exponential and division intrinsics (a few ulp in fp32, far below the bf16
// rounding of the result; the accurate forms made the prefill gate/up epilogue ALU-latency-bound)
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ float4 ld_bf16x4(const void* p, size_t i) {
  const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p) + i);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st_bf16x4(void* p, size_t i, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p) + i) = u;
}
// Element-wise helpers with explicit rounding (no contraction across them): a primary row and an
// auxiliary row with equal inputs get bit-equal results whatever code surrounds them.
__device__ __forceinline__ float4 f4_add(float4 a, float4 b) {
  return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}
__device__ __forceinline__ float4 f4_mul(float4 a, float4 b) {
  return make_float4(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y), __fmul_rn(a.z, b.z), __fmul_rn(a.w, b.w));
}
__device__ __forceinline__ float4 f4_scale(float4 a, float s) {
  return make_float4(__fmul_rn(a.x, s), __fmul_rn(a.y, s), __fmul_rn(a.z, s), __fmul_rn(a.w, s));
}
__device__ __forceinline__ float4 f4_fma(float4 a, float4 b, float4 c) {  // a * b + c, one rounding
  return make_float4(__fmaf_rn(a.x, b.x, c.x), __fmaf_rn(a.y, b.y, c.y), __fmaf_rn(a.z, b.z, c.z),
                     __fmaf_rn(a.w, b.w, c.w));
}
// acc + a.x^2 + a.y^2 + a.z^2 + a.w^2, accumulated in that order
__device__ __forceinline__ float f4_sumsq_acc(float acc, float4 a) {
  return __fmaf_rn(a.w, a.w, __fmaf_rn(a.z, a.z, __fmaf_rn(a.y, a.y, __fmaf_rn(a.x, a.x, acc))));
}
__device__ __forceinline__ float4 f4_silu_mul(float4 g, float4 u) {
  return make_float4(__fmul_rn(silu(g.x), u.x), __fmul_rn(silu(g.y), u.y), __fmul_rn(silu(g.z), u.z),
                     __fmul_rn(silu(g.w), u.w));
}
__device__ __forceinline__ float f4_get(const float4& v, int j) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; }

// Rotary pair (x at feature i, xp at i + 64) by the angles of features i..i+3 at one position:
// lo = x cos - xp sin, hi = xp cos + x sin (each with one final rounding of a fused product).
__device__ __forceinline__ float rot_lo(float x, float xp, float c, float s) { return __fmaf_rn(x, c, -__fmul_rn(xp, s)); }
__device__ __forceinline__ float rot_hi(float x, float xp, float c, float s) { return __fmaf_rn(xp, c, __fmul_rn(x, s)); }
__device__ __forceinline__ void rope4(const float2* cs, float4 x, float4 xp, float4& lo, float4& hi) {
  const float4 c0 = *reinterpret_cast<const float4*>(cs), c1 = *reinterpret_cast<const float4*>(cs + 2);
  // c0 = (cos0, sin0, cos1, sin1), c1 = (cos2, sin2, cos3, sin3)
  lo = make_float4(rot_lo(x.x, xp.x, c0.x, c0.y), rot_lo(x.y, xp.y, c0.z, c0.w), rot_lo(x.z, xp.z, c1.x, c1.y),
                   rot_lo(x.w, xp.w, c1.z, c1.w));
  hi = make_float4(rot_hi(x.x, xp.x, c0.x, c0.y), rot_hi(x.y, xp.y, c0.z, c0.w), rot_hi(x.z, xp.z, c1.x, c1.y),
                   rot_hi(x.w, xp.w, c1.z, c1.w));
}

// Epilogue operands of one (row, quad) unit loaded before the accumulator is ready (see the kernel).
struct EpiPre {
  float4 y1[2], y2[2], c[2], g[2];  // residual rows / rotary angles (QKV: y1 = cos/sin pairs), coupling, gain
  int pos;                          // QKV: the row's position
};

__device__ __forceinline__ void rope4_pre(float4 c0, float4 c1, float4 x, float4 xp, float4& lo, float4& hi) {
  lo = make_float4(rot_lo(x.x, xp.x, c0.x, c0.y), rot_lo(x.y, xp.y, c0.z, c0.w), rot_lo(x.z, xp.z, c1.x, c1.y),
                   rot_lo(x.w, xp.w, c1.z, c1.w));
  hi = make_float4(rot_hi(x.x, xp.x, c0.x, c0.y), rot_hi(x.y, xp.y, c0.z, c0.w), rot_hi(x.z, xp.z, c1.x, c1.y),
                   rot_hi(x.w, xp.w, c1.z, c1.w));
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

// Where a CTA finds the fp32 partial tiles of its output slice. S == 1: its own accumulator tile
// acc[n][128] in shared memory. S > 1: rank k's partial of the slice at g + k * gstride in the
// exchange area, [n][2nl] with local feature fl < nl the tile feature lo0 + fl and fl >= nl its
// partner lo0 + 64 + fl - nl.
struct RedSrc {
  const float* base;
  const float* g;
  int gstride;
  int S, nl;
};

// Reduced accumulators of activation row n at the slice's quad qd: low features (lo) and their
// partners 64 apart (hi), summed over the S partials in rank order.
__device__ __forceinline__ void reduce_pair(const RedSrc& r, int lo0, int n, int qd, float4& lo, float4& hi) {
  if (r.S == 1) {
    const float* e = r.base + n * kGemmTileN + lo0 + 4 * qd;
    lo = *reinterpret_cast<const float4*>(e);
    hi = *reinterpret_cast<const float4*>(e + 64);
    return;
  }
  {
    const float* e = r.g + n * 2 * r.nl + 4 * qd;
    float4 pl[8], ph[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < r.S) {
        pl[k] = __ldcg(reinterpret_cast<const float4*>(e + k * r.gstride));
        ph[k] = __ldcg(reinterpret_cast<const float4*>(e + k * r.gstride + r.nl));
      }
    lo = pl[0];
    hi = ph[0];
#pragma unroll
    for (int k = 1; k < 8; ++k)
      if (k < r.S) {
        lo = f4_add(lo, pl[k]);
        hi = f4_add(hi, ph[k]);
      }
    return;
  }
}

// Stores four features fg..fg+3 of one output row (vector when the row allows it).
template <int EPI>
__device__ __forceinline__ void store4(const GemmArgs& a, int vec_ok, int n, int fg, float4 v) {
  if (EPI == EPI_STORE_BF16) {
    if (vec_ok && fg + 3 < a.n_out) {
      st_bf16x4(a.y, (size_t)n * a.ldy + fg, v);
    } else {
      for (int j = 0; j < 4; ++j)
        if (fg + j < a.n_out)
          reinterpret_cast<__nv_bfloat16*>(a.y)[(size_t)n * a.ldy + fg + j] = __float2bfloat16_rn(f4_get(v, j));
    }
    return;
  }
  float* y = reinterpret_cast<float*>(a.y) + (size_t)n * a.ldy + fg;
  if (vec_ok && fg + 3 < a.n_out) {
    if (EPI == EPI_ADD_F32) v = f4_add(v, *reinterpret_cast<const float4*>(y));
    *reinterpret_cast<float4*>(y) = v;
  } else {
    for (int j = 0; j < 4; ++j)
      if (fg + j < a.n_out) y[j] = (EPI == EPI_ADD_F32 ? y[j] : 0.f) + f4_get(v, j);
  }
}

// Grouped (expert) launches may run three CTAs per SM (see the stage budgets), the others two.
template <int EPI>
constexpr int min_ctas_per_sm() { return (EPI == EPI_MOE_GATEUP || EPI == EPI_MOE_DOWN) ? 3 : 2; }

// RB: the row-blocked (prefill) instantiation, whose accumulator may be drained in passes; the
// others drain it in one pass, with that loop resolved at compile time. PRE2: the O and QKV
// projections of a batch of 64, whose epilogue has two units per thread, preload both units'
// operands (a separate instantiation: the registers it takes slow the one-unit launches).
template <int EPI, bool RB, bool PRE2 = false>
__global__ void __launch_bounds__(kThreads, min_ctas_per_sm<EPI>())
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                   const __grid_constant__ CUtensorMap map_pf, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int b_bytes = p.n_pad * 128;
  uint8_t* sA = smem;
  const int nst = p.stages;
  uint8_t* sB = smem + nst * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.region);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint64_t* prod_done = done + 1;  // the producer has issued its last load; tmem_slot[2] = how many
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(prod_done + 1);
  float* rstd_s = reinterpret_cast<float*>(tmem_slot + 4);  // [256] 1 / rms of each activation row
  int* sel_s = reinterpret_cast<int*>(rstd_s + kGemmMaxAct);  // [256] grouped: row selected this expert
  // grouped: the rows whose epilogue has work (the expert's rows), in row order; their count is
  // tmem_slot[3]
  int* sel_list = sel_s + kGemmMaxAct;
  // S == 1: after the main loop the pipeline bytes hold the accumulator tile acc[n][128]
  float* acc_s = reinterpret_cast<float*>(smem);

  GemmArgs a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // row-blocked launches: CTAs in launch order sweep groups of kRowGroup row blocks, every tile of a
  // group before the next group, so the weight tiles and row blocks in flight stay L2-resident
  int tile = blockIdx.x, rblk = 0;
  if (p.row_blocks > 1) {
    const int lin = blockIdx.x + gridDim.x * blockIdx.y, per = kRowGroup * gridDim.x;
    const int g0 = (lin / per) * kRowGroup, in_g = min(kRowGroup, p.row_blocks - g0), w_ = lin % per;
    rblk = g0 + w_ % in_g;
    tile = w_ / in_g;
  }
  const int split = p.row_blocks > 1 ? 0 : blockIdx.y;
  int grp = blockIdx.z;
  int rbase = rblk * kGemmMaxAct;  // first activation row of this CTA
  int rows_left = p.a.m_p - rbase;
  if (a.blk_info != nullptr) {
    // gathered expert rows: this row block is one expert's rows (the grid is sized for the most
    // blocks the routing can produce; the ones beyond it leave before any setup)
    if (rblk >= *a.n_blk) return;
    const int4 bi = a.blk_info[rblk];
    grp = bi.x;
    rbase = bi.y;
    rows_left = bi.z;
  }
  if (p.row_blocks > 1) {
    // this CTA's block of rows: the epilogue's row-indexed operands start at its first row
    const size_t ye = (EPI == EPI_STORE_BF16 || EPI == EPI_SWIGLU) ? 2 : 4;
    a.m_p = min(kGemmMaxAct, rows_left);
    a.row_base = rbase;
    if (a.y) a.y = static_cast<uint8_t*>(a.y) + (size_t)rbase * a.ldy * ye;
    if (a.x_next) a.x_next = static_cast<__nv_bfloat16*>(a.x_next) + (size_t)rbase * a.n_out;
    if (a.ss_out) a.ss_out += (size_t)rbase * a.ss_ld;
    if (a.ss_in) a.ss_in += (size_t)rbase * a.ss_ld;
  }
  const int kb0 = (int)((long long)split * p.kb_total / p.splits);
  const int kb1 = (int)((long long)(split + 1) * p.kb_total / p.splits);
  const int nkb = kb1 - kb0;
  const int m = a.m_p + a.m_a;
  uint32_t ncols = 32;
  while ((int)ncols < p.n_pad) ncols <<= 1;
  const int S = p.splits;
  const int nl = 64 / S, lo0 = split * nl, nq = nl / 4, nfs = 2 * nl;
  // S > 1: the tile's S partials sit side by side in the exchange area, each cut into S slices
  // [n_pad][2nl] (slice r is read by rank r)
  const size_t cta_floats = (size_t)kGemmTileN * p.n_pad;
  const size_t tile_cta0 = ((size_t)grp * p.n_tiles + tile) * S;  // the tile's rank-0 CTA
  const size_t slice_off = (size_t)split * p.n_pad * nfs;         // this CTA's slice in a partial

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    mbar_init(prod_done, 1);
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
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;

  int row0, row1;
  if (EPI == EPI_SWIGLU || EPI == EPI_MOE_GATEUP) {
    row0 = 64 * tile;                 // gate rows of hidden units [64 tile, 64 tile + 64)
    row1 = a.n_out + 64 * tile;       // up rows of the same units
  } else {
    row0 = kGemmTileN * tile;
    row1 = row0 + 64;
  }
  row0 += grp * a.w_group_rows;       // this expert's weights (grouped launch)
  row1 += grp * a.w_group_rows;
  const int xrow = grp * a.x_group_rows + rbase;

  if (warp == 0 && lane == 0) {
    // TMA producer: weights are streamed once (evict-first), activations stay L2-resident.
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    const int npre = nkb < nst ? nkb : nst;
    // weights of the first stages do not depend on the preceding kernel: request them first
    for (int i = 0; i < npre; ++i) {
      mbar_arrive_expect_tx(&full[i], (uint32_t)(kABytes + b_bytes));
      const int kc = (kb0 + i) * kGemmTileK;
      tma_load_2d_hint(sA + i * kABytes, &map_w, &full[i], kc, row0, pol_w);
      tma_load_2d_hint(sA + i * kABytes + kABytes / 2, &map_w, &full[i], kc, row1, pol_w);
    }
    griddep_wait();
    for (int i = 0; i < npre; ++i)
      tma_load_2d_hint(sB + i * b_bytes, &map_x, &full[i], (kb0 + i) * kGemmTileK, xrow, pol_x);
    int issued = npre;
    for (int i = npre; i < nkb; ++i) {
      const int s = i % nst;
      const uint32_t ph = (uint32_t)(i / nst) & 1u;
      if (!mbar_wait(&empty[s], ph ^ 1u, p.wait_ns)) {
        set_status(p.status, DF_ERR_TIMEOUT);
        break;
      }
      mbar_arrive_expect_tx(&full[s], (uint32_t)(kABytes + b_bytes));
      const int kc = (kb0 + i) * kGemmTileK;
      tma_load_2d_hint(sA + s * kABytes, &map_w, &full[s], kc, row0, pol_w);
      tma_load_2d_hint(sA + s * kABytes + kABytes / 2, &map_w, &full[s], kc, row1, pol_w);
      tma_load_2d_hint(sB + s * b_bytes, &map_x, &full[s], kc, xrow, pol_x);
      ++issued;
    }
    if (a.pf_W != nullptr && a.pf_depth > 0) {
      // every tile of this launch is requested: warm L2 with the next launch's first k-blocks
      const int ncur = gridDim.x * gridDim.y * gridDim.z;
      const int cid = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
      const int nnext = a.pf_tiles * a.pf_splits, kbn = a.pf_k / kGemmTileK;
      for (int q = (int)((long long)cid * nnext / ncur); q < (int)((long long)(cid + 1) * nnext / ncur); ++q) {
        const int t = q / a.pf_splits, sp = q % a.pf_splits;
        const int k0 = (int)((long long)sp * kbn / a.pf_splits), k1 = (int)((long long)(sp + 1) * kbn / a.pf_splits);
        const int r0 = t * a.pf_tile_rows;
        for (int kb = k0; kb < k1 && kb < k0 + a.pf_depth; ++kb) {
          tma_prefetch_l2_2d(&map_pf, kb * kGemmTileK, r0);
          tma_prefetch_l2_2d(&map_pf, kb * kGemmTileK, r0 + a.pf_half);
        }
      }
    }
    // how many iterations were issued, for the MMA thread's drain after a wait that gave up
    tmem_slot[2] = (uint32_t)issued;
    mbar_arrive(prod_done);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: 4 x (M=128, N=n_pad, K=16) per stage, accumulate in TMEM.
    const uint32_t idesc = idesc_bf16_f32(kGemmTileN, p.n_pad);
    int failed = -1;  // the iteration whose wait gave up
    for (int i = 0; i < nkb; ++i) {
      const int s = i % nst;
      const uint32_t ph = (uint32_t)(i / nst) & 1u;
      if (!mbar_wait(&full[s], ph, p.wait_ns)) {
        set_status(p.status, DF_ERR_TIMEOUT);
        failed = i;
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
    if (failed >= 0) {
      // Every load the producer issued lands before the stages are reused for the accumulator tile
      // or the CTA exits: once it has stopped issuing (its own waits are bounded too), wait for the
      // iterations it issued that this thread did not consume. Only after a wait gave up; a normal
      // main loop has consumed them all.
      if (mbar_wait(prod_done, 0)) {
        const int issued = (int)tmem_slot[2];
        for (int j = failed; j < issued; ++j)
          if (!mbar_wait(&full[j % nst], (uint32_t)(j / nst) & 1u)) break;
      }
    }
    umma_commit(done);
  } else if (warp >= 2 && (a.ss_in != nullptr || a.sel_pos != nullptr || EPI == EPI_PREFILL_QKV)) {
    // idle during the main loop: which rows selected this launch's expert (grouped launches) and
    // 1 / rms of every activation row, from the producer's partials
    griddep_wait();
    if (EPI == EPI_PREFILL_QKV) {
      // every row's cache slot and position (prompt token t of prompt sequence i is activation row
      // i * seq_rows + t, held by cache slot b = slots[i], at position seq_len[b] + t): the
      // epilogue's units then start from shared memory instead of two dependent global loads
      for (int n = threadIdx.x - 64; n < m; n += 64) {
        const int grow = a.row_base + n, si = grow / a.seq_rows, b = a.slots ? a.slots[si] : si;
        const bool slot_ok = b >= 0 && b < a.max_batch;
        sel_list[n] = b;
        sel_s[n] = slot_ok ? a.seq_len[b] + grow % a.seq_rows : -1;
      }
    }
    if (a.sel_pos != nullptr) {
      for (int n = threadIdx.x - 64; n < m; n += 64) sel_s[n] = a.sel_pos[(size_t)n * a.n_groups + grp] >= 0;
      if (warp == 2) {
        // the epilogue's rows: gate/up pairs primary row n with auxiliary row m_p + n and has work
        // when either selected the expert; down has one unit row per activation row
        const int nr = EPI == EPI_MOE_GATEUP ? a.m_p : m;
        int cnt = 0;
        for (int b0 = 0; b0 < nr; b0 += 32) {
          const int n = b0 + lane;
          bool s = false;
          if (n < nr) {
            s = a.sel_pos[(size_t)n * a.n_groups + grp] >= 0;
            if (EPI == EPI_MOE_GATEUP && a.m_a > 0) s = s || a.sel_pos[(size_t)(a.m_p + n) * a.n_groups + grp] >= 0;
          }
          const unsigned bal = __ballot_sync(0xffffffffu, s);
          if (s) sel_list[cnt + __popc(bal & ((1u << lane) - 1u))] = n;
          cnt += __popc(bal);
        }
        if (lane == 0) tmem_slot[3] = (uint32_t)cnt;
      }
    }
    for (int n = threadIdx.x - 64; a.ss_in != nullptr && n < m; n += 64) {
      const float* row = a.ss_in + (size_t)n * a.ss_ld;
      float ss = 0.f;
      int q = 0;
      // up to 16 vector loads in flight, summed in partial order afterwards
      if ((a.ss_ld & 3) == 0)
        while (q + 4 <= a.ss_parts) {
          float4 v[16];
          const int nv = min(16, (a.ss_parts - q) / 4);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < nv) v[j] = *reinterpret_cast<const float4*>(row + q + 4 * j);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < nv) {
              ss += v[j].x;
              ss += v[j].y;
              ss += v[j].z;
              ss += v[j].w;
            }
          q += 4 * nv;
        }
      for (; q < a.ss_parts; ++q) ss += row[q];
      rstd_s[n] = 1.0f / sqrtf(ss * a.inv_d + a.eps);
    }
  }
  __syncwarp();

  const bool scaled = a.ss_in != nullptr;
  const bool norm_out = (EPI == EPI_ADD_F32 || EPI == EPI_COUPLE_ADD) && a.g_next != nullptr;
  // units of work: (activation row, quad); paired epilogues take the primary row and its auxiliary row
  const bool paired = EPI == EPI_COUPLE_ADD || EPI == EPI_SWIGLU || EPI == EPI_QKV || EPI == EPI_MOE_GATEUP;
  const int rows = (EPI == EPI_Q2) ? a.m_a : paired ? a.m_p : m;

  // ---- epilogue operands that do not depend on the accumulator ----
  // When every thread has at most one (row, quad) unit (the decode launches), its operands -- residual
  // rows, the next norm's gain, the coupling vector, the rotary angles -- are final once the preceding
  // kernel has completed, so they are loaded now, while the MMAs finish, instead of after the split-K
  // exchange; the epilogue then waits for the partials alone.
  EpiPre pre[2];
  constexpr int pre_units = (PRE2 && (EPI == EPI_ADD_F32 || EPI == EPI_QKV)) ? 2 : 1;
  const bool pre_ok = !RB && rows * nq <= pre_units * kThreads &&
                      (EPI == EPI_ADD_F32 || EPI == EPI_COUPLE_ADD || EPI == EPI_SWIGLU || EPI == EPI_QKV ||
                       EPI == EPI_Q2);
  if (pre_ok && (int)threadIdx.x < rows * nq) griddep_wait();  // the operands were written by preceding kernels
#pragma unroll
  for (int u = 0; u < pre_units; ++u) {
    const int it = u * kThreads + threadIdx.x;
    if (!pre_ok || it >= rows * nq) continue;
    EpiPre& pre_w = pre[u];
    const int n = it / nq, qd = it % nq;
    const int fa = lo0 + 4 * qd, fg = tile * kGemmTileN + fa;
    if (EPI == EPI_ADD_F32 && norm_out) {
      const float* y = reinterpret_cast<const float*>(a.y) + (size_t)n * a.ldy;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        if (fg + 64 * hh < a.n_out) {
          pre_w.y1[hh] = *reinterpret_cast<const float4*>(y + fg + 64 * hh);
          pre_w.g[hh] = ld_bf16x4(a.g_next, fg + 64 * hh);
        }
    } else if (EPI == EPI_COUPLE_ADD) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int f = fg + 64 * hh;
        if (p.vec_ok && f + 3 < a.n_out) {
          pre_w.y1[hh] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.y) + (size_t)n * a.ldy + f);
          if (a.m_a > 0) {
            pre_w.y2[hh] =
                *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.y) + (size_t)(a.m_p + n) * a.ldy + f);
            pre_w.c[hh] = ld_bf16x4(a.vec, f);
          }
          if (norm_out) pre_w.g[hh] = ld_bf16x4(a.g_next, f);
        }
      }
    } else if (EPI == EPI_SWIGLU) {
      if (a.m_a > 0) pre_w.c[0] = ld_bf16x4(a.vec, tile * 64 + fa);
    } else if (EPI == EPI_QKV) {
      const int pos = a.seq_len[n];
      pre_w.pos = pos;
      if (pos >= 0 && pos <= a.max_ctx) {
        const float2* cs = a.rope + (size_t)pos * 64 + fa;
        pre_w.y1[0] = *reinterpret_cast<const float4*>(cs);
        pre_w.y1[1] = *reinterpret_cast<const float4*>(cs + 2);
      }
      if (tile < a.n_q_heads && a.m_a > 0) {
        pre_w.c[0] = ld_bf16x4(a.vec, tile * kHeadDim + fa);
        pre_w.c[1] = ld_bf16x4(a.vec, tile * kHeadDim + fa + 64);
      }
    } else if (EPI == EPI_Q2) {
      // the attention-only call: row n is sequence n's auxiliary query, tile = query head
      const int pos = a.seq_len[n];
      pre_w.pos = pos;
      if (pos >= 0 && pos <= a.max_ctx) {
        const float2* cs = a.rope + (size_t)pos * 64 + fa;
        pre_w.y1[0] = *reinterpret_cast<const float4*>(cs);
        pre_w.y1[1] = *reinterpret_cast<const float4*>(cs + 2);
      }
      const size_t qi = ((size_t)n * a.n_q_heads + tile) * kHeadDim;
      pre_w.y2[0] = ld_bf16x4(a.q1_in, qi + fa);
      pre_w.y2[1] = ld_bf16x4(a.q1_in, qi + fa + 64);
      pre_w.c[0] = ld_bf16x4(a.vec, tile * kHeadDim + fa);
      pre_w.c[1] = ld_bf16x4(a.vec, tile * kHeadDim + fa + 64);
    }
  }

  // ---- accumulator: TMEM -> registers -> shared memory (S == 1) or the exchange area ----
  const bool acc_ok = mbar_wait(done, 0);
  tc_fence_after();
  if (!acc_ok) set_status(p.status, DF_ERR_TIMEOUT);
  const int tf = threadIdx.x;  // TMEM lane == output feature within the tile
  const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
  const int hf = tf & 63, dst_rank = hf / nl;  // split-K: the rank that owns feature tf
  const int fl = (tf >> 6) * nl + hf % nl;     // and its index there
  float* dst = acc_s + tf;  // S == 1: acc[n][128 - row offset of the pass]
  float* gdst = S > 1 ? p.part + (tile_cta0 + split) * cta_floats + (size_t)dst_rank * p.n_pad * nfs + fl : nullptr;
  RedSrc red;
  red.base = acc_s;
  red.g = S > 1 ? p.part + tile_cta0 * cta_floats + slice_off : nullptr;
  red.gstride = (int)cta_floats;
  red.S = S;
  red.nl = nl;
  // S == 1 with a tile larger than the pipeline bytes (row-blocked launches on a small budget): the
  // accumulator is drained and its epilogue run in passes of `chunk` rows (no auxiliary rows there)
  const int chunk = (RB && S == 1 && p.chunk > 0) ? p.chunk : p.n_pad;
  const int n_pass = RB ? (p.n_pad + chunk - 1) / chunk : 1;
  for (int pass = 0; pass < n_pass; ++pass) {
  const int cb = RB ? pass * chunk : 0;
  // four 16-column TMEM loads in flight per wait
  for (int c0 = cb; c0 < cb + chunk && c0 < p.n_pad; c0 += 64) {
    uint32_t v[4][16];
    const int nblk = (p.n_pad - c0) >= 64 ? 4 : (p.n_pad - c0) / 16;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (q < nblk) tmem_ld16_nowait(lane_base + (uint32_t)(c0 + 16 * q), v[q]);
    tmem_ld_wait();
    if (S > 1) {
      // feature tf's column into its owner's slice of this CTA's partial (cached in L2 only)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < nblk)
#pragma unroll
          for (int j = 0; j < 16; ++j) __stcg(gdst + (size_t)(c0 + 16 * q + j) * nfs, __uint_as_float(v[q][j]));
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < nblk)
#pragma unroll
          for (int j = 0; j < 16; ++j) dst[(c0 - cb + 16 * q + j) * kGemmTileN] = __uint_as_float(v[q][j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (cb + chunk >= p.n_pad && warp == 1) tmem_dealloc(tmem, ncols);
  if (cb == 0) {
    griddep_wait();  // the epilogue reads and writes buffers of the preceding kernels
    if (S > 1) {
      cluster_arrive();  // this CTA's partial is written (release: its global stores included)
      cluster_wait();    // and so are the other ranks'
    }
  }
  red.base = acc_s - (size_t)cb * kGemmTileN;  // row n of this pass at acc_s[(n - cb) * 128]
  const int r_end = min(cb + chunk, rows);
  int units = r_end > cb ? (r_end - cb) * nq : 0;
  // grouped expert launches (one pass, no split): only the rows that selected the expert
  constexpr bool kListed = EPI == EPI_MOE_GATEUP || EPI == EPI_MOE_DOWN;
  const bool listed = kListed && !RB && S == 1 && a.sel_pos != nullptr;
  if (listed) units = (int)tmem_slot[3] * nq;
  if (EPI == EPI_SWIGLU && !RB && S > 1 && units <= 2 * kThreads) {
    // gate/up of a split launch with up to two units per thread: every partial load of both units,
    // and the coupling vector b, is issued before any of their arithmetic, so the exchange costs
    // one round trip to L2
    float4 lo[2], hi[2], g2[2], p2[2], bv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int it = u * kThreads + threadIdx.x, n = it / nq, qd = it % nq;
      if (it < units) {
        reduce_pair(red, lo0, n, qd, lo[u], hi[u]);
        if (a.m_a > 0) {
          reduce_pair(red, lo0, a.m_p + n, qd, g2[u], p2[u]);
          bv[u] = ld_bf16x4(a.vec, tile * 64 + lo0 + 4 * qd);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int it = u * kThreads + threadIdx.x, n = it / nq, qd = it % nq;
      if (it >= units) continue;
      const int j = tile * 64 + lo0 + 4 * qd;  // hidden unit: gate at tile feature fa, up at fa + 64
      if (scaled) {
        lo[u] = f4_scale(lo[u], rstd_s[n]);
        hi[u] = f4_scale(hi[u], rstd_s[n]);
      }
      const float4 u1 = f4_silu_mul(lo[u], hi[u]);
      st_bf16x4(a.y, (size_t)n * a.ldy + j, u1);
      if (a.m_a > 0) {
        if (scaled) {
          g2[u] = f4_scale(g2[u], rstd_s[a.m_p + n]);
          p2[u] = f4_scale(p2[u], rstd_s[a.m_p + n]);
        }
        st_bf16x4(a.y, (size_t)(a.m_p + n) * a.ldy + j, f4_fma(bv[u], u1, f4_silu_mul(g2[u], p2[u])));
      }
    }
    units = 0;  // done: the loop below has nothing left
  }
  // row-blocked residual epilogues (prefill): every thread walks many units whose residual rows
  // come from HBM; L2 is asked for them kRbAhead iterations ahead, so that a unit's loads hit L2
  constexpr int kRbAhead = 4;
  constexpr bool kRbResidual = RB && (EPI == EPI_ADD_F32 || EPI == EPI_COUPLE_ADD);
  auto rb_prefetch = [&](int itp) {
    if (itp >= units) return;
    const int np = cb + itp / nq, fp = tile * kGemmTileN + lo0 + 4 * (itp % nq);
    const float* yp = reinterpret_cast<const float*>(a.y) + (size_t)np * a.ldy + fp;
    if (fp < a.n_out) prefetch_l2(yp);
    if (fp + 64 < a.n_out) prefetch_l2(yp + 64);
  };
  // and each unit's residual rows are in registers one iteration before they are used
  float4 ynx[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  auto rb_load = [&](int itn) {
    if (itn >= units) return;
    const int nn = cb + itn / nq, fn = tile * kGemmTileN + lo0 + 4 * (itn % nq);
    const float* yp = reinterpret_cast<const float*>(a.y) + (size_t)nn * a.ldy + fn;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      if (fn + 64 * hh < a.n_out) ynx[hh] = *reinterpret_cast<const float4*>(yp + 64 * hh);
  };
  if constexpr (kRbResidual) {
    for (int j = 0; j < kRbAhead; ++j) rb_prefetch(j * kThreads + threadIdx.x);
    rb_load(threadIdx.x);
  }
  for (int base = 0; base < units; base += kThreads) {
    const int it = base + threadIdx.x;
    float4 ycur[2] = {ynx[0], ynx[1]};
    if constexpr (kRbResidual) {
      rb_prefetch(it + kRbAhead * kThreads);
      rb_load(it + kThreads);
    }
    // this iteration's preloaded operands (with two units, a select, so that both stay in registers)
    EpiPre pu_sel;
    if constexpr (pre_units > 1) pu_sel = base != 0 ? pre[1] : pre[0];
    const EpiPre& pu = pre_units > 1 ? pu_sel : pre[0];
    const bool live = it < units;
    const int n = live ? (listed ? sel_list[it / nq] : cb + it / nq) : 0, qd = it % nq;
    const int fa = lo0 + 4 * qd;        // tile feature of the low quad
    const int fg = tile * kGemmTileN + fa;
    float ss0 = 0.f, ss1 = 0.f;         // norm outputs: sum of h^2 of row n (and its auxiliary row)
    if (live) {
      float4 lo, hi;
      reduce_pair(red, lo0, n, qd, lo, hi);
      if (scaled) {
        const float r = rstd_s[n];
        lo = f4_scale(lo, r);
        hi = f4_scale(hi, r);
      }
      if (EPI == EPI_STORE_F32 || EPI == EPI_STORE_BF16 || (EPI == EPI_ADD_F32 && !norm_out)) {
        store4<EPI>(a, p.vec_ok, n, fg, lo);
        store4<EPI>(a, p.vec_ok, n, fg + 64, hi);
      } else if (EPI == EPI_ADD_F32) {
        // residual update, then the next norm's input (n_out is d, a multiple of 64)
        float* y = reinterpret_cast<float*>(a.y) + (size_t)n * a.ldy;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int f = fg + 64 * hh;
          if (f >= a.n_out) continue;
          const float4 hv = f4_add(kRbResidual ? ycur[hh] : pre_ok ? pu.y1[hh] : *reinterpret_cast<const float4*>(y + f),
                                   hh ? hi : lo);
          *reinterpret_cast<float4*>(y + f) = hv;
          st_bf16x4(a.x_next, (size_t)n * a.n_out + f, f4_mul(hv, pre_ok ? pu.g[hh] : ld_bf16x4(a.g_next, f)));
          ss0 = f4_sumsq_acc(ss0, hv);
        }
      } else if (EPI == EPI_COUPLE_ADD) {
        float4 z2lo = make_float4(0.f, 0.f, 0.f, 0.f), z2hi = z2lo;
        if (a.m_a > 0) {
          reduce_pair(red, lo0, a.m_p + n, qd, z2lo, z2hi);
          if (scaled) {
            const float r = rstd_s[a.m_p + n];
            z2lo = f4_scale(z2lo, r);
            z2hi = f4_scale(z2hi, r);
          }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int f = fg + 64 * hh;
          const float4 z1 = hh ? hi : lo;
          const float4 z2 = hh ? z2hi : z2lo;
          if (p.vec_ok && f + 3 < a.n_out) {
            float* y1 = reinterpret_cast<float*>(a.y) + (size_t)n * a.ldy + f;
            const float4 h1 =
                f4_add(kRbResidual ? ycur[hh] : pre_ok ? pu.y1[hh] : *reinterpret_cast<const float4*>(y1), z1);
            *reinterpret_cast<float4*>(y1) = h1;
            float4 h2 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (a.m_a > 0) {
              float* y2 = reinterpret_cast<float*>(a.y) + (size_t)(a.m_p + n) * a.ldy + f;
              h2 = f4_add(pre_ok ? pu.y2[hh] : *reinterpret_cast<const float4*>(y2),
                          f4_fma(pre_ok ? pu.c[hh] : ld_bf16x4(a.vec, f), z1, z2));
              *reinterpret_cast<float4*>(y2) = h2;
            }
            if (norm_out) {
              const float4 g = pre_ok ? pu.g[hh] : ld_bf16x4(a.g_next, f);
              st_bf16x4(a.x_next, (size_t)n * a.n_out + f, f4_mul(h1, g));
              ss0 = f4_sumsq_acc(ss0, h1);
              if (a.m_a > 0) {
                st_bf16x4(a.x_next, (size_t)(a.m_p + n) * a.n_out + f, f4_mul(h2, g));
                ss1 = f4_sumsq_acc(ss1, h2);
              }
            }
          } else {
            for (int j = 0; j < 4; ++j) {
              if (f + j >= a.n_out) continue;
              float* y = reinterpret_cast<float*>(a.y);
              const float z1j = f4_get(z1, j);
              y[(size_t)n * a.ldy + f + j] += z1j;
              if (a.m_a > 0)
                y[(size_t)(a.m_p + n) * a.ldy + f + j] +=
                    f4_get(z2, j) + __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.vec)[f + j]) * z1j;
            }
          }
        }
      } else if (EPI == EPI_MOE_GATEUP) {
        // expert grp: rows that selected it; the auxiliary row couples to the primary row only
        // when the primary selected the same expert
        const int j = tile * 64 + fa;
        __nv_bfloat16* u = reinterpret_cast<__nv_bfloat16*>(a.y) + (size_t)grp * a.y_group_stride;
        const bool s1 = sel_s[n] != 0;
        const bool s2 = a.m_a > 0 && sel_s[a.m_p + n] != 0;
        const float4 u1 = f4_silu_mul(lo, hi);
        if (s1) st_bf16x4(u, (size_t)n * a.ldy + j, u1);
        if (s2) {
          float4 g2, p2;
          reduce_pair(red, lo0, a.m_p + n, qd, g2, p2);
          if (scaled) {
            const float r = rstd_s[a.m_p + n];
            g2 = f4_scale(g2, r);
            p2 = f4_scale(p2, r);
          }
          float4 u2 = f4_silu_mul(g2, p2);
          if (s1) u2 = f4_fma(ld_bf16x4(a.vec, j), u1, u2);
          st_bf16x4(u, (size_t)(a.m_p + n) * a.ldy + j, u2);
        }
      } else if (EPI == EPI_MOE_DOWN) {
        if (sel_s[n] != 0) {
          float* y = reinterpret_cast<float*>(a.y) + (size_t)grp * a.y_group_stride + (size_t)n * a.ldy;
          if (fg < a.n_out) *reinterpret_cast<float4*>(y + fg) = lo;
          if (fg + 64 < a.n_out) *reinterpret_cast<float4*>(y + fg + 64) = hi;
        }
      } else if (EPI == EPI_SWIGLU) {
        const int j = tile * 64 + fa;  // hidden unit: gate at tile feature fa, up at fa + 64
        const float4 u1 = f4_silu_mul(lo, hi);
        st_bf16x4(a.y, (size_t)n * a.ldy + j, u1);
        if (a.m_a > 0) {
          float4 g2, p2;
          reduce_pair(red, lo0, a.m_p + n, qd, g2, p2);
          if (scaled) {
            const float r = rstd_s[a.m_p + n];
            g2 = f4_scale(g2, r);
            p2 = f4_scale(p2, r);
          }
          st_bf16x4(a.y, (size_t)(a.m_p + n) * a.ldy + j,
                    f4_fma(pre_ok ? pu.c[0] : ld_bf16x4(a.vec, j), u1, f4_silu_mul(g2, p2)));
        }
      } else if (EPI == EPI_QKV) {
        const int Hq = a.n_q_heads, Hkv = a.n_kv_heads, B = a.m_p, b = n;
        const int pos = pre_ok ? pu.pos : a.seq_len[b];
        if (pos < 0 || pos > a.max_ctx) {
          set_status(p.status, DF_ERR_DEVICE_BOUNDS);
        } else {
          const float2* cs = a.rope + (size_t)pos * 64 + fa;
          const float4 cs0 = pre_ok ? pu.y1[0] : *reinterpret_cast<const float4*>(cs);
          const float4 cs1 = pre_ok ? pu.y1[1] : *reinterpret_cast<const float4*>(cs + 2);
          float4 r_lo, r_hi;
          if (tile < Hq) {
            const int h = tile;
            rope4_pre(cs0, cs1, lo, hi, r_lo, r_hi);
            const size_t o1 = (((size_t)0 * B + b) * Hq + h) * kHeadDim;
            st_bf16x4(a.q_out, o1 + fa, r_lo);
            st_bf16x4(a.q_out, o1 + fa + 64, r_hi);
            if (a.m_a > 0) {
              float4 x2, x2p;
              reduce_pair(red, lo0, B + b, qd, x2, x2p);
              if (scaled) {
                const float r = rstd_s[B + b];
                x2 = f4_scale(x2, r);
                x2p = f4_scale(x2p, r);
              }
              x2 = f4_fma(pre_ok ? pu.c[0] : ld_bf16x4(a.vec, h * kHeadDim + fa), lo, x2);
              x2p = f4_fma(pre_ok ? pu.c[1] : ld_bf16x4(a.vec, h * kHeadDim + fa + 64), hi, x2p);
              rope4_pre(cs0, cs1, x2, x2p, r_lo, r_hi);
              const size_t o2 = (((size_t)1 * B + b) * Hq + h) * kHeadDim;
              st_bf16x4(a.q_out, o2 + fa, r_lo);
              st_bf16x4(a.q_out, o2 + fa + 64, r_hi);
            }
          } else {
            const bool is_k = tile < Hq + Hkv;
            const int hk = is_k ? tile - Hq : tile - Hq - Hkv;
            bool ok;
            const size_t off = cache_slot(a, b, hk, pos, p.status, &ok);
            if (ok) {
              void* cache = is_k ? a.k_cache : a.v_cache;
              if (is_k) {
                rope4_pre(cs0, cs1, lo, hi, r_lo, r_hi);
              } else {
                r_lo = lo;
                r_hi = hi;
              }
              st_bf16x4(cache, off + fa, r_lo);
              st_bf16x4(cache, off + fa + 64, r_hi);
            }
          }
        }
      } else if (EPI == EPI_PREFILL_QKV) {
        // prompt token t of prompt sequence i (activation row i * seq_rows + t), held by cache slot
        // b = slots[i], at position seq_len[b] + t
        const int Hq = a.n_q_heads, Hkv = a.n_kv_heads, grow = a.row_base + n;
        const int b = sel_list[n], pos = sel_s[n];  // staged by the idle warps (see above)
        if (pos < 0 || pos >= a.max_ctx) {
          set_status(p.status, DF_ERR_DEVICE_BOUNDS);
        } else {
          const float2* cs = a.rope + (size_t)pos * 64 + fa;
          float4 r_lo, r_hi;
          if (tile < Hq) {
            rope4(cs, lo, hi, r_lo, r_hi);
            const size_t o1 = ((size_t)grow * Hq + tile) * kHeadDim;
            st_bf16x4(a.q_out, o1 + fa, r_lo);
            st_bf16x4(a.q_out, o1 + fa + 64, r_hi);
          } else {
            const bool is_k = tile < Hq + Hkv;
            const int hk = is_k ? tile - Hq : tile - Hq - Hkv;
            bool ok;
            const size_t off = cache_slot(a, b, hk, pos, p.status, &ok);
            if (ok) {
              if (is_k) {
                rope4(cs, lo, hi, r_lo, r_hi);
              } else {
                r_lo = lo;
                r_hi = hi;
              }
              st_bf16x4(is_k ? a.k_cache : a.v_cache, off + fa, r_lo);
              st_bf16x4(is_k ? a.k_cache : a.v_cache, off + fa + 64, r_hi);
            }
          }
        }
      } else if (EPI == EPI_Q2) {
        const int Hq = a.n_q_heads, B = a.m_a, h = tile, b = n;
        const int pos = pre_ok ? pu.pos : a.seq_len[b];
        if (pos < 0 || pos > a.max_ctx) {
          set_status(p.status, DF_ERR_DEVICE_BOUNDS);
        } else {
          const float2* cs = a.rope + (size_t)pos * 64 + fa;
          const float4 cs0 = pre_ok ? pu.y1[0] : *reinterpret_cast<const float4*>(cs);
          const float4 cs1 = pre_ok ? pu.y1[1] : *reinterpret_cast<const float4*>(cs + 2);
          const size_t qi = ((size_t)b * Hq + h) * kHeadDim;
          const float4 x1 = pre_ok ? pu.y2[0] : ld_bf16x4(a.q1_in, qi + fa);
          const float4 x1p = pre_ok ? pu.y2[1] : ld_bf16x4(a.q1_in, qi + fa + 64);
          float4 r_lo, r_hi;
          rope4_pre(cs0, cs1, x1, x1p, r_lo, r_hi);
          const size_t o1 = (((size_t)0 * B + b) * Hq + h) * kHeadDim;
          st_bf16x4(a.q_out, o1 + fa, r_lo);
          st_bf16x4(a.q_out, o1 + fa + 64, r_hi);
          const float4 x2 = f4_fma(pre_ok ? pu.c[0] : ld_bf16x4(a.vec, h * kHeadDim + fa), x1, lo);
          const float4 x2p = f4_fma(pre_ok ? pu.c[1] : ld_bf16x4(a.vec, h * kHeadDim + fa + 64), x1p, hi);
          rope4_pre(cs0, cs1, x2, x2p, r_lo, r_hi);
          const size_t o2 = (((size_t)1 * B + b) * Hq + h) * kHeadDim;
          st_bf16x4(a.q_out, o2 + fa, r_lo);
          st_bf16x4(a.q_out, o2 + fa + 64, r_hi);
        }
      }
    }
    if (norm_out) {
      // sum of h^2 over this CTA's features of each row: the nq units of a row are adjacent lanes
      for (int off = 1; off < nq; off <<= 1) {
        ss0 += __shfl_xor_sync(0xffffffffu, ss0, off);
        ss1 += __shfl_xor_sync(0xffffffffu, ss1, off);
      }
      if (live && qd == 0) {
        const int part = tile * S + split;  // this CTA's features of row n
        a.ss_out[(size_t)n * a.ss_ld + part] = ss0;
        if (EPI == EPI_COUPLE_ADD && a.m_a > 0) a.ss_out[(size_t)(a.m_p + n) * a.ss_ld + part] = ss1;
      }
    }
  }
  if (cb + chunk < p.n_pad) __syncthreads();  // the next pass overwrites the drained rows
  }
  if (a.stamp != nullptr) {  // in-graph timing: this launch's end
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(a.stamp, (unsigned long long)globaltimer());
  }
}

template <int EPI, bool RB = false, bool PRE2 = false>
int launch_epi(const CUtensorMap& mw, const CUtensorMap& mx, const CUtensorMap& mpf, const GemmParams& p, size_t smem,
               cudaStream_t s) {
  auto kern = gemm_tc_kernel<EPI, RB, PRE2>;
  if (set_smem_attrs_once(reinterpret_cast<const void*>(kern)) != DF_OK) return DF_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_tiles, p.row_blocks > 1 ? p.row_blocks : p.splits,
                     (p.a.n_groups > 0 && !p.a.blk_info) ? p.a.n_groups : 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = 1;
  attr[na].val.clusterDim.y = (unsigned)p.splits;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (p.a.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, mw, mx, mpf, p) == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace

void gemm_prefetch_next(const dualflow_ctx* ctx, GemmArgs& cur, const GemmArgs& next) {
  const bool swiglu = next.epi == EPI_SWIGLU;
  cur.pf_W = next.W;
  cur.pf_k = next.k;
  cur.pf_rows = swiglu ? 2 * next.n_out : next.n_out;
  cur.pf_tiles = gemm_tiles(next.n_out, next.epi);
  cur.pf_splits = gemm_splits(ctx, next.n_out, next.k, next.epi);
  cur.pf_tile_rows = swiglu ? 64 : kGemmTileN;
  cur.pf_half = swiglu ? next.n_out : 64;
  cur.pf_depth = kSharedStages;
}

int gemm_tiles(int n_out, int epi) {
  return (epi == EPI_SWIGLU || epi == EPI_MOE_GATEUP) ? n_out / 64 : (n_out + kGemmTileN - 1) / kGemmTileN;
}

// Reduction splits (cluster size): the smallest power of two, at most 8, that gives every SM a
// tile slice, with at least 2 k-blocks per CTA. Depends only on the weight shape and the context's
// capacity, never on which flows are present. Contexts with more than 208 rows of capacity do not
// split (the split-K exchange area is sized for at most 208 padded rows).
// The QKV projection takes at most kQkvSplits ranks: in the decode step the projection before it
// has already warmed its weights in L2, so its CTAs are bound by how many bytes each keeps in flight
// and by the split-K exchange after the last MMA, not by HBM. Fewer, deeper CTAs (one per SM, six
// stages) cut the exchange and leave SMs free for the attention CTAs that follow it (measured on
// B300: 2.373 -> 2.351 ms for the 24-layer dense step).
int gemm_splits(const dualflow_ctx* ctx, int n_out, int k, int epi, int groups) {
  const int tiles = gemm_tiles(n_out, epi) * groups;
  const int kb = k / kGemmTileK;
  const int max_rows = ((2 * ctx->cfg.max_batch + 15) / 16) * 16;
  if (max_rows > kSplitMaxRows) return 1;
  const int cap = epi == EPI_QKV ? kQkvSplits : 8;
  int s = 1;
  while (s < cap && tiles * s < ctx->num_sms && 2 * (2 * s) <= kb) s *= 2;
  return s;
}

// Floats of the split-K exchange area: every CTA of the largest split launch (tiles x S < 2 SMs'
// worth, see gemm_splits) holds a 128 x padded-rows partial.
size_t gemm_part_floats(const dualflow_ctx* ctx) {
  const int max_rows = ((2 * ctx->cfg.max_batch + 15) / 16) * 16;
  if (max_rows > kSplitMaxRows) return 0;
  return (size_t)2 * ctx->num_sms * kGemmTileN * max_rows;
}

int launch_gemm_tc(dualflow_ctx* ctx, const GemmArgs& a, cudaStream_t s) {
  const int m = a.m_p + a.m_a;
  if (m <= 0) return DF_OK;
  if (a.k % kGemmTileK != 0 || a.k <= 0) return DF_ERR_SHAPE;
  if (a.blk_info && !a.row_blocked) return DF_ERR_ARG;
  if (a.row_blocked) {
    // grouped row-blocked launches take their rows gathered per group
    if (a.m_a != 0 || (a.n_groups > 0) != (a.blk_info != nullptr) || !(a.blk_info == nullptr || a.n_blk) ||
        a.seq_rows <= 0)
      return DF_ERR_ARG;
  } else if (m > kGemmMaxAct || m > 2 * ctx->cfg.max_batch) {
    return DF_ERR_SHAPE;
  }
  if ((a.epi == EPI_SWIGLU || a.epi == EPI_MOE_GATEUP) && a.n_out % 64 != 0) return DF_ERR_SHAPE;
  const int groups = a.n_groups > 0 ? a.n_groups : 1;
  if ((a.epi == EPI_MOE_GATEUP || a.epi == EPI_MOE_DOWN) && (!a.sel_pos || a.n_groups <= 0)) return DF_ERR_ARG;
  if (a.epi == EPI_MOE_DOWN && a.n_out % 4 != 0) return DF_ERR_SHAPE;
  if (a.g_next != nullptr && (a.n_out % 64 != 0 || !a.x_next || !a.ss_out)) return DF_ERR_ARG;
  GemmParams p;
  p.a = a;
  p.n_pad = m >= kGemmMaxAct ? kGemmMaxAct : ((m + 15) / 16) * 16;
  // gathered rows: every group's last block may be partial, so at most one block more per group
  p.row_blocks = a.row_blocked ? (m + kGemmMaxAct - 1) / kGemmMaxAct + (a.blk_info ? groups : 0) : 1;
  p.kb_total = a.k / kGemmTileK;
  p.n_tiles = gemm_tiles(a.n_out, a.epi);
  p.splits = a.row_blocked ? 1 : gemm_splits(ctx, a.n_out, a.k, a.epi, groups);
  p.status = ctx->status;
  p.wait_ns = ctx->wait_ns ? ctx->wait_ns : kWaitLimitNs;
  if (p.a.stamp == nullptr) p.a.stamp = ctx->cur_stamp;
  const uintptr_t align = (a.epi == EPI_STORE_BF16 || a.epi == EPI_SWIGLU || a.epi == EPI_MOE_GATEUP) ? 8 : 16;
  p.vec_ok = a.y != nullptr && (reinterpret_cast<uintptr_t>(a.y) % align == 0) && (a.ldy % 4 == 0) ? 1 : 0;
  if (a.g_next != nullptr && !p.vec_ok) return DF_ERR_ARG;
  uint64_t w_rows = (a.epi == EPI_SWIGLU || a.epi == EPI_MOE_GATEUP) ? 2ull * a.n_out : (uint64_t)a.n_out;
  if (groups > 1) w_rows = (uint64_t)groups * a.w_group_rows;
  const uint64_t x_rows = (groups > 1 && a.x_group_rows > 0) ? (uint64_t)groups * a.x_group_rows : (uint64_t)m;
  if (groups > 1 && a.x_group_rows > 0 && a.x_group_rows < m) return DF_ERR_ARG;
  CUtensorMap mw, mx;
  int rc = encode_map_2d_bf16(&mw, a.W, (uint64_t)a.k, w_rows, (uint64_t)a.k * 2, kGemmTileK, 64);
  if (rc != DF_OK) return rc;
  rc = encode_map_2d_bf16(&mx, a.x, (uint64_t)a.k, x_rows, (uint64_t)a.k * 2, kGemmTileK, (uint32_t)p.n_pad);
  if (rc != DF_OK) return rc;
  CUtensorMap mpf = mw;
  if (a.pf_W != nullptr) {
    rc = encode_map_2d_bf16(&mpf, a.pf_W, (uint64_t)a.pf_k, (uint64_t)a.pf_rows, (uint64_t)a.pf_k * 2, kGemmTileK, 64);
    if (rc != DF_OK) return rc;
  }
  // data region: the pipeline stages; after the main loop, unsplit, the accumulator tile (512 B
  // per activation row). Then the barriers, the TMEM address slot and the 256-float row-scale array.
  // as many stages (up to 4) as fit the budget that keeps two CTAs per SM; a grouped launch of more
  // than two CTAs per SM keeps three per SM on fewer stages, so that it runs as one wave
  const int ctas = p.n_tiles * p.splits * groups;
  uint32_t tcols = 32;
  while ((int)tcols < p.n_pad) tcols <<= 1;
  const bool grouped_epi = a.epi == EPI_MOE_GATEUP || a.epi == EPI_MOE_DOWN;  // built for three per SM
  const bool three = grouped_epi && ctas > 2 * ctx->num_sms && ctas <= 3 * ctx->num_sms && 3 * tcols <= 512 &&
                     2 * (kABytes + p.n_pad * 128) <= kStageBudget3 && 512 * p.n_pad <= kStageBudget3;
  // row-blocked (prefill) launches take the two-CTA budget too: while one CTA drains its accumulator
  // tile (in passes, through its pipeline bytes) the other streams its main loop
  p.stages = (three ? kStageBudget3 : kStageBudget) / (kABytes + p.n_pad * 128);
  p.stages = p.stages > kSharedStages ? kSharedStages : (p.stages < 2 ? 2 : p.stages);
  // the decode QKV projection runs one CTA per SM (see gemm_splits): a deeper pipeline
  if (a.epi == EPI_QKV && kQkvStages * (kABytes + p.n_pad * 128) <= 2 * kStageBudget) p.stages = kQkvStages;
  const int pipe = p.stages * (kABytes + p.n_pad * 128);
  // split-K partials go to the exchange area (sized at init for the largest split launch)
  p.part = nullptr;
  if (p.splits > 1) {
    if (ctx->gemm_part == nullptr || (size_t)ctas * kGemmTileN * p.n_pad > ctx->gemm_part_floats)
      return DF_ERR_UNSUPPORTED;
    p.part = ctx->gemm_part;
  }
  // S == 1: the accumulator tile. The row-blocked instantiation drains it through the pipeline
  // bytes in passes of as many 64-row groups as they hold when the whole tile does not fit; every
  // other launch holds the whole tile after its main loop.
  p.chunk = 0;
  if (a.row_blocked && p.splits == 1 && 512 * p.n_pad > pipe) {
    p.chunk = (pipe / (512 * 64)) * 64;
    if (p.chunk < 64) return DF_ERR_UNSUPPORTED;
  }
  const int parts = p.splits == 1 ? 512 * (p.chunk > 0 ? p.chunk : p.n_pad) : 0;
  p.region = ((pipe > parts ? pipe : parts) + 1023) & ~1023;
  const size_t smem = 1024 + (size_t)p.region + 256 + kGemmMaxAct * 12;  // barriers, TMEM slot, row arrays
  if (a.row_blocked) {
    switch (a.epi) {
      case EPI_STORE_F32: return launch_epi<EPI_STORE_F32, true>(mw, mx, mpf, p, smem, s);
      case EPI_ADD_F32: return launch_epi<EPI_ADD_F32, true>(mw, mx, mpf, p, smem, s);
      case EPI_COUPLE_ADD: return launch_epi<EPI_COUPLE_ADD, true>(mw, mx, mpf, p, smem, s);
      case EPI_SWIGLU: return launch_epi<EPI_SWIGLU, true>(mw, mx, mpf, p, smem, s);
      case EPI_PREFILL_QKV: return launch_epi<EPI_PREFILL_QKV, true>(mw, mx, mpf, p, smem, s);
      default: return DF_ERR_UNSUPPORTED;
    }
  }
  // the O and QKV projections with two epilogue units per thread (PRE2)
  const int rows_epi = a.epi == EPI_QKV ? a.m_p : m, units_epi = rows_epi * ((64 / p.splits) / 4);
  const bool pre2 = (a.epi == EPI_ADD_F32 || a.epi == EPI_QKV) && units_epi > kThreads && units_epi <= 2 * kThreads;
  switch (a.epi) {
    case EPI_STORE_F32: return launch_epi<EPI_STORE_F32>(mw, mx, mpf, p, smem, s);
    case EPI_STORE_BF16: return launch_epi<EPI_STORE_BF16>(mw, mx, mpf, p, smem, s);
    case EPI_ADD_F32:
      return pre2 ? launch_epi<EPI_ADD_F32, false, true>(mw, mx, mpf, p, smem, s)
                  : launch_epi<EPI_ADD_F32>(mw, mx, mpf, p, smem, s);
    case EPI_COUPLE_ADD: return launch_epi<EPI_COUPLE_ADD>(mw, mx, mpf, p, smem, s);
    case EPI_QKV:
      return pre2 ? launch_epi<EPI_QKV, false, true>(mw, mx, mpf, p, smem, s)
                  : launch_epi<EPI_QKV>(mw, mx, mpf, p, smem, s);
    case EPI_Q2: return launch_epi<EPI_Q2>(mw, mx, mpf, p, smem, s);
    case EPI_SWIGLU: return launch_epi<EPI_SWIGLU>(mw, mx, mpf, p, smem, s);
    case EPI_MOE_GATEUP: return launch_epi<EPI_MOE_GATEUP>(mw, mx, mpf, p, smem, s);
    case EPI_MOE_DOWN: return launch_epi<EPI_MOE_DOWN>(mw, mx, mpf, p, smem, s);
    default: return DF_ERR_ARG;
  }
}

}  // namespace df
