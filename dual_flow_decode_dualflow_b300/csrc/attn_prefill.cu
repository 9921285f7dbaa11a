// Causal attention of the primary-only prefill, bf16 storage / fp32 accumulation, sm_103a.
//
// Prefill ("Custos de Inferencia vs. Treinamento", gist.science technical summary: the auxiliary
// flow is off while a prompt is processed): prompt token t of sequence b sits at absolute position
// p = seq_len[b] + t, and its query attends the cached keys/values of positions 0 .. p (the
// prompt's own keys/values are already in the cache, written by the QKV projection).
//
// Prompt sequence i is held by cache slot b = slots[i] (or i); its keys/values sit in the contiguous
// cache [max_batch, Hkv, max_ctx, D] or in the pages the slot's page-table row maps (every 16-byte
// chunk of a key row is fetched from the row's own page, so any page size works).
//
// One CTA per (block of prompt positions, KV head g, prompt sequence i): its 64 query rows are the G query
// heads of group g at 64 / G consecutive positions, so every K/V tile it loads serves all of
// them. Four warps each own 16 query rows (one head, 16 positions): S = Q K^T and O += P V with
// mma.sync m16n8k16 (queries as M), online softmax per row in the log2 domain, the causal bound
// applied to the tiles that cross it. P enters P V as a bf16 pair hi + lo (lo = the rounding
// residual of hi, two MMAs), so the probabilities keep ~16 significant bits, as in the decode
// attention. K/V tiles of 64 keys are double-buffered in shared memory by
// cp.async, rows XOR-swizzled in 16-byte chunks so that ldmatrix reads are conflict-free.
#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

constexpr int kPfThreads = 128;
constexpr int kPfRows = 64;    // query rows per CTA
constexpr int kPfKeys = 64;    // keys per tile
constexpr int kPfTile = kPfKeys * kHeadDim * 2;  // 16 KB (K or V tile, or the Q block)

__device__ __forceinline__ uint32_t pf_swz(int row, int chunk) {
  return (uint32_t)(row * (kHeadDim * 2) + ((chunk ^ (row & 7)) << 4));
}

// 16-byte global -> shared copy; src_bytes = 0 fills zeros without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct PrefillAttnArgs {
  const __nv_bfloat16* q;  // [B * n_tok, Hq, D] post-RoPE
  __nv_bfloat16* o;        // [B * n_tok, Hq, D]
  const __nv_bfloat16* k_cache;  // [max_batch, Hkv, max_ctx, D], or pages [max_pages, Hkv, page_size, D]
  const __nv_bfloat16* v_cache;
  const int32_t* seq_len;  // [max_batch] positions cached before the prompt
  const int32_t* slots;    // [n_seq] cache slot of each prompt sequence (nullptr: slot i)
  const int32_t* page_table;  // paged: [max_batch, pages_per_seq]
  int n_tok, n_q_heads, n_kv_heads, max_ctx, max_batch;
  int paged, page_size, pages_per_seq, max_pages;
  float scale_log2;
  int32_t* status;
};

__global__ void __launch_bounds__(kPfThreads) attn_prefill_kernel(const PrefillAttnArgs A) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const uint32_t sQ = smem_u32(smem), sK = sQ + kPfTile, sV = sK + 2 * kPfTile;
  const int Hq = A.n_q_heads, Hkv = A.n_kv_heads, G = Hq / Hkv, PP = kPfRows / G;
  const int g = blockIdx.y, si = blockIdx.z, t0 = blockIdx.x * PP;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = A.slots ? A.slots[si] : si;  // cache slot
  if (b < 0 || b >= A.max_batch) {
    if (tid == 0) atomicCAS(A.status, 0, DF_ERR_DEVICE_BOUNDS);
    return;
  }
  const int L = A.seq_len[b];
  if (L < 0 || L + A.n_tok > A.max_ctx) {
    if (tid == 0) atomicCAS(A.status, 0, DF_ERR_DEVICE_BOUNDS);
    return;
  }
  const int npos = min(PP, A.n_tok - t0);
  const int last = L + t0 + npos - 1;       // the block's last absolute position
  const int ntiles = last / kPfKeys + 1;    // key tiles 0 .. last
  const size_t kv_base = A.paged ? 0 : ((size_t)b * Hkv + g) * A.max_ctx * kHeadDim;  // contiguous

  // Q block: row r = head hh (of the group) * PP + local position tl; rows past the prompt are zero
  for (int e = tid; e < kPfRows * 16; e += kPfThreads) {
    const int r = e >> 4, ch = e & 15, hh = r / PP, tl = r % PP;
    const bool ok = tl < npos;
    const __nv_bfloat16* src =
        A.q + (((size_t)si * A.n_tok + (ok ? t0 + tl : 0)) * Hq + g * G + hh) * kHeadDim + ch * 8;
    cp_async16(sQ + pf_swz(r, ch), src, ok ? 16u : 0u);
  }
  auto load_tile = [&](int j, int st) {
    for (int e = tid; e < kPfKeys * 16; e += kPfThreads) {
      const int r = e >> 4, ch = e & 15, key = j * kPfKeys + r;
      bool ok = key <= last;  // later keys are masked; they are never read from global
      size_t off = 0;
      if (ok && !A.paged) {
        off = kv_base + (size_t)key * kHeadDim + ch * 8;
      } else if (ok) {
        const int lp = key / A.page_size;
        const int pid = lp < A.pages_per_seq ? A.page_table[(size_t)b * A.pages_per_seq + lp] : -1;
        if (pid < 0 || pid >= A.max_pages) {
          ok = false;  // unmapped page: zeros, and the error is latched
          atomicCAS(A.status, 0, DF_ERR_DEVICE_BOUNDS);
        } else {
          off = (((size_t)pid * Hkv + g) * A.page_size + key % A.page_size) * kHeadDim + ch * 8;
        }
      }
      cp_async16(sK + st * kPfTile + pf_swz(r, ch), A.k_cache + off, ok ? 16u : 0u);
      cp_async16(sV + st * kPfTile + pf_swz(r, ch), A.v_cache + off, ok ? 16u : 0u);
    }
  };
  load_tile(0, 0);
  cp_async_commit();

  // this thread's two query rows (mma layout): rows lane/4 and lane/4 + 8 of the warp's 16
  const int r0 = warp * 16 + (lane >> 2), r1 = r0 + 8;
  const int p0 = L + t0 + r0 % PP, p1 = L + t0 + r1 % PP;  // absolute positions
  const float NEG_INF = -INFINITY;
  float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  uint32_t qa[8][4];

  for (int j = 0; j < ntiles; ++j) {
    const int st = j & 1;
    if (j + 1 < ntiles) load_tile(j + 1, st ^ 1);
    cp_async_commit();
    cp_async_wait<1>();  // tile j (and the Q block) landed
    __syncthreads();
    if (j == 0) {
      // the warp's 16 query rows as A fragments for the 8 k-steps of D = 128
      const int row = warp * 16 + (lane & 15), cb = lane >> 4;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        ldmatrix_x4(sQ + pf_swz(row, 2 * ks + cb), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
    }
    // S = Q K^T over 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    const uint32_t Kt = sK + st * kPfTile, Vt = sV + st * kPfTile;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {  // keys 16 np .. 16 np + 15
        const int key = 16 * np + ((lane >> 4) << 3) + (lane & 7), ch = 2 * ks + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(Kt + pf_swz(key, ch), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    }
    // scale, causal mask, online softmax (log2 domain); rows r0 (s[.][0..1]) and r1 (s[.][2..3])
    const int kbase = j * kPfKeys + 2 * (lane & 3);
    float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int k0 = kbase + 8 * nt, k1 = k0 + 1;
      s[nt][0] = (k0 <= p0) ? s[nt][0] * A.scale_log2 : NEG_INF;
      s[nt][1] = (k1 <= p0) ? s[nt][1] * A.scale_log2 : NEG_INF;
      s[nt][2] = (k0 <= p1) ? s[nt][2] * A.scale_log2 : NEG_INF;
      s[nt][3] = (k1 <= p1) ? s[nt][3] * A.scale_log2 : NEG_INF;
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float base0 = (n0 == NEG_INF) ? 0.f : n0, base1 = (n1 == NEG_INF) ? 0.f : n1;
    const float c0 = exp2f(m0 - base0), c1 = exp2f(m1 - base1);
    float sum0 = 0.f, sum1 = 0.f;
    uint32_t pa[4][4], pl[4][4];  // P (hi, lo) as A fragments for the 4 k-steps of 16 keys
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float e0 = exp2f(s[nt][0] - base0), e1 = exp2f(s[nt][1] - base0);
      const float e2 = exp2f(s[nt][2] - base1), e3 = exp2f(s[nt][3] - base1);
      sum0 += e0 + e1;
      sum1 += e2 + e3;
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(e0, e1), h23 = __floats2bfloat162_rn(e2, e3);
      const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
      pa[nt >> 1][(nt & 1) * 2 + 0] = *reinterpret_cast<const uint32_t*>(&h01);
      pa[nt >> 1][(nt & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
      pl[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(e0 - f01.x, e1 - f01.y);
      pl[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(e2 - f23.x, e3 - f23.y);
    }
    l0 = l0 * c0 + sum0;
    l1 = l1 * c1 + sum1;
    m0 = n0;
    m1 = n1;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= c0;
      o[i][1] *= c0;
      o[i][2] *= c1;
      o[i][3] *= c1;
    }
    // O += P V: 4 k-steps of 16 keys, 16 n-tiles of 8 dims
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {  // dims 16 dp .. 16 dp + 15
        const int key = 16 * ks + (((lane >> 3) & 1) << 3) + (lane & 7), ch = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(Vt + pf_swz(key, ch), b0, b1, b2, b3);
        // A fragment: a0 (row, keys 16ks + 2(l%4)), a1 (row + 8), a2 (row, +8 keys), a3 (row + 8, +8)
        mma_bf16_16816(o[2 * dp], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b2, b3);
        mma_bf16_16816(o[2 * dp], pl[ks][0], pl[ks][1], pl[ks][2], pl[ks][3], b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pl[ks][0], pl[ks][1], pl[ks][2], pl[ks][3], b2, b3);
      }
    }
    __syncthreads();  // stage st is refilled by the next iteration's loads
  }
  cp_async_wait<0>();

  // row sums over the quad, normalise, store the rows inside the prompt
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int tl0 = r0 % PP, tl1 = r1 % PP, h0 = g * G + r0 / PP, h1 = g * G + r1 / PP;
  const int dcol = 2 * (lane & 3);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int d = 8 * i + dcol;
    if (tl0 < npos)
      *reinterpret_cast<uint32_t*>(A.o + (((size_t)si * A.n_tok + t0 + tl0) * Hq + h0) * kHeadDim + d) =
          pack_bf16x2(o[i][0] * inv0, o[i][1] * inv0);
    if (tl1 < npos)
      *reinterpret_cast<uint32_t*>(A.o + (((size_t)si * A.n_tok + t0 + tl1) * Hq + h1) * kHeadDim + d) =
          pack_bf16x2(o[i][2] * inv1, o[i][3] * inv1);
  }
}

}  // namespace

int launch_attention_prefill(const dualflow_config& c, const void* q, void* o, const void* k_cache,
                             const void* v_cache, const int32_t* seq_len, const int32_t* page_table,
                             const int32_t* slots, int n_seq, int n_tok, int32_t* status, cudaStream_t s) {
  if (n_seq <= 0 || n_tok <= 0) return DF_OK;
  if (c.paged && (!page_table || c.page_size <= 0)) return DF_ERR_ARG;
  const int G = c.n_q_heads / c.n_kv_heads;
  if (c.head_dim != kHeadDim || (G != 1 && G != 2 && G != 4)) return DF_ERR_UNSUPPORTED;
  PrefillAttnArgs A;
  A.q = static_cast<const __nv_bfloat16*>(q);
  A.o = static_cast<__nv_bfloat16*>(o);
  A.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  A.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  A.seq_len = seq_len;
  A.slots = slots;
  A.page_table = page_table;
  A.paged = c.paged;
  A.page_size = c.paged ? c.page_size : 1;
  A.pages_per_seq = c.paged ? (c.max_ctx + c.page_size - 1) / c.page_size : 0;
  A.max_pages = c.max_pages;
  A.max_batch = c.max_batch;
  A.n_tok = n_tok;
  A.n_q_heads = c.n_q_heads;
  A.n_kv_heads = c.n_kv_heads;
  A.max_ctx = c.max_ctx;
  A.scale_log2 = (float)(1.4426950408889634 / 11.313708498984761);  // log2(e) / sqrt(128)
  A.status = status;
  const int PP = kPfRows / G;
  const size_t smem = 128 + 5 * (size_t)kPfTile;  // Q block + 2 K tiles + 2 V tiles
  if (cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return DF_ERR_CUDA;
  dim3 grid((n_tok + PP - 1) / PP, c.n_kv_heads, n_seq);
  attn_prefill_kernel<<<grid, kPfThreads, smem, s>>>(A);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace df
