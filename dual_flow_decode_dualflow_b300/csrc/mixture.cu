// Mixture head and token choice of the dual-flow decoder, fp32, sm_103a.
//
// "Objetivo de Mistura" (gist.science technical summary, "Mecanismos Chave"): the next-token
// distribution mixes both flows' predictions with a weight that grows with the primary flow's
// confidence and never drops below one half. The reading implemented here: p_f = softmax(logits_f),
// alpha = 1/2 + 1/2 * sum_i p1_i^2 (the collision probability of p1 mapped to [1/2, 1]),
// p_mix = alpha * p1 + (1 - alpha) * p2. The token is the argmax of p_mix (ties to the lower index)
// or, given a uniform u in [0, 1), the smallest i whose cumulative p_mix exceeds u (inverse-transform
// sampling; the last i with p_mix_i > 0 when rounding leaves none).
//
// One thread-block cluster per sequence; its S CTAs (S <= 8) split the vocabulary into contiguous
// slices. Pass 1: each CTA reduces its slice of both flows' logits to an online-softmax triple
// (max, sum of exp, sum of exp^2), exchanged over distributed shared memory and combined in rank
// order, so every CTA holds the same (M1, Z1, Q1, M2, Z2) and alpha = 1/2 + Q1 / (2 Z1^2). Pass 2:
// every thread owns a contiguous run of its CTA's slice, computes p_mix there (stored if asked),
// its running argmax and its sum; block and cluster scans in fixed order give each run its start
// on the cumulative axis, and the one run whose interval holds u walks its elements. All
// reductions have a fixed order: the result does not depend on scheduling.
#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

constexpr int kMixThreads = 256;
constexpr int kMixWarps = kMixThreads / 32;
constexpr int kMixMaxCluster = 8;

struct Soft {  // online softmax state of one flow: max, sum e^(l - m), sum e^(2 (l - m))
  float m, s, q;
};

__device__ __forceinline__ Soft soft_add(Soft a, float l) {
  if (l > a.m) {
    const float f = expf(a.m - l);  // 0 when a.m = -inf
    a.s = __fmaf_rn(a.s, f, 1.f);
    a.q = __fmaf_rn(a.q, f * f, 1.f);
    a.m = l;
  } else {
    const float e = expf(l - a.m);
    a.s = __fadd_rn(a.s, e);
    a.q = __fmaf_rn(e, e, a.q);
  }
  return a;
}

__device__ __forceinline__ Soft soft_merge(Soft a, Soft b) {
  const float M = fmaxf(a.m, b.m);
  if (M == -INFINITY) return a;
  const float fa = expf(a.m - M), fb = expf(b.m - M);
  Soft r;
  r.m = M;
  r.s = __fadd_rn(a.s * fa, b.s * fb);
  r.q = __fadd_rn(a.q * (fa * fa), b.q * (fb * fb));
  return r;
}

__device__ __forceinline__ Soft soft_shfl(Soft a, int off) {
  Soft b;
  b.m = __shfl_xor_sync(0xffffffffu, a.m, off);
  b.s = __shfl_xor_sync(0xffffffffu, a.s, off);
  b.q = __shfl_xor_sync(0xffffffffu, a.q, off);
  return b;
}

// (value, index) argmax step: larger value wins, equal values go to the lower index.
__device__ __forceinline__ void arg_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

struct MixShared {
  Soft soft[2][kMixWarps];  // per-warp partials, then [f][0] the CTA's
  float best_v[kMixWarps];
  int best_i[kMixWarps];
  int last_pos[kMixWarps];
  float warp_total[kMixWarps];
  float run_start[kMixThreads];  // exclusive scan of the runs' sums of p_mix
  // the CTA's results read by the other CTAs of the cluster
  float cta_soft[2][3];
  float cta_best_v;
  int cta_best_i;
  int cta_last_pos;
  float cta_total;
  int cta_pick;
};

// grid (S, B), cluster (S, 1, 1), 256 threads. logits [2][B][V] fp32. primary_only: the choice is
// made from softmax(logits_1) alone (alpha = 1; the auxiliary logits are not read). token2: a second
// copy of the chosen tokens (the next decode step's input), or null.
__global__ void __launch_bounds__(kMixThreads) mixture_head_kernel(const float* __restrict__ logits, int B, int V,
                                                                   const float* __restrict__ u, float* alpha_out,
                                                                   float* p_mix, int32_t* token_out, int32_t* token2,
                                                                   int primary_only) {
  __shared__ MixShared sh;
  const int S = gridDim.x, r = blockIdx.x, b = blockIdx.y;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int chunk = (V + S - 1) / S;
  const int lo = r * chunk, hi = min(V, lo + chunk), n = max(0, hi - lo);
  const float* l1 = logits + (size_t)b * V + lo;
  const float* l2 = logits + ((size_t)B + b) * V + lo;

  // ---- pass 1: online softmax triples of both flows over the slice ----
  Soft s1 = {-INFINITY, 0.f, 0.f}, s2 = {-INFINITY, 0.f, 0.f};
  // sixteen of the thread's logits per flow requested at a time, then added in index order
  constexpr int kMixLoads = 16;
  for (int i0 = t; i0 < n; i0 += kMixLoads * kMixThreads) {
    float a1[kMixLoads], a2[kMixLoads];
#pragma unroll
    for (int j = 0; j < kMixLoads; ++j) {
      const int i = i0 + j * kMixThreads;
      a1[j] = i < n ? __ldg(l1 + i) : 0.f;
      a2[j] = (i < n && !primary_only) ? __ldg(l2 + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kMixLoads; ++j)
      if (i0 + j * kMixThreads < n) {
        s1 = soft_add(s1, a1[j]);
        if (!primary_only) s2 = soft_add(s2, a2[j]);
      }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    s1 = soft_merge(s1, soft_shfl(s1, off));
    s2 = soft_merge(s2, soft_shfl(s2, off));
  }
  if (lane == 0) {
    sh.soft[0][warp] = s1;
    sh.soft[1][warp] = s2;
  }
  __syncthreads();
  if (t < 2) {
    Soft acc = sh.soft[t][0];
    for (int w = 1; w < kMixWarps; ++w) acc = soft_merge(acc, sh.soft[t][w]);
    sh.cta_soft[t][0] = acc.m;
    sh.cta_soft[t][1] = acc.s;
    sh.cta_soft[t][2] = acc.q;
  }
  cluster_sync();
  // every CTA combines the S triples in rank order (identical result in every CTA)
  Soft g1 = {-INFINITY, 0.f, 0.f}, g2 = {-INFINITY, 0.f, 0.f};
  const uint32_t soft_addr = smem_u32(&sh.cta_soft[0][0]);
  for (int k = 0; k < S; ++k) {
    const uint32_t ra = mapa_shared(soft_addr, (uint32_t)k);
    const Soft a1 = {ld_dsmem_f32(ra), ld_dsmem_f32(ra + 4), ld_dsmem_f32(ra + 8)};
    const Soft a2 = {ld_dsmem_f32(ra + 12), ld_dsmem_f32(ra + 16), ld_dsmem_f32(ra + 20)};
    g1 = soft_merge(g1, a1);
    g2 = soft_merge(g2, a2);
  }
  const float iz1 = 1.f / g1.s, iz2 = primary_only ? 0.f : 1.f / g2.s;
  const float alpha = primary_only ? 1.f : __fmaf_rn(0.5f, g1.q * (iz1 * iz1), 0.5f);
  const float beta = 1.f - alpha;

  // ---- pass 2: p_mix over this thread's contiguous run ----
  const int per = (n + kMixThreads - 1) / kMixThreads;
  const int i0 = min(n, t * per), i1 = min(n, i0 + per);
  float run = 0.f, bv = -INFINITY;
  int bi = 0x7fffffff, lastpos = -1;
  for (int c0 = i0; c0 < i1; c0 += kMixLoads) {
    float x1[kMixLoads], x2[kMixLoads];
#pragma unroll
    for (int j = 0; j < kMixLoads; ++j) {
      const int i = c0 + j;
      x1[j] = i < i1 ? __ldg(l1 + i) : 0.f;
      x2[j] = (i < i1 && !primary_only) ? __ldg(l2 + i) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kMixLoads; ++j) {
      const int i = c0 + j;
      if (i >= i1) continue;
      const float p1 = expf(x1[j] - g1.m) * iz1;
      const float p2 = primary_only ? 0.f : expf(x2[j] - g2.m) * iz2;
      const float pm = __fmaf_rn(alpha, p1, beta * p2);
      if (p_mix) p_mix[(size_t)b * V + lo + i] = pm;
      if (pm > bv) {
        bv = pm;
        bi = lo + i;
      }
      if (pm > 0.f) lastpos = lo + i;
      run = __fadd_rn(run, pm);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    arg_merge(bv, bi, __shfl_xor_sync(0xffffffffu, bv, off), __shfl_xor_sync(0xffffffffu, bi, off));
    lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off));
  }
  // scan of the runs' sums in thread order: a fixed shuffle tree inside each warp, then the warps'
  // totals in order
  float incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl = __fadd_rn(y, incl);
  }
  float excl_w = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl_w = 0.f;
  if (lane == 31) sh.warp_total[warp] = incl;
  if (lane == 0) {
    sh.best_v[warp] = bv;
    sh.best_i[warp] = bi;
    sh.last_pos[warp] = lastpos;
  }
  __syncthreads();
  if (t == 0) {
    float v = sh.best_v[0];
    int ix = sh.best_i[0], lp = sh.last_pos[0];
    for (int w = 1; w < kMixWarps; ++w) {
      arg_merge(v, ix, sh.best_v[w], sh.best_i[w]);
      lp = max(lp, sh.last_pos[w]);
    }
    float acc = 0.f;
    for (int w = 0; w < kMixWarps; ++w) {
      const float x = sh.warp_total[w];
      sh.warp_total[w] = acc;  // now the warp's exclusive offset
      acc = __fadd_rn(acc, x);
    }
    sh.cta_best_v = v;
    sh.cta_best_i = ix;
    sh.cta_last_pos = lp;
    sh.cta_total = acc;
    sh.cta_pick = 0x7fffffff;
  }
  __syncthreads();
  sh.run_start[t] = __fadd_rn(sh.warp_total[warp], excl_w);  // this run's start within the CTA's slice
  cluster_sync();
  // cluster view, in rank order: argmax, last positive index, this CTA's offset on the cumulative axis
  float gv = -INFINITY, offset = 0.f, total = 0.f;
  int gi = 0x7fffffff, glast = -1;
  {
    const uint32_t bv_addr = smem_u32(&sh.cta_best_v), bi_addr = smem_u32(&sh.cta_best_i);
    const uint32_t lp_addr = smem_u32(&sh.cta_last_pos), tot_addr = smem_u32(&sh.cta_total);
    for (int k = 0; k < S; ++k) {
      arg_merge(gv, gi, ld_dsmem_f32(mapa_shared(bv_addr, (uint32_t)k)),
                (int)ld_dsmem_u32(mapa_shared(bi_addr, (uint32_t)k)));
      glast = max(glast, (int)ld_dsmem_u32(mapa_shared(lp_addr, (uint32_t)k)));
      const float tk = ld_dsmem_f32(mapa_shared(tot_addr, (uint32_t)k));
      if (k == r) offset = total;
      total = __fadd_rn(total, tk);
    }
  }
  int pick = -1;
  if (u != nullptr) {
    // run r covers [e_r, e_r+1) with e_r = fl(offset + start of r); the next CTA's first run starts at
    // fl(offset + total), this CTA's last boundary. Consecutive intervals share their boundary, so
    // every u in [0, total) lies in some run's interval; where rounding makes two overlap, the
    // lower index wins.
    const float uu = __ldg(u + b);
    const float start = __fadd_rn(offset, sh.run_start[t]);
    const float end = __fadd_rn(offset, (t + 1 < kMixThreads) ? sh.run_start[t + 1] : sh.cta_total);
    if (i1 > i0 && start <= uu && uu < end) {
      float c = start;
      int lastp = -1;
      for (int i = i0; i < i1; ++i) {
        const float p1 = expf(__ldg(l1 + i) - g1.m) * iz1;
        const float p2 = primary_only ? 0.f : expf(__ldg(l2 + i) - g2.m) * iz2;
        const float pm = __fmaf_rn(alpha, p1, beta * p2);
        if (pm > 0.f) lastp = lo + i;
        c = __fadd_rn(c, pm);
        if (c > uu) {
          pick = lo + i;
          break;
        }
      }
      if (pick < 0) pick = lastp >= 0 ? lastp : lo + i1 - 1;  // rounding ended the walk at or below u
      atomicMin(&sh.cta_pick, pick);
    }
  }
  cluster_sync();
  if (r == 0 && t == 0) {
    if (alpha_out) alpha_out[b] = alpha;
    if (token_out) {
      int tok = gi;
      if (u != nullptr) {
        int p = 0x7fffffff;
        const uint32_t pk_addr = smem_u32(&sh.cta_pick);
        for (int k = 0; k < S; ++k) p = min(p, (int)ld_dsmem_u32(mapa_shared(pk_addr, (uint32_t)k)));
        tok = (p != 0x7fffffff) ? p : glast;
      }
      token_out[b] = tok;
      if (token2) token2[b] = tok;
    }
  }
  cluster_sync();  // no CTA leaves while its shared memory may still be read
}

// After a decode step of the generation loop: every sequence's length grows by one (its new entry
// is in the cache), and a paged sequence whose next slot opens a page gets one from the free list,
// taken from the top in sequence order. The page assignment is one thread's, so it does not depend
// on scheduling. A length that would reach max_ctx, a page slot beyond the table, or an empty free
// list latches DF_ERR_DEVICE_BOUNDS and leaves that sequence as it is.
__global__ void gen_advance_kernel(int32_t* seq_len, int B, int max_ctx, int paged, int page_size, int32_t* table,
                                   int pages_per_seq, int max_pages, int32_t* free_pages, int32_t* n_free,
                                   int32_t* status) {
  // every length is read at once (one round trip), then advanced; page allocation, when a next slot
  // opens a page, stays with one thread in sequence order (the free list is taken from the top)
  extern __shared__ int32_t next_len[];  // [B]
  for (int b = threadIdx.x; b < B; b += blockDim.x) next_len[b] = seq_len[b] + 1;  // the next step writes slot L
  __syncthreads();
  if (!paged) {
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      const int L = next_len[b];
      if (L < 1 || L >= max_ctx)
        atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
      else
        seq_len[b] = L;
    }
    return;
  }
  if (threadIdx.x != 0) return;
  for (int b = 0; b < B; ++b) {
    const int L = next_len[b];
    if (L < 1 || L >= max_ctx) {
      atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
      continue;
    }
    if (L % page_size == 0) {
      const int j = L / page_size;
      int32_t* slot = table + (size_t)b * pages_per_seq + j;
      if (j >= pages_per_seq) {
        atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
        continue;
      }
      if (*slot < 0) {
        const int nf = n_free ? *n_free : 0;
        const int pid = (free_pages && nf > 0) ? free_pages[nf - 1] : -1;
        if (pid < 0 || pid >= max_pages) {
          atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
          continue;
        }
        *slot = pid;
        *n_free = nf - 1;
      }
    }
    seq_len[b] = L;
  }
}

__global__ void seq_advance_kernel(int32_t* seq_len, const int32_t* slots, int n_seq, int max_batch, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_seq) return;
  const int b = slots ? slots[i] : i;
  if (b >= 0 && b < max_batch) seq_len[b] += n;
}

// Before a prefill of n positions into the cache slots of the prompt sequences (slots[i], or i):
// every page of a paged slot that positions seq_len[b] .. seq_len[b] + n touch (the prompt, and the
// slot the next decode step writes, while it is below max_ctx) and that the table does not map yet
// is taken from the top of the free list, in prompt order and page order. One thread: the page
// assignment does not depend on scheduling. A slot or page outside the table, or an empty free
// list, latches DF_ERR_DEVICE_BOUNDS and leaves the rest of that sequence's pages unmapped (the
// prefill's accesses there are then skipped and latch the same error).
__global__ void prefill_pages_kernel(const int32_t* seq_len, const int32_t* slots, int n_seq, int n, int max_batch,
                                     int max_ctx, int page_size, int32_t* table, int pages_per_seq, int max_pages,
                                     int32_t* free_pages, int32_t* n_free, int32_t* status) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  for (int i = 0; i < n_seq; ++i) {
    const int b = slots ? slots[i] : i;
    if (b < 0 || b >= max_batch) {
      atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
      continue;
    }
    const int L = seq_len[b];
    if (L < 0 || L + n > max_ctx) {
      atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
      continue;
    }
    const int last = min(L + n, max_ctx - 1);
    for (int j = L / page_size; j <= last / page_size; ++j) {
      int32_t* e = table + (size_t)b * pages_per_seq + j;
      if (j >= pages_per_seq) {
        atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
        break;
      }
      if (*e >= 0) continue;
      const int nf = *n_free;
      const int pid = nf > 0 ? free_pages[nf - 1] : -1;
      if (pid < 0 || pid >= max_pages) {
        atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
        break;
      }
      *e = pid;
      *n_free = nf - 1;
    }
  }
}

// Ends the sequences held by the listed cache slots: a paged slot's mapped pages go back on top of
// the free list in page order and its table row is cleared; every listed slot's length becomes 0.
// One thread. A slot outside the table, or a free list that already holds max_pages entries,
// latches DF_ERR_DEVICE_BOUNDS (the page then stays mapped to the slot).
__global__ void release_slots_kernel(int32_t* seq_len, const int32_t* slots, int n, int max_batch, int paged,
                                     int32_t* table, int pages_per_seq, int max_pages, int32_t* free_pages,
                                     int32_t* n_free, int32_t* status) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  for (int i = 0; i < n; ++i) {
    const int b = slots[i];
    if (b < 0 || b >= max_batch) {
      atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
      continue;
    }
    if (paged)
      for (int j = 0; j < pages_per_seq; ++j) {
        int32_t* e = table + (size_t)b * pages_per_seq + j;
        if (*e < 0) continue;
        const int nf = *n_free;
        if (nf < 0 || nf >= max_pages) {
          atomicCAS(status, 0, DF_ERR_DEVICE_BOUNDS);
          continue;
        }
        free_pages[nf] = *e;
        *n_free = nf + 1;
        *e = -1;
      }
    seq_len[b] = 0;
  }
}

}  // namespace

// After a prefill of n positions: the cached length of every prompt sequence's slot grows by n (the
// bounds were checked by the kernels that wrote the entries).
int launch_seq_advance(int32_t* seq_len, const int32_t* slots, int n_seq, int max_batch, int n, cudaStream_t s) {
  seq_advance_kernel<<<(n_seq + 127) / 128, 128, 0, s>>>(seq_len, slots, n_seq, max_batch, n);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_prefill_pages(const dualflow_config& c, const int32_t* seq_len, const int32_t* slots, int n_seq, int n,
                         int32_t* table, int32_t* free_pages, int32_t* n_free, int32_t* status, cudaStream_t s) {
  const int pps = (c.max_ctx + c.page_size - 1) / c.page_size;
  prefill_pages_kernel<<<1, 32, 0, s>>>(seq_len, slots, n_seq, n, c.max_batch, c.max_ctx, c.page_size, table, pps,
                                        c.max_pages, free_pages, n_free, status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_release_slots(const dualflow_config& c, int32_t* seq_len, const int32_t* slots, int n_slots, int32_t* table,
                         int32_t* free_pages, int32_t* n_free, int32_t* status, cudaStream_t s) {
  const int pps = c.paged ? (c.max_ctx + c.page_size - 1) / c.page_size : 0;
  release_slots_kernel<<<1, 32, 0, s>>>(seq_len, slots, n_slots, c.max_batch, c.paged, table, pps, c.max_pages,
                                        free_pages, n_free, status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_gen_advance(const dualflow_config& c, int32_t* seq_len, int batch, int32_t* table, int32_t* free_pages,
                       int32_t* n_free, int32_t* status, cudaStream_t s) {
  const int pps = c.paged ? (c.max_ctx + c.page_size - 1) / c.page_size : 0;
  gen_advance_kernel<<<1, 256, (size_t)batch * sizeof(int32_t), s>>>(seq_len, batch, c.max_ctx, c.paged, c.page_size,
                                                                      table, pps, c.max_pages, free_pages, n_free,
                                                                      status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_mixture_head(const float* logits, int batch, int vocab, const float* u, float* alpha, float* p_mix,
                        int32_t* token, int32_t* token2, int aux_on, cudaStream_t s) {
  int S = (vocab + 4095) / 4096;
  S = S < 1 ? 1 : (S > kMixMaxCluster ? kMixMaxCluster : S);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(S, batch, 1);
  lc.blockDim = dim3(kMixThreads, 1, 1);
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, mixture_head_kernel, logits, batch, vocab, u, alpha, p_mix, token, token2,
                            aux_on ? 0 : 1) == cudaSuccess
             ? DF_OK
             : DF_ERR_CUDA;
}

}  // namespace df
