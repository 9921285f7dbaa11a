// Asymmetric shared-KV decode attention, bf16 storage / fp32 accumulation, sm_103a.
//
// "Atencao de KV Compartilhada Assimetrica" (gist.science technical summary, "Mecanismos Chave"):
// the auxiliary query attends the primary flow's K1/V1, so one load of each K1/V1 tile can serve
// both flows. For every (sequence b, KV head g) the kernel scores the 2*G query rows of group g --
// the G primary heads and the G coupled auxiliary heads -- against the same tile:
//   S^T (16 keys x 8 rows) = K_tile (16 x 128) . Q^T   and   O^T (128 x 8) += V^T . P^T
// with mma.sync m16n8k16 (keys as M, the 8 query rows as N: no padding; P enters as a bf16
// hi/lo pair, two MMAs, so the probabilities are not truncated to 8 significant bits). Tiles of 64 keys are
// staged in shared memory by TMA (128-byte swizzle) through a 3-stage mbarrier pipeline fed by a
// producer warp; four consumer warps take 16 keys each and keep their own online-softmax state
// (running max via warp shuffles), merged at the end of a segment.
//
// Work split (flash-decoding): all (b, g, tile) triples are laid end to end and cut into equal
// contiguous ranges, one per CTA, so ragged lengths balance across the GPU. When every pair has the
// same length T tiles and the grid holds at least one CTA per pair, each pair goes to
// k = min(grid / pairs, T, max(1, T / 8)) CTAs instead, CTA j taking the pair's tiles j, j + k,
// j + 2k, ...: no CTA changes pair, and the pair's CTAs stream through its cache rows side by side.
// A pair cut across
// several CTAs writes per-CTA partials (O, max, sum); the last CTA to arrive (atomic counter, no
// waiting) merges them in CTA order, with all four consumer warps, so the result does not depend
// on arrival order. The query rows of a pair reach shared memory by bulk copy with the pair's
// first tile.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace df {
namespace {

constexpr int kStagesA = 3;
// Per-pair cut: at least this many tiles per CTA. A short call (few tiles per pair) then runs on
// fewer CTAs, all of which find room on the SMs next to the preceding kernel's CTAs and request
// their first tiles before it ends, with fewer partials to merge (config-2 shapes, 8 sequences of
// 2048 keys: 288 -> 128 CTAs, the call 20.3 -> 17.6 us on B300); long pairs are unaffected.
constexpr int kAttnMinTiles = 8;
constexpr int kConsumers = 4;
constexpr int kAttnThreads = (kConsumers + 1) * 32;
constexpr int kHalf = kAttnTileKeys * 128;   // 64 keys x 64 dims x 2 B = 8 KB (one swizzled box)
constexpr int kTileBytes = 2 * kHalf;         // K (or V) tile: 16 KB
constexpr int kStageBytes = 2 * kTileBytes;   // K + V: 32 KB
constexpr int kQBytes = kMaxGroupRows * kHeadDim * 2;  // both flows' query rows of one group: 2 KB
constexpr int kMergeFloats = 36 * 32;         // one warp's state: m0, m1, l0, l1, o[32] for 32 lanes

struct AttnParams {
  AttnArgs a;
  float* part;       // partial slots [pairs + CTAs][kAttnPartFloats]
  int32_t* cnt;      // [pairs] CTAs done with each pair (zero between launches)
  int32_t* status;
  float scale_log2;  // log2(e) / sqrt(D)
  unsigned long long wait_ns;  // limit of the pipeline's bounded waits
};

__device__ __forceinline__ void set_status(int32_t* st, int code) { atomicCAS(st, 0, code); }

// A pipeline wait that gives up after `limit` ns, or at once when another warp of the CTA already
// gave up (err), so that one expired wait ends the CTA's main loop without further waiting.
__device__ __forceinline__ bool wait_or_fail(uint64_t* bar, uint32_t parity, volatile int* err, int32_t* status,
                                             uint64_t limit) {
  if (*err) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (*err) return false;
    if (globaltimer() - t0 > limit) {
      *err = 1;
      set_status(status, DF_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Walks a CTA's (b, g, tile) sequence: consecutive tiles of the global order (stride 0), or every
// stride-th tile of one pair.
struct Walker {
  int b, g, j, tiles_b, stride;
};

__device__ __forceinline__ int tiles_of(const int* sched, int b, int Hkv) { return (sched[b + 1] - sched[b]) / Hkv; }

__device__ __forceinline__ void walker_seek(Walker& w, const int* sched, int B, int Hkv, int t) {
  int b = 0;
  while (b < B - 1 && sched[b + 1] <= t) ++b;
  w.b = b;
  w.tiles_b = tiles_of(sched, b, Hkv);
  const int rem = t - sched[b];
  w.g = w.tiles_b ? rem / w.tiles_b : 0;
  w.j = w.tiles_b ? rem % w.tiles_b : 0;
}

__device__ __forceinline__ void walker_next(Walker& w, const int* sched, int B, int Hkv) {
  if (w.stride > 0) {
    w.j += w.stride;
    return;
  }
  if (++w.j < w.tiles_b) return;
  w.j = 0;
  if (++w.g < Hkv) return;
  w.g = 0;
  do {
    ++w.b;
    w.tiles_b = (w.b < B) ? tiles_of(sched, w.b, Hkv) : 1;
  } while (w.tiles_b == 0);
}

// owner CTA of global tile t when T tiles are cut into C equal contiguous ranges
__device__ __forceinline__ int owner_of(long long t, long long T, int C) { return (int)(((t + 1) * C - 1) / T); }

__device__ __forceinline__ uint32_t swz(int key, int chunk) { return (uint32_t)(key * 128 + ((chunk ^ (key & 7)) << 4)); }

// Global -> shared bulk copy (16-byte aligned, size a multiple of 16), completion on an mbarrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__global__ void __launch_bounds__(kAttnThreads, 2) attn_bf16_kernel(const __grid_constant__ CUtensorMap map_k,
                                                                     const __grid_constant__ CUtensorMap map_v,
                                                                     const AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const AttnArgs& a = P.a;
  const int B = a.batch, Hkv = a.n_kv_heads, Hq = a.n_q_heads, G = Hq / Hkv;
  uint8_t* qbuf = smem + kStagesA * kStageBytes;                           // [kStagesA][kQBytes]
  float* mbuf = reinterpret_cast<float*>(qbuf + kStagesA * kQBytes);       // [kMergeFloats]
  uint64_t* full = reinterpret_cast<uint64_t*>(mbuf + kMergeFloats);
  uint64_t* empty = full + kStagesA;
  volatile int* err = reinterpret_cast<volatile int*>(empty + kStagesA);  // [0] error, [1] merge here
  int* sched = const_cast<int*>(err) + 4;  // [B + 1] exclusive prefix of tiles
  int* lens = sched + B + 1;                // [B] attended positions of each sequence

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers);
    }
    err[0] = 0;
    fence_mbar_init();
  }
  // seq_len is an input of the call, never written by the preceding kernel: read before the
  // programmatic wait. lens[b] holds the attended positions, sched the prefix of tiles.
  for (int b = threadIdx.x; b < B; b += kAttnThreads) {
    const int L = a.seq_len[b] + a.extra;
    lens[b] = (L < 0 || L > a.max_ctx) ? -1 : L;  // out-of-range length: skip the sequence, report it
    if (L < 0 || L > a.max_ctx) set_status(P.status, DF_ERR_DEVICE_BOUNDS);
  }
  __syncthreads();
  for (int b = threadIdx.x; b <= B; b += kAttnThreads) {
    int acc = 0;
    for (int j = 0; j < b; ++j) acc += lens[j] > 0 ? (lens[j] + kAttnTileKeys - 1) / kAttnTileKeys * Hkv : 0;
    sched[b] = acc;
  }
  __syncthreads();
  griddep_launch_dependents();
  const long long T = sched[B];
  // Cut the T tiles over C = min(grid, T) CTAs so that every participating CTA owns at least one
  // tile (the partial-merge counts rely on it); CTAs beyond C only zero empty sequences. When every
  // pair has the same number of tiles and the grid holds k >= 1 CTAs per pair, C = pairs * k: the
  // cuts fall on pair boundaries, every CTA works on one pair, and no CTA pays for a pair change.
  int C = (int)(T < (long long)gridDim.x ? T : (long long)gridDim.x);
  int kpp = 0;  // > 0: kpp CTAs per pair, each taking every kpp-th tile of its pair
  {
    const int per = B > 0 ? sched[1] / Hkv : 0;  // tiles of one pair of sequence 0
    const int pairs = B * Hkv;
    if (per > 0 && pairs <= (int)gridDim.x && T == (long long)pairs * per) {
      bool uniform = true;
      for (int b = 1; b < B && uniform; ++b) uniform = (sched[b + 1] - sched[b] == per * Hkv);
      if (uniform) {
        kpp = min(min((int)gridDim.x / pairs, per), max(1, per / kAttnMinTiles));
        C = pairs * kpp;
      }
    }
  }
  // This CTA's tiles. Contiguous: global tiles [t0, t1). Per pair: CTA c takes tiles j0, j0 + kpp,
  // ... of pair c % pairs (j0 = c / pairs), so the pair's first tiles are every CTA's first tiles,
  // and the CTAs that share a pair are far apart in launch order: the CTAs that become resident
  // first (while the preceding kernel still holds SMs) are spread over the pairs instead of making
  // up whole pairs (measured on B300: -9 us per 24-layer dense step). c_eff = pair * kpp + j0 is
  // the CTA's place in the order of the contiguous cut, which numbers the pair's partial slots and
  // its merge order (owner_of below) in both cases.
  const long long t0 = (c < C) ? T * c / C : 0, t1 = (c < C) ? T * (c + 1) / C : 0;
  int n_my = (int)(t1 - t0);
  int c_eff = c;
  Walker w0;
  if (kpp > 0) {
    const int pairs = B * Hkv;
    const int pr = c % pairs, j0 = c / pairs, per = (c < C) ? tiles_of(sched, pr / Hkv, Hkv) : 0;
    c_eff = pr * kpp + j0;
    n_my = (c < C && j0 < per) ? (per - j0 + kpp - 1) / kpp : 0;
    w0.b = pr / Hkv;
    w0.g = pr % Hkv;
    w0.j = j0;
    w0.tiles_b = per;
    w0.stride = kpp;
  } else if (n_my > 0) {
    walker_seek(w0, sched, B, Hkv, (int)t0);
    w0.stride = 0;
  }

  if (warp == kConsumers) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0 && n_my > 0) {
      tma_prefetch_map(&map_k);
      tma_prefetch_map(&map_v);
      const uint64_t pol = policy_evict_first();
      const int nf = a.aux_on ? 2 : 1;
      const uint32_t qbytes = (uint32_t)(nf * G * kHeadDim * 2);
      Walker w = w0;
      // Under programmatic dependent launch the first stages' tiles are requested before waiting
      // for the preceding kernel, unless they hold the slot that kernel appends (seq_len[b] when
      // extra = 1): the older cache positions are never written by it. The query rows of a
      // segment (written by the preceding kernel) follow the wait; they land in the query area of
      // the stage that holds the segment's first tile, not refilled before the consumers read them.
      bool waited = false;
      int pend_s[kStagesA], pend_b[kStagesA], pend_g[kStagesA], npend = 0;
      auto issue_q = [&](int s, int b, int g) {
        for (int f = 0; f < nf; ++f)
          bulk_load(qbuf + s * kQBytes + f * G * kHeadDim * 2,
                    reinterpret_cast<const __nv_bfloat16*>(a.q) + (((size_t)f * B + b) * Hq + g * G) * kHeadDim,
                    (uint32_t)(G * kHeadDim * 2), &full[s]);
      };
      int issued = 0;
      for (int i = 0; i < n_my; ++i) {
        const int s = (int)(i % kStagesA);
        const uint32_t ph = (uint32_t)(i / kStagesA) & 1u;
        const int key0 = w.j * kAttnTileKeys;
        const int Leff = lens[w.b];
        if (!waited && (i >= kStagesA || (a.extra && key0 + kAttnTileKeys >= Leff))) {
          griddep_wait();
          waited = true;
          for (int k = 0; k < npend; ++k) issue_q(pend_s[k], pend_b[k], pend_g[k]);
          npend = 0;
        }
        if (!wait_or_fail(&empty[s], ph ^ 1u, err, P.status, P.wait_ns)) break;
        const bool seg_start = (w.j == 0) || (i == 0);
        uint8_t* Kst = smem + s * kStageBytes;
        uint8_t* Vst = Kst + kTileBytes;
        if (!a.paged) {
          const int row = w.b * Hkv + w.g;
          mbar_arrive_expect_tx(&full[s], (uint32_t)kStageBytes + (seg_start ? qbytes : 0u));
          tma_load_3d_hint(Kst, &map_k, &full[s], 0, key0, row, pol);
          tma_load_3d_hint(Kst + kHalf, &map_k, &full[s], 64, key0, row, pol);
          tma_load_3d_hint(Vst, &map_v, &full[s], 0, key0, row, pol);
          tma_load_3d_hint(Vst + kHalf, &map_v, &full[s], 64, key0, row, pol);
        } else {
          const int ps = a.page_size, npg = kAttnTileKeys / ps;
          int pid[kAttnTileKeys / 16];
          uint32_t bytes = seg_start ? qbytes : 0u;
          for (int jj = 0; jj < npg; ++jj) {
            const int lp = key0 / ps + jj;
            pid[jj] = -1;
            if (lp * ps < Leff && lp < a.pages_per_seq) {
              const int v = a.page_table[(size_t)w.b * a.pages_per_seq + lp];
              if (v >= 0 && v < a.max_pages) {
                pid[jj] = v;
                bytes += 4u * (uint32_t)ps * 128u;
              } else {
                set_status(P.status, DF_ERR_DEVICE_BOUNDS);
              }
            }
          }
          mbar_arrive_expect_tx(&full[s], bytes);
          for (int jj = 0; jj < npg; ++jj) {
            if (pid[jj] < 0) continue;
            const int row = pid[jj] * Hkv + w.g;
            const int off = jj * ps * 128;
            tma_load_3d_hint(Kst + off, &map_k, &full[s], 0, 0, row, pol);
            tma_load_3d_hint(Kst + kHalf + off, &map_k, &full[s], 64, 0, row, pol);
            tma_load_3d_hint(Vst + off, &map_v, &full[s], 0, 0, row, pol);
            tma_load_3d_hint(Vst + kHalf + off, &map_v, &full[s], 64, 0, row, pol);
          }
        }
        if (seg_start) {
          if (waited) {
            issue_q(s, w.b, w.g);
          } else {
            pend_s[npend] = s;
            pend_b[npend] = w.b;
            pend_g[npend] = w.g;
            ++npend;
          }
        }
        walker_next(w, sched, B, Hkv);
        ++issued;
      }
      if (!waited) {
        griddep_wait();
        for (int k = 0; k < npend; ++k) issue_q(pend_s[k], pend_b[k], pend_g[k]);
      }
      // Every copy issued into the stages has landed before this warp exits, so that none writes
      // into the CTA's shared memory after the CTA is gone (after a wait gave up, the consumers
      // stop reading the stages and may exit first).
      if (!mbar_drain(full, kStagesA, issued)) set_status(P.status, DF_ERR_TIMEOUT);
    }
    return;
  }

  // ------------------------------ consumers ------------------------------
  griddep_wait();  // q is written by the preceding kernel; o may still be read by an older one
  // sequences with nothing to attend: o = 0
  for (int b = c; b < B; b += gridDim.x) {
    if (sched[b + 1] != sched[b]) continue;
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.o);
    const int nf = a.aux_on ? 2 : 1;
    for (int f = 0; f < nf; ++f)
      for (int i = threadIdx.x; i < Hq * kHeadDim; i += kConsumers * 32)
        o[((size_t)f * B + b) * Hq * kHeadDim + i] = __float2bfloat16_rn(0.f);
  }
  if (n_my <= 0) {
    if (a.stamp != nullptr && threadIdx.x == 0) atomicMax(a.stamp, (unsigned long long)globaltimer());
    return;
  }

  const int kw = 16 * warp;
  const int qn = lane >> 2;          // query row this lane feeds into the B fragment
  const int q0 = 2 * (lane & 3);     // the two query rows this lane accumulates
  const float NEG_INF = -INFINITY;
  const uint32_t sbase = smem_u32(smem);

  float m[2] = {NEG_INF, NEG_INF}, l[2] = {0.f, 0.f};
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  uint32_t qb[8][2];

  Walker w = w0;
  bool new_seg = true;
  for (int i = 0; i < n_my; ++i) {
    const int Leff = lens[w.b];
    const int s = (int)(i % kStagesA);
    const uint32_t ph = (uint32_t)(i / kStagesA) & 1u;
    const bool ok = wait_or_fail(&full[s], ph, err, P.status, P.wait_ns);
    if (new_seg) {
      // this group's 2G query rows (primary heads, then auxiliary heads) as B fragments, from the
      // stage's query area
      const int f = qn / G;
      const bool valid = ok && (qn < 2 * G) && (f == 0 || a.aux_on);
      const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qbuf + s * kQBytes + qn * kHeadDim * 2);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qb[kk][0] = valid ? q32[(16 * kk + q0) >> 1] : 0u;
        qb[kk][1] = valid ? q32[(16 * kk + 8 + q0) >> 1] : 0u;
      }
      new_seg = false;
    }
    const int key0 = w.j * kAttnTileKeys;
    const int valid = Leff - key0;
    const uint32_t Kb = sbase + s * kStageBytes, Vb = Kb + kTileBytes;
    if (ok) {
      bool zeroed = false;
      if (valid < kw + 16) {
        // rows past the sequence end: zero V so that p = 0 cannot meet a non-finite value
        uint8_t* Vp = smem + s * kStageBytes + kTileBytes;
        for (int e = lane; e < 16 * 16; e += 32) {
          const int r = kw + (e >> 4), half = (e >> 3) & 1, ch = e & 7;
          if (r >= valid) *reinterpret_cast<uint4*>(Vp + half * kHalf + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        zeroed = true;
      }
      // S^T = K . Q^T for my 16 keys
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int mi = lane >> 3;
        const int key = kw + (lane & 7) + ((mi & 1) << 3);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int chunk = ((kk & 3) << 1) + (mi >> 1);
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4(Kb + (kk >> 2) * kHalf + swz(key, chunk), a0, a1, a2, a3);
          mma_bf16_16816(sc, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        }
      }
      // mask and online softmax (log2 domain)
      const int r0 = kw + qn, r1 = r0 + 8;
      float s0 = (r0 < valid) ? sc[0] * P.scale_log2 : NEG_INF;
      float s1 = (r0 < valid) ? sc[1] * P.scale_log2 : NEG_INF;
      float s2 = (r1 < valid) ? sc[2] * P.scale_log2 : NEG_INF;
      float s3 = (r1 < valid) ? sc[3] * P.scale_log2 : NEG_INF;
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      const float base0 = (mn0 == NEG_INF) ? 0.f : mn0, base1 = (mn1 == NEG_INF) ? 0.f : mn1;
      const float cr0 = exp2f(m[0] - base0), cr1 = exp2f(m[1] - base1);
      const float p0 = exp2f(s0 - base0), p1 = exp2f(s1 - base1), p2 = exp2f(s2 - base0), p3 = exp2f(s3 - base1);
      l[0] = l[0] * cr0 + p0 + p2;
      l[1] = l[1] * cr1 + p1 + p3;
      m[0] = mn0;
      m[1] = mn1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= cr0;
        o[mt][1] *= cr1;
        o[mt][2] *= cr0;
        o[mt][3] *= cr1;
      }
      // P^T (keys x rows) -> B fragments via an in-register 8x8 transpose. P is carried as a bf16
      // pair hi + lo (lo = the rounding residual of hi), so the probabilities enter the fp32
      // accumulation with ~16 significant bits instead of bf16's 8.
      uint32_t ph0, ph1, pl0, pl1;
      {
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1), h23 = __floats2bfloat162_rn(p2, p3);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        ph0 = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&h01));
        ph1 = movmatrix_trans(*reinterpret_cast<const uint32_t*>(&h23));
        pl0 = movmatrix_trans(pack_bf16x2(p0 - f01.x, p1 - f01.y));
        pl1 = movmatrix_trans(pack_bf16x2(p2 - f23.x, p3 - f23.y));
      }
      // O^T += V^T . P^T
      {
        const int mi = lane >> 3;
        const int key = kw + (lane & 7) + ((mi >> 1) << 3);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int chunk = ((mt & 3) << 1) + (mi & 1);
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4_trans(Vb + (mt >> 2) * kHalf + swz(key, chunk), a0, a1, a2, a3);
          mma_bf16_16816(o[mt], a0, a1, a2, a3, ph0, ph1);
          mma_bf16_16816(o[mt], a0, a1, a2, a3, pl0, pl1);
        }
      }
      if (zeroed) fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    // ---- end of this CTA's segment of pair (b, g): merge warps, write result or partial ----
    const bool seg_end = (w.j == w.tiles_b - 1) || (i == n_my - 1);
    if (seg_end) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
      }
      auto put = [&]() {
        mbuf[0 * 32 + lane] = m[0];
        mbuf[1 * 32 + lane] = m[1];
        mbuf[2 * 32 + lane] = l[0];
        mbuf[3 * 32 + lane] = l[1];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int r = 0; r < 4; ++r) mbuf[(4 + mt * 4 + r) * 32 + lane] = o[mt][r];
      };
      auto merge = [&]() {
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const float mb = mbuf[qq * 32 + lane], lb = mbuf[(2 + qq) * 32 + lane];
          const float M = fmaxf(m[qq], mb);
          const float sa = (M == NEG_INF) ? 0.f : exp2f(m[qq] - M);
          const float sb = (M == NEG_INF) ? 0.f : exp2f(mb - M);
          l[qq] = l[qq] * sa + lb * sb;
          m[qq] = M;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            o[mt][qq] = o[mt][qq] * sa + mbuf[(4 + mt * 4 + qq) * 32 + lane] * sb;
            o[mt][qq + 2] = o[mt][qq + 2] * sa + mbuf[(4 + mt * 4 + qq + 2) * 32 + lane] * sb;
          }
        }
      };
      // the four warps' states through one buffer: 3 -> 2, 1 -> 0, 2 -> 0
      constexpr int kBar = 1, kBarThreads = kConsumers * 32;
      named_bar_sync(kBar, kBarThreads);
      if (warp == 3) put();
      named_bar_sync(kBar, kBarThreads);
      if (warp == 2) merge();
      named_bar_sync(kBar, kBarThreads);
      if (warp == 1) put();
      named_bar_sync(kBar, kBarThreads);
      if (warp == 0) merge();
      named_bar_sync(kBar, kBarThreads);
      if (warp == 2) put();
      named_bar_sync(kBar, kBarThreads);
      const int p = w.b * Hkv + w.g;
      const long long pstart = sched[w.b] + (long long)w.g * w.tiles_b;
      const int first = owner_of(pstart, T, C), last = owner_of(pstart + w.tiles_b - 1, T, C);
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(a.o);
      if (warp == 0) {
        merge();
        if (first == last) {
          if (!err[0]) {
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
              const int q = q0 + qq, f = q / G, hh = q % G;
              if (q >= 2 * G || (f == 1 && !a.aux_on)) continue;
              const float inv = 1.0f / l[qq];
              const size_t base = (((size_t)f * B + w.b) * Hq + w.g * G + hh) * kHeadDim;
#pragma unroll
              for (int mt = 0; mt < 8; ++mt) {
                ob[base + 16 * mt + qn] = __float2bfloat16_rn(o[mt][qq] * inv);
                ob[base + 16 * mt + qn + 8] = __float2bfloat16_rn(o[mt][qq + 2] * inv);
              }
            }
          }
        } else {
          float* slot = P.part + (size_t)(p + c_eff) * kAttnPartFloats;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
              slot[(q0 + qq) * kHeadDim + 16 * mt + qn] = o[mt][qq];
              slot[(q0 + qq) * kHeadDim + 16 * mt + qn + 8] = o[mt][qq + 2];
            }
          if (qn == 0) {
            slot[8 * kHeadDim + q0] = m[0];
            slot[8 * kHeadDim + q0 + 1] = m[1];
            slot[8 * kHeadDim + 8 + q0] = l[0];
            slot[8 * kHeadDim + 8 + q0 + 1] = l[1];
          }
          // the warp's writes are ordered before lane 0's release of the count
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            err[1] = (atomicAdd(&P.cnt[p], 1) == last - first) ? 1 : 0;
          }
        }
      }
      if (first != last) {
        named_bar_sync(kBar, kBarThreads);
        if (err[1] && !err[0]) {
          // this CTA finished the pair last: merge the partials of CTAs first..last in CTA order,
          // 8 dims of one query row per consumer thread
          __threadfence();
          const int r = threadIdx.x >> 4, d0 = (threadIdx.x & 15) * 8;
          const float* part0 = P.part + (size_t)(p + first) * kAttnPartFloats;
          const int n = last - first + 1;
          float M = NEG_INF;
#pragma unroll 4
          for (int k = 0; k < n; ++k) M = fmaxf(M, __ldcg(part0 + (size_t)k * kAttnPartFloats + 8 * kHeadDim + r));
          float den = 0.f;
          float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
          for (int k = 0; k < n; ++k) {
            const float* sl = part0 + (size_t)k * kAttnPartFloats;
            const float mv = __ldcg(sl + 8 * kHeadDim + r), lv = __ldcg(sl + 8 * kHeadDim + 8 + r);
            const float4 v0 = __ldcg(reinterpret_cast<const float4*>(sl + r * kHeadDim + d0));
            const float4 v1 = __ldcg(reinterpret_cast<const float4*>(sl + r * kHeadDim + d0 + 4));
            const float wt = (M == NEG_INF) ? 0.f : exp2f(mv - M);
            den += lv * wt;
            acc[0] += v0.x * wt;
            acc[1] += v0.y * wt;
            acc[2] += v0.z * wt;
            acc[3] += v0.w * wt;
            acc[4] += v1.x * wt;
            acc[5] += v1.y * wt;
            acc[6] += v1.z * wt;
            acc[7] += v1.w * wt;
          }
          const int f = r / G, hh = r % G;
          if (r < 2 * G && (f == 0 || a.aux_on)) {
            const float inv = 1.0f / den;
            uint4 u;
            u.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
            u.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
            u.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
            u.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
            *reinterpret_cast<uint4*>(ob + (((size_t)f * B + w.b) * Hq + w.g * G + hh) * kHeadDim + d0) = u;
          }
          if (threadIdx.x == 0) P.cnt[p] = 0;
        }
      }
      // reset the running state for the next pair
      m[0] = m[1] = NEG_INF;
      l[0] = l[1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      new_seg = true;
    }
    walker_next(w, sched, B, Hkv);
  }
  if (a.stamp != nullptr && threadIdx.x == 0) atomicMax(a.stamp, (unsigned long long)globaltimer());
}

}  // namespace

int launch_attention_bf16(dualflow_ctx* ctx, const AttnArgs& a, cudaStream_t s, int pdl) {
  AttnArgs at = a;
  if (at.stamp == nullptr) at.stamp = ctx->cur_stamp;
  return launch_attention_bf16_ws(ctx->cfg, at, ctx->attn_part, ctx->attn_cnt, ctx->status, ctx->attn_ctas, s, pdl,
                                  ctx->wait_ns);
}

int launch_attention_bf16_ws(const dualflow_config& cfg, const AttnArgs& a, float* part, int32_t* cnt,
                             int32_t* status, int ctas, cudaStream_t s, int pdl, unsigned long long wait_ns) {
  if (a.batch <= 0) return DF_OK;
  if (ctas <= 0 || !part || !cnt || !status) return DF_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(a.q) & 15u) return DF_ERR_ARG;  // bulk copies of query rows
  CUtensorMap mk, mv;
  int rc;
  if (!a.paged) {
    const uint64_t rows = (uint64_t)cfg.max_batch * cfg.n_kv_heads;
    const uint64_t seq_stride = (uint64_t)cfg.max_ctx * kHeadDim * 2;
    rc = encode_map_3d_bf16(&mk, a.k_cache, kHeadDim, (uint64_t)cfg.max_ctx, rows, kHeadDim * 2, seq_stride, 64,
                            kAttnTileKeys, 1);
    if (rc == DF_OK)
      rc = encode_map_3d_bf16(&mv, a.v_cache, kHeadDim, (uint64_t)cfg.max_ctx, rows, kHeadDim * 2, seq_stride, 64,
                              kAttnTileKeys, 1);
  } else {
    const uint64_t rows = (uint64_t)cfg.max_pages * cfg.n_kv_heads;
    const uint64_t page_stride = (uint64_t)cfg.page_size * kHeadDim * 2;
    rc = encode_map_3d_bf16(&mk, a.k_cache, kHeadDim, (uint64_t)cfg.page_size, rows, kHeadDim * 2, page_stride, 64,
                            (uint32_t)cfg.page_size, 1);
    if (rc == DF_OK)
      rc = encode_map_3d_bf16(&mv, a.v_cache, kHeadDim, (uint64_t)cfg.page_size, rows, kHeadDim * 2, page_stride, 64,
                              (uint32_t)cfg.page_size, 1);
  }
  if (rc != DF_OK) return rc;
  AttnParams p;
  p.a = a;
  p.part = part;
  p.cnt = cnt;
  p.status = status;
  p.scale_log2 = (float)(1.4426950408889634 / 11.313708498984761);  // log2(e) / sqrt(128)
  p.wait_ns = wait_ns ? wait_ns : kWaitLimitNs;
  const size_t smem = 1024 + (size_t)kStagesA * (kStageBytes + kQBytes) + kMergeFloats * 4 + 2 * kStagesA * 8 + 16 +
                      (size_t)(2 * a.batch + 1) * 4;
  if (set_smem_attrs_once(reinterpret_cast<const void*>(attn_bf16_kernel)) != DF_OK) return DF_ERR_CUDA;
  // No more CTAs than the per-pair cut can use at the longest length the cache holds: the CTAs
  // that would find no tile are not launched at all.
  const long long pairs = (long long)a.batch * cfg.n_kv_heads;
  const long long max_tiles = (cfg.max_ctx + kAttnTileKeys - 1) / kAttnTileKeys;
  const long long useful = pairs * std::max(1LL, (max_tiles + kAttnMinTiles - 1) / kAttnMinTiles);
  const int grid = (int)std::min((long long)ctas, useful);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)grid, 1, 1);
  lc.blockDim = dim3(kAttnThreads, 1, 1);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, attn_bf16_kernel, mk, mv, p) == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace df
