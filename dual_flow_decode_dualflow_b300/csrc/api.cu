// C ABI of the Dual-Flow decode library: validation, workspace, orchestration of the step,
// CUDA-graph capture and replay. Every arithmetic step runs in the kernels of this library.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include "internal.h"

using namespace df;

namespace df {

// ------------------------------------------------------------------ tensor maps
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
}  // namespace
thread_local char t_driver_error[96] = "";  // last driver call of this library that failed here
namespace {
thread_local int t_context_bound = -1;      // device whose primary context this thread made current

// The tensor-map encoder is a driver call: it needs the device's context current in the calling
// thread, which a host thread that has made no runtime call yet does not have. cudaSetDevice makes
// the device's primary context current (creating nothing once the device is initialised).
int bind_context() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DF_ERR_CUDA;
  if (dev != t_context_bound) {
    if (cudaSetDevice(dev) != cudaSuccess) return DF_ERR_CUDA;
    t_context_bound = dev;
  }
  return DF_OK;
}

int encode_failed(CUresult r) {
  snprintf(t_driver_error, sizeof(t_driver_error), "cuTensorMapEncodeTiled returned CUresult %d", (int)r);
  return DF_ERR_CUDA;
}

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? DF_OK : DF_ERR_CUDA;
}
}  // namespace

int set_smem_attrs_once(const void* kernel) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;  // (kernel, device) already set
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DF_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& e : done)
    if (e.first == kernel && e.second == dev) return DF_OK;
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || optin <= 0)
    return DF_ERR_CUDA;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess ||
      cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return DF_ERR_CUDA;
  done.emplace_back(kernel, dev);
  return DF_OK;
}

int encode_map_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                       uint32_t box_inner, uint32_t box_rows) {
  if (get_encoder() != DF_OK || bind_context() != DF_OK) return DF_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (row_stride_bytes & 15u)) return DF_ERR_ARG;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DF_OK : encode_failed(r);
}

int encode_map_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                       uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
  if (get_encoder() != DF_OK || bind_context() != DF_OK) return DF_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || (stride1_bytes & 15u) || (stride2_bytes & 15u)) return DF_ERR_ARG;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DF_OK : encode_failed(r);
}

}  // namespace df

// ------------------------------------------------------------------ helpers
namespace {

size_t elem_size(const dualflow_config& c) { return c.dtype == DF_DTYPE_BF16 ? 2 : 4; }

int validate_config(const dualflow_config* c) {
  if (!c) return DF_ERR_ARG;
  if (c->dtype != DF_DTYPE_F32 && c->dtype != DF_DTYPE_BF16) return DF_ERR_DTYPE;
  if (c->n_layers < 0 || c->d_model <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
      c->ffn_hidden < 0 || c->vocab < 0 || c->max_batch <= 0 || c->max_ctx <= 0 || c->n_experts < 0)
    return DF_ERR_ARG;
  if (c->n_q_heads % c->n_kv_heads != 0 || c->head_dim % 2 != 0) return DF_ERR_SHAPE;
  if (!(c->rms_eps >= 0.f) || !(c->rope_base > 0.f)) return DF_ERR_ARG;
  if (c->paged && (c->page_size <= 0 || c->max_pages <= 0)) return DF_ERR_ARG;
  if (c->n_experts > 0 && (c->topk_primary <= 0 || c->topk_aux <= 0 || c->topk_primary > c->n_experts ||
                           c->topk_aux > c->n_experts))
    return DF_ERR_SHAPE;
  if (c->dtype == DF_DTYPE_BF16) {
    const int G = c->n_q_heads / c->n_kv_heads;
    if (c->head_dim != kHeadDim || 2 * G > kMaxGroupRows) return DF_ERR_UNSUPPORTED;
    if (c->d_model % 64 || c->ffn_hidden % 64 || (c->n_q_heads * c->head_dim) % 64) return DF_ERR_UNSUPPORTED;
    if (2 * c->max_batch > kGemmMaxAct) return DF_ERR_UNSUPPORTED;
    if (c->paged && c->page_size != 16 && c->page_size != 32 && c->page_size != 64) return DF_ERR_UNSUPPORTED;
    if (c->n_experts > 32) return DF_ERR_UNSUPPORTED;  // routing keeps one expert per lane of a warp
  } else {
    if (c->head_dim / 2 > 1024 || c->max_ctx > 40000 || c->d_model % 4) return DF_ERR_UNSUPPORTED;
    if (c->n_experts > 0) return DF_ERR_UNSUPPORTED;
  }
  return DF_OK;
}

template <typename T>
int dalloc(T** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  return cudaMalloc(reinterpret_cast<void**>(p), bytes) == cudaSuccess ? DF_OK : DF_ERR_OOM;
}

cudaStream_t S(dualflow_stream s) { return reinterpret_cast<cudaStream_t>(s); }

#define DF_TRY(x)              \
  do {                         \
    int _rc = (x);             \
    if (_rc != DF_OK) return _rc; \
  } while (0)

int pages_per_seq(const dualflow_config& c) { return c.paged ? (c.max_ctx + c.page_size - 1) / c.page_size : 0; }

GemmArgs gemm_args(const dualflow_ctx* ctx) {
  GemmArgs g;
  memset(&g, 0, sizeof(g));
  const dualflow_config& c = ctx->cfg;
  g.n_q_heads = c.n_q_heads;
  g.n_kv_heads = c.n_kv_heads;
  g.rope = ctx->rope;
  g.paged = c.paged;
  g.page_size = c.paged ? c.page_size : 1;
  g.max_ctx = c.max_ctx;
  g.max_pages = c.max_pages;
  g.pages_per_seq = pages_per_seq(c);
  return g;
}

AttnArgs attn_args(const dualflow_ctx* ctx, const dualflow_kv* kv, int layer, int batch, int extra, int aux_on) {
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  const dualflow_config& c = ctx->cfg;
  a.q = ctx->q;
  a.o = ctx->o;
  a.k_cache = kv->k[layer];
  a.v_cache = kv->v[layer];
  a.seq_len = kv->seq_len;
  a.page_table = kv->page_table;
  a.batch = batch;
  a.n_q_heads = c.n_q_heads;
  a.n_kv_heads = c.n_kv_heads;
  a.paged = c.paged;
  a.page_size = c.paged ? c.page_size : 1;
  a.max_ctx = c.max_ctx;
  a.max_pages = c.max_pages;
  a.pages_per_seq = pages_per_seq(c);
  a.extra = extra;
  a.aux_on = aux_on;
  return a;
}

int check_kv(const dualflow_ctx* ctx, const dualflow_kv* kv, int layer) {
  if (!kv || !kv->k || !kv->v || !kv->seq_len) return DF_ERR_ARG;
  if (layer < 0 || layer >= kv->n_layers) return DF_ERR_ARG;
  if (!kv->k[layer] || !kv->v[layer]) return DF_ERR_ARG;
  if (ctx->cfg.paged && !kv->page_table) return DF_ERR_ARG;
  return DF_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every weight pointer must be non-null and 16-byte aligned (TMA and vector loads).
int check_weights(const dualflow_ctx* ctx, const dualflow_weights* w) {
  const dualflow_config& c = ctx->cfg;
  if (!w || w->n_layers != c.n_layers) return DF_ERR_ARG;
  auto ok = [](const void* p) { return p != nullptr && aligned16(p); };
  if (!ok(w->E1) || !ok(w->E2) || !ok(w->W_lm) || !ok(w->g_final)) return DF_ERR_ARG;
  if (!w->g_attn || !w->g_mlp || !w->Wqkv || !w->Wo || !w->a || !w->b || !w->c) return DF_ERR_ARG;
  if (c.n_experts == 0 && (!w->Wgu || !w->Wd)) return DF_ERR_ARG;
  if (c.n_experts > 0 && (!w->Wr || !w->We_gu || !w->We_d)) return DF_ERR_ARG;
  for (int l = 0; l < c.n_layers; ++l) {
    if (!ok(w->g_attn[l]) || !ok(w->g_mlp[l]) || !ok(w->Wqkv[l]) || !ok(w->Wo[l]) || !ok(w->a[l]) || !ok(w->b[l]) ||
        !ok(w->c[l]))
      return DF_ERR_ARG;
    if (c.n_experts == 0 && (!ok(w->Wgu[l]) || !ok(w->Wd[l]))) return DF_ERR_ARG;
    if (c.n_experts > 0 && (!ok(w->Wr[l]) || !ok(w->We_gu[l]) || !ok(w->We_d[l]))) return DF_ERR_ARG;
  }
  return DF_OK;
}

// ------------------------------------------------------------------ launch bookkeeping
const char* const kFamNames[DF_PROF_FAMILIES] = {"norm", "qkv", "attention", "o_proj", "gate_up", "down", "lm_head",
                                                 "other"};

// Counts every kernel the step launches by family. Profiling mode 1 brackets each launch with a
// CUDA event pair on the launching stream (external event nodes when the step is being captured,
// so the replayed graph records them; this serialises the launches). Mode 2 gives each launch a
// stamp slot that its CTAs raise to the globaltimer value at their end (no serialisation). With
// NVTX on, each launch is a named range (host side: eager launches, or the capture).
struct Launcher {
  dualflow_ctx* ctx;
  cudaStream_t s;
  template <class F>
  int operator()(int fam, F&& f) {
    ctx->step_launches[fam]++;
    ProfRec* r = nullptr;
    if (ctx->profiling == 1 && ctx->prof_n < (int)ctx->prof.size()) {
      r = &ctx->prof[ctx->prof_n++];
      r->fam = fam;
      if (cudaEventRecordWithFlags(r->a, s, cudaEventRecordExternal) != cudaSuccess) return DF_ERR_CUDA;
    } else if (ctx->profiling == 2 && ctx->prof_n < (int)ctx->prof_fam.size()) {
      ctx->prof_fam[ctx->prof_n] = fam;
      ctx->cur_stamp = ctx->stamps + 1 + ctx->prof_n;
      ctx->prof_n++;
    }
    if (ctx->nvtx) nvtxRangePushA(kFamNames[fam]);
    const int rc = f();
    if (ctx->nvtx) nvtxRangePop();
    ctx->cur_stamp = nullptr;
    if (r && cudaEventRecordWithFlags(r->b, s, cudaEventRecordExternal) != cudaSuccess) return DF_ERR_CUDA;
    return rc;
  }
};

int reset_counts(dualflow_ctx* ctx, cudaStream_t s) {
  for (int& n : ctx->step_launches) n = 0;
  ctx->prof_n = 0;
  ctx->cur_stamp = nullptr;
  // mode 2: the step's start slot is lowered by its first kernel from the largest value
  if (ctx->profiling == 2 && cudaMemsetAsync(ctx->stamps, 0xff, sizeof(unsigned long long), s) != cudaSuccess)
    return DF_ERR_CUDA;
  return DF_OK;
}

// NVTX range for one layer of the step (host side), closed on scope exit.
struct LayerRange {
  bool on;
  LayerRange(const dualflow_ctx* ctx, int l) : on(ctx->nvtx != 0) {
    if (on) {
      char name[32];
      snprintf(name, sizeof(name), "layer %d", l);
      nvtxRangePushA(name);
    }
  }
  ~LayerRange() {
    if (on) nvtxRangePop();
  }
};

// ------------------------------------------------------------------ the MoE MLP (bf16)
// x (the norm-fed operand, rows scaled by 1 / rms from ss_parts partials) -> router logits ->
// routing decision -> every expert's gate/up for the rows that chose it -> every expert's down ->
// combine with output coupling and residual into h (and, with g_next, the next norm's operand).
int run_moe(dualflow_ctx* ctx, float* h, const dualflow_weights* w, int l, int batch, int aux_on, int ss_parts,
            int32_t* ids, const void* g_next, int pdl, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  const int mp = batch, ma = aux_on ? batch : 0, E = c.n_experts, mrows = 2 * c.max_batch;
  Launcher L{ctx, s};
  auto normed = [&](GemmArgs& g) {
    g.ss_in = ctx->ss;
    g.ss_parts = ss_parts;
    g.ss_ld = ctx->ss_ld;
    g.inv_d = 1.0f / (float)c.d_model;
    g.eps = c.rms_eps;
    g.pdl = pdl;
  };
  // this layer's router logits, kept per layer for dualflow_router_logits
  float* rlog = ctx->rlog + (size_t)l * mrows * E;
  GemmArgs r = gemm_args(ctx);
  r.x = ctx->x;
  r.W = w->Wr[l];
  r.n_out = E;
  r.k = c.d_model;
  r.m_p = mp;
  r.m_a = ma;
  r.epi = EPI_STORE_F32;
  r.y = rlog;
  r.ldy = E;
  normed(r);
  DF_TRY(L(DF_PROF_GATEUP, [&] { return launch_gemm_tc(ctx, r, s); }));
  DF_TRY(L(DF_PROF_GATEUP, [&] { return launch_moe_route(ctx, rlog, batch, aux_on, ids, s, pdl); }));
  GemmArgs g = gemm_args(ctx);
  g.x = ctx->x;
  g.W = w->We_gu[l];
  g.n_out = c.ffn_hidden;
  g.k = c.d_model;
  g.m_p = mp;
  g.m_a = ma;
  g.epi = EPI_MOE_GATEUP;
  g.y = ctx->moe_u;
  g.ldy = c.ffn_hidden;
  g.vec = w->b[l];
  g.n_groups = E;
  g.w_group_rows = 2 * c.ffn_hidden;
  g.y_group_stride = (size_t)mrows * c.ffn_hidden;
  g.sel_pos = ctx->sel_pos;
  normed(g);
  DF_TRY(L(DF_PROF_GATEUP, [&] { return launch_gemm_tc(ctx, g, s); }));
  GemmArgs d = gemm_args(ctx);
  d.x = ctx->moe_u;
  d.W = w->We_d[l];
  d.n_out = c.d_model;
  d.k = c.ffn_hidden;
  d.m_p = mp;
  d.m_a = ma;
  d.epi = EPI_MOE_DOWN;
  d.y = ctx->moe_y;
  d.ldy = c.d_model;
  d.n_groups = E;
  d.w_group_rows = c.d_model;
  d.x_group_rows = mrows;
  d.y_group_stride = (size_t)mrows * c.d_model;
  d.sel_pos = ctx->sel_pos;
  d.pdl = pdl;
  DF_TRY(L(DF_PROF_DOWN, [&] { return launch_gemm_tc(ctx, d, s); }));
  return L(DF_PROF_DOWN, [&] { return launch_moe_combine(ctx, h, batch, aux_on, w->c[l], g_next, s, pdl); });
}

// ------------------------------------------------------------------ the MLP block
int run_mlp(dualflow_ctx* ctx, float* h, const dualflow_weights* w, int l, int batch, int aux_on, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  const int mp = batch, ma = aux_on ? batch : 0;
  Launcher L{ctx, s};
  if (c.dtype == DF_DTYPE_BF16 && c.n_experts > 0) {
    DF_TRY(L(DF_PROF_NORM, [&] { return launch_norm_prep(ctx, h, w->g_mlp[l], batch, aux_on, s); }));
    const int kmax = std::max(c.topk_primary, c.topk_aux);
    int32_t* ids = ctx->moe_ids + (size_t)l * 2 * batch * kmax;
    DF_TRY(run_moe(ctx, h, w, l, batch, aux_on, 1, ids, nullptr, 0, s));
    return DF_OK;
  }
  if (c.dtype == DF_DTYPE_BF16) {
    // x = bf16(h (*) g_mlp) with per-row sums of squares; gate/up scales its rows by 1 / rms
    DF_TRY(L(DF_PROF_NORM, [&] { return launch_norm_prep(ctx, h, w->g_mlp[l], batch, aux_on, s); }));
    GemmArgs g = gemm_args(ctx);
    g.ss_in = ctx->ss;
    g.ss_parts = 1;
    g.ss_ld = ctx->ss_ld;
    g.inv_d = 1.0f / (float)c.d_model;
    g.eps = c.rms_eps;
    g.x = ctx->x;
    g.W = w->Wgu[l];
    g.n_out = c.ffn_hidden;
    g.k = c.d_model;
    g.m_p = mp;
    g.m_a = ma;
    g.epi = EPI_SWIGLU;
    g.y = ctx->u;
    g.ldy = c.ffn_hidden;
    g.vec = w->b[l];
    DF_TRY(L(DF_PROF_GATEUP, [&] { return launch_gemm_tc(ctx, g, s); }));
    GemmArgs d = gemm_args(ctx);
    d.x = ctx->u;
    d.W = w->Wd[l];
    d.n_out = c.d_model;
    d.k = c.ffn_hidden;
    d.m_p = mp;
    d.m_a = ma;
    d.epi = EPI_COUPLE_ADD;
    d.y = h;
    d.ldy = c.d_model;
    d.vec = w->c[l];
    return L(DF_PROF_DOWN, [&] { return launch_gemm_tc(ctx, d, s); });
  }
  const int M = mp + ma, F = c.ffn_hidden;
  DF_TRY(L(DF_PROF_NORM, [&] { return launch_rmsnorm(ctx, h, w->g_mlp[l], ctx->x, batch, aux_on, s); }));
  DF_TRY(L(DF_PROF_GATEUP, [&] {
    return launch_linear_f32(ctx, (const float*)ctx->x, M, (const float*)w->Wgu[l], 2 * F, c.d_model, ctx->raw, 0, s);
  }));
  DF_TRY(L(DF_PROF_OTHER,
           [&] { return launch_swiglu_f32(ctx, ctx->raw, batch, aux_on, (const float*)w->b[l], (float*)ctx->u, s); }));
  DF_TRY(L(DF_PROF_DOWN, [&] {
    return launch_linear_f32(ctx, (const float*)ctx->u, M, (const float*)w->Wd[l], c.d_model, F, ctx->raw, 0, s);
  }));
  return L(DF_PROF_OTHER, [&] {
    return launch_couple_add_f32(ctx, ctx->raw, batch, aux_on, c.d_model, (const float*)w->c[l], h, s);
  });
}

// ------------------------------------------------------------------ the whole step
// bf16: five kernels per layer. RMSNorm is carried between kernels (see gemm_tc.cu): the residual
// epilogues (O projection, down projection) and the embedding kernel write x = bf16(h (*) g) and
// per-tile row sums of h^2; the next projection scales its rows by 1 / rms. Every kernel after the
// first is launched with programmatic dependent launch, so it becomes resident and starts
// streaming its weights while its predecessor drains.
int run_step_bf16(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv, const int32_t* tokens,
                  int batch, float* logits, int aux_on, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  const int mp = batch, ma = aux_on ? batch : 0;
  const int qkv_n = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim, qd = c.n_q_heads * c.head_dim;
  const int d_tiles = (c.d_model + kGemmTileN - 1) / kGemmTileN;
  const int ss_ld = ctx->ss_ld;
  // row sums of squares left by the O projection and by the down projection: one per CTA
  const int o_parts = d_tiles * gemm_splits(ctx, c.d_model, qd, EPI_ADD_F32);
  const int kmax = std::max(c.topk_primary, c.topk_aux);
  const int d_parts = d_tiles * gemm_splits(ctx, c.d_model, c.ffn_hidden, EPI_COUPLE_ADD);
  Launcher L{ctx, s};
  DF_TRY(L(DF_PROF_NORM, [&] {
    return launch_embed_prep(ctx, w->E1, w->E2, tokens, c.n_layers > 0 ? w->g_attn[0] : w->g_final, batch, aux_on,
                             s);
  }));
  // programmatic dependent launch on explicit streams (the legacy default stream keeps plain order)
  const int pdl = s != nullptr ? 1 : 0;
  int ss_parts = 1;  // partial sums of squares behind the rows currently in ctx->x
  auto normed_input = [&](GemmArgs& g) {
    g.ss_in = ctx->ss;
    g.ss_parts = ss_parts;
    g.ss_ld = ss_ld;
    g.inv_d = 1.0f / (float)c.d_model;
    g.eps = c.rms_eps;
    g.pdl = pdl;
  };
  auto norm_output = [&](GemmArgs& g, const void* g_next) {
    g.g_next = g_next;
    g.x_next = ctx->x;
    g.ss_out = ctx->ss;
    g.ss_ld = ss_ld;
    g.pdl = pdl;
  };
  // the projection that follows (weights, shape, epilogue): its first k-blocks are warmed in L2
  auto prefetch = [&](GemmArgs& cur, const void* W, int n_out, int k, int epi) {
    GemmArgs nx = gemm_args(ctx);
    nx.W = W;
    nx.n_out = n_out;
    nx.k = k;
    nx.epi = epi;
    gemm_prefetch_next(ctx, cur, nx);
  };
  for (int l = 0; l < c.n_layers; ++l) {
    LayerRange range(ctx, l);
    GemmArgs g = gemm_args(ctx);
    g.x = ctx->x;
    g.W = w->Wqkv[l];
    g.n_out = qkv_n;
    g.k = c.d_model;
    g.m_p = mp;
    g.m_a = ma;
    g.epi = EPI_QKV;
    g.vec = w->a[l];
    g.q_out = ctx->q;
    g.seq_len = kv->seq_len;
    g.k_cache = kv->k[l];
    g.v_cache = kv->v[l];
    g.page_table = kv->page_table;
    normed_input(g);
    DF_TRY(L(DF_PROF_QKV, [&] { return launch_gemm_tc(ctx, g, s); }));
    const AttnArgs at = attn_args(ctx, kv, l, batch, 1, aux_on);
    DF_TRY(L(DF_PROF_ATTN, [&] { return launch_attention_bf16(ctx, at, s, pdl); }));
    GemmArgs o = gemm_args(ctx);
    o.x = ctx->o;
    o.W = w->Wo[l];
    o.n_out = c.d_model;
    o.k = qd;
    o.m_p = mp;
    o.m_a = ma;
    o.epi = EPI_ADD_F32;
    o.y = ctx->h;
    o.ldy = c.d_model;
    norm_output(o, w->g_mlp[l]);
    if (c.n_experts == 0) prefetch(o, w->Wgu[l], c.ffn_hidden, c.d_model, EPI_SWIGLU);
    DF_TRY(L(DF_PROF_OPROJ, [&] { return launch_gemm_tc(ctx, o, s); }));
    ss_parts = o_parts;
    const void* g_next = l + 1 < c.n_layers ? w->g_attn[l + 1] : w->g_final;
    if (c.n_experts > 0) {
      int32_t* ids = ctx->moe_ids + (size_t)l * 2 * batch * kmax;
      DF_TRY(run_moe(ctx, ctx->h, w, l, batch, aux_on, ss_parts, ids, g_next, pdl, s));
      ss_parts = (c.d_model + 511) / 512;
      continue;
    }
    GemmArgs gu = gemm_args(ctx);
    gu.x = ctx->x;
    gu.W = w->Wgu[l];
    gu.n_out = c.ffn_hidden;
    gu.k = c.d_model;
    gu.m_p = mp;
    gu.m_a = ma;
    gu.epi = EPI_SWIGLU;
    gu.y = ctx->u;
    gu.ldy = c.ffn_hidden;
    gu.vec = w->b[l];
    normed_input(gu);
    prefetch(gu, w->Wd[l], c.d_model, c.ffn_hidden, EPI_COUPLE_ADD);
    DF_TRY(L(DF_PROF_GATEUP, [&] { return launch_gemm_tc(ctx, gu, s); }));
    GemmArgs dn = gemm_args(ctx);
    dn.x = ctx->u;
    dn.W = w->Wd[l];
    dn.n_out = c.d_model;
    dn.k = c.ffn_hidden;
    dn.m_p = mp;
    dn.m_a = ma;
    dn.epi = EPI_COUPLE_ADD;
    dn.y = ctx->h;
    dn.ldy = c.d_model;
    dn.vec = w->c[l];
    norm_output(dn, g_next);
    if (l + 1 < c.n_layers)
      prefetch(dn, w->Wqkv[l + 1], qkv_n, c.d_model, EPI_QKV);
    else
      prefetch(dn, w->W_lm, c.vocab, c.d_model, EPI_STORE_F32);
    DF_TRY(L(DF_PROF_DOWN, [&] { return launch_gemm_tc(ctx, dn, s); }));
    ss_parts = d_parts;
  }
  GemmArgs g = gemm_args(ctx);
  g.x = ctx->x;
  g.W = w->W_lm;
  g.n_out = c.vocab;
  g.k = c.d_model;
  g.m_p = mp;
  g.m_a = ma;
  g.epi = EPI_STORE_F32;
  g.y = logits;
  g.ldy = c.vocab;
  normed_input(g);
  return L(DF_PROF_LMHEAD, [&] { return launch_gemm_tc(ctx, g, s); });
}

int run_step(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv, const int32_t* tokens, int batch,
             float* logits, int aux_on, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  DF_TRY(reset_counts(ctx, s));
  if (c.dtype == DF_DTYPE_BF16) return run_step_bf16(ctx, w, kv, tokens, batch, logits, aux_on, s);
  const int mp = batch, ma = aux_on ? batch : 0, M = mp + ma;
  const int qkv_n = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim, qd = c.n_q_heads * c.head_dim;
  Launcher L{ctx, s};
  DF_TRY(L(DF_PROF_NORM, [&] {
    return launch_embed_rmsnorm(ctx, w->E1, w->E2, tokens, c.n_layers > 0 ? w->g_attn[0] : w->g_final, batch,
                                aux_on, s);
  }));
  for (int l = 0; l < c.n_layers; ++l) {
    if (l > 0)
      DF_TRY(L(DF_PROF_NORM, [&] { return launch_rmsnorm(ctx, ctx->h, w->g_attn[l], ctx->x, batch, aux_on, s); }));
    DF_TRY(L(DF_PROF_QKV, [&] {
      return launch_linear_f32(ctx, (const float*)ctx->x, M, (const float*)w->Wqkv[l], qkv_n, c.d_model, ctx->raw,
                               0, s);
    }));
    DF_TRY(L(DF_PROF_OTHER, [&] {
      return launch_qkv_post_f32(ctx, ctx->raw, batch, aux_on, (const float*)w->a[l], kv->k[l], kv->v[l],
                                 kv->page_table, kv->seq_len, (float*)ctx->q, s);
    }));
    DF_TRY(L(DF_PROF_ATTN, [&] {
      return launch_attention_f32(ctx, (const float*)ctx->q, (float*)ctx->o, kv->k[l], kv->v[l], kv->page_table,
                                  kv->seq_len, batch, 1, aux_on, s);
    }));
    DF_TRY(L(DF_PROF_OPROJ, [&] {
      return launch_linear_f32(ctx, (const float*)ctx->o, M, (const float*)w->Wo[l], c.d_model, qd, ctx->h, 1, s);
    }));
    DF_TRY(run_mlp(ctx, ctx->h, w, l, batch, aux_on, s));
  }
  DF_TRY(L(DF_PROF_NORM, [&] { return launch_rmsnorm(ctx, ctx->h, w->g_final, ctx->x, batch, aux_on, s); }));
  return L(DF_PROF_LMHEAD, [&] {
    return launch_linear_f32(ctx, (const float*)ctx->x, M, (const float*)w->W_lm, c.vocab, c.d_model, logits, 0, s);
  });
}

void graph_key(std::vector<uint64_t>& k, const dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv,
               const int32_t* tokens, int batch, const float* logits, int aux_on, cudaStream_t s) {
  const int L = ctx->cfg.n_layers;
  auto P = [&](const void* p) { k.push_back(reinterpret_cast<uint64_t>(p)); };
  P(s);
  P(tokens);
  P(logits);
  k.push_back((uint64_t)batch);
  k.push_back((uint64_t)aux_on);
  k.push_back((uint64_t)ctx->profiling);
  k.push_back((uint64_t)ctx->wait_ns);
  P(w->E1), P(w->E2), P(w->W_lm), P(w->g_final);
  P(kv->seq_len), P(kv->page_table);
  for (int l = 0; l < L; ++l) {
    P(w->g_attn[l]), P(w->g_mlp[l]), P(w->Wqkv[l]), P(w->Wo[l]), P(w->a[l]), P(w->b[l]), P(w->c[l]);
    P(w->Wgu ? w->Wgu[l] : nullptr), P(w->Wd ? w->Wd[l] : nullptr);
    P(w->Wr ? w->Wr[l] : nullptr), P(w->We_gu ? w->We_gu[l] : nullptr), P(w->We_d ? w->We_d[l] : nullptr);
    P(kv->k[l]), P(kv->v[l]);
  }
}

void drop_graphs(dualflow_ctx* ctx) {
  for (auto& g : ctx->graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  ctx->graphs.clear();
}

// The MoE MLP of a prefill layer, primary flow only, on the R prompt rows (x = the norm operand
// with ss_parts partial sums of squares per row, in the context's prefill buffers): router logits,
// the top-k decision, every row gathered once per chosen expert (expert-major), each expert's
// gate/up + SwiGLU and down projection on its own rows only (row-blocked tcgen05 launches over
// the gathered blocks), then the mix in set order with the residual and the next layer's norm
// operand. The same arithmetic per row as the decode step's MoE MLP for the primary flow.
int prefill_moe(dualflow_ctx* ctx, const dualflow_weights* w, int l, int R, int ss_parts, cudaStream_t s) {
  const dualflow_config& c = ctx->cfg;
  const int E = c.n_experts, RK = R * c.topk_primary, d = c.d_model, F = c.ffn_hidden;
  auto scaled = [&](GemmArgs& g, const float* ss) {
    g.ss_in = ss;
    g.ss_parts = ss_parts;
    g.ss_ld = ctx->ss_ld;
    g.inv_d = 1.0f / (float)d;
    g.eps = c.rms_eps;
  };
  GemmArgs r = gemm_args(ctx);
  r.x = ctx->x;
  r.W = w->Wr[l];
  r.n_out = E;
  r.k = d;
  r.m_p = R;
  r.row_blocked = 1;
  r.seq_rows = 1;
  r.epi = EPI_STORE_F32;
  r.y = ctx->pf_rlog;
  r.ldy = E;
  scaled(r, ctx->ss);
  DF_TRY(launch_gemm_tc(ctx, r, s));
  DF_TRY(launch_moe_route_rows(c, ctx->pf_rlog, R, ctx->pf_sel_pos, ctx->pf_sel_w, s));
  DF_TRY(launch_moe_plan(c, R, ctx->pf_sel_pos, ctx->pf_perm, ctx->pf_pos, ctx->pf_blk, ctx->pf_nblk, ctx->status, s));
  DF_TRY(launch_moe_gather(RK, R, d, ctx->x, ctx->ss, ctx->ss_ld, ctx->pf_perm, ctx->pf_xg, ctx->pf_ssg, ctx->status,
                           s));
  auto gathered = [&](GemmArgs& g) {
    g.m_p = RK;
    g.row_blocked = 1;
    g.seq_rows = 1;
    g.n_groups = E;
    g.blk_info = ctx->pf_blk;
    g.n_blk = ctx->pf_nblk;
  };
  GemmArgs gu = gemm_args(ctx);
  gu.x = ctx->pf_xg;
  gu.W = w->We_gu[l];
  gu.n_out = F;
  gu.k = d;
  gu.epi = EPI_SWIGLU;
  gu.y = ctx->pf_ug;
  gu.ldy = F;
  gu.vec = w->b[l];
  gu.w_group_rows = 2 * F;
  gathered(gu);
  scaled(gu, ctx->pf_ssg);
  DF_TRY(launch_gemm_tc(ctx, gu, s));
  GemmArgs dn = gemm_args(ctx);
  dn.x = ctx->pf_ug;
  dn.W = w->We_d[l];
  dn.n_out = d;
  dn.k = F;
  dn.epi = EPI_STORE_F32;
  dn.y = ctx->pf_yg;
  dn.ldy = d;
  dn.w_group_rows = d;
  gathered(dn);
  DF_TRY(launch_gemm_tc(ctx, dn, s));
  const void* g_next = l + 1 < c.n_layers ? w->g_attn[l + 1] : nullptr;
  return launch_moe_combine_rows(c, R, ctx->pf_yg, ctx->pf_sel_pos, ctx->pf_sel_w, ctx->pf_pos, ctx->h, g_next, ctx->x,
                                 ctx->ss, ctx->ss_ld, ctx->status, s);
}

// Frees the prefill MoE workspace (nullptr-safe).
void free_prefill_moe(dualflow_ctx* ctx) {
  void* ps[] = {ctx->pf_rlog, ctx->pf_sel_pos, ctx->pf_sel_w, ctx->pf_perm, ctx->pf_pos, ctx->pf_xg,
                ctx->pf_ssg,  ctx->pf_ug,      ctx->pf_yg,    ctx->pf_blk,  ctx->pf_nblk};
  for (void* p : ps)
    if (p) cudaFree(p);
  ctx->pf_rlog = ctx->pf_sel_w = ctx->pf_ssg = ctx->pf_yg = nullptr;
  ctx->pf_sel_pos = ctx->pf_perm = ctx->pf_pos = ctx->pf_nblk = nullptr;
  ctx->pf_xg = ctx->pf_ug = nullptr;
  ctx->pf_blk = nullptr;
}

}  // namespace

// ================================================================== C ABI
extern "C" {

const char* dualflow_cuda_error_string(void) {
  const cudaError_t e = cudaPeekAtLastError();
  if (e != cudaSuccess || df::t_driver_error[0] == 0) return cudaGetErrorString(e);
  return df::t_driver_error;
}

const char* dualflow_status_string(int st) {
  switch (st) {
    case DF_OK: return "ok";
    case DF_ERR_ARG: return "invalid argument";
    case DF_ERR_SHAPE: return "shape inconsistent with the config";
    case DF_ERR_DTYPE: return "unknown storage dtype";
    case DF_ERR_UNSUPPORTED: return "configuration not supported by this library";
    case DF_ERR_CUDA: return "CUDA runtime error";
    case DF_ERR_OOM: return "device allocation failed";
    case DF_ERR_DEVICE_BOUNDS: return "device-side bounds check failed (page id, token or cache slot)";
    case DF_ERR_TIMEOUT: return "bounded device wait expired";
    default: return "unknown status";
  }
}

int dualflow_init(const dualflow_config* cfg, dualflow_ctx** out) {
  if (!out) return DF_ERR_ARG;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc != DF_OK) return rc;
  dualflow_ctx* ctx = new dualflow_ctx();
  ctx->cfg = *cfg;
  const dualflow_config& c = ctx->cfg;
  auto fail = [&](int code) {
    dualflow_free(ctx);
    return code;
  };
  if (cudaGetDevice(&ctx->device) != cudaSuccess) return fail(DF_ERR_CUDA);
  if (cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess)
    return fail(DF_ERR_CUDA);
  const size_t es = elem_size(c);
  const int MB = 2 * c.max_batch;
  const int half = c.head_dim / 2;
  const int qkv_n = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim, qd = c.n_q_heads * c.head_dim;
  // RoPE table in fp64 on the host, stored fp32: (cos, sin)(pos * base^(-2i/D)), pos = 0..max_ctx
  {
    std::vector<float2> tab((size_t)(c.max_ctx + 1) * half);
    for (int p = 0; p <= c.max_ctx; ++p)
      for (int i = 0; i < half; ++i) {
        const double ang = (double)p * pow((double)c.rope_base, -2.0 * i / c.head_dim);
        tab[(size_t)p * half + i] = make_float2((float)cos(ang), (float)sin(ang));
      }
    if (dalloc(&ctx->rope, tab.size() * sizeof(float2)) != DF_OK) return fail(DF_ERR_OOM);
    if (cudaMemcpy(ctx->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
      return fail(DF_ERR_CUDA);
  }
  if (dalloc(&ctx->status, sizeof(int32_t)) != DF_OK) return fail(DF_ERR_OOM);
  if (dalloc(&ctx->gen_tokens, (size_t)c.max_batch * sizeof(int32_t)) != DF_OK) return fail(DF_ERR_OOM);
  if (dalloc(&ctx->gen_out_dev, (size_t)kGenHostMaxSteps * c.max_batch * sizeof(int32_t)) != DF_OK)
    return fail(DF_ERR_OOM);
  if (dalloc(&ctx->gen_u_dev, (size_t)kGenHostMaxSteps * c.max_batch * sizeof(float)) != DF_OK)
    return fail(DF_ERR_OOM);
  cudaMemset(ctx->status, 0, sizeof(int32_t));
  // decode attention: persistent grid of 2 CTAs per SM; partial slots = pairs + CTAs
  ctx->attn_ctas = 2 * ctx->num_sms;
  const int pairs = c.max_batch * c.n_kv_heads;
  ctx->attn_slots = pairs + ctx->attn_ctas;
  if (dalloc(&ctx->attn_part, (size_t)ctx->attn_slots * kAttnPartFloats * sizeof(float)) != DF_OK)
    return fail(DF_ERR_OOM);
  if (dalloc(&ctx->attn_cnt, (size_t)pairs * sizeof(int32_t)) != DF_OK) return fail(DF_ERR_OOM);
  cudaMemset(ctx->attn_cnt, 0, (size_t)pairs * sizeof(int32_t));
  ctx->gemm_part_floats = df::gemm_part_floats(ctx);
  if (ctx->gemm_part_floats > 0 && dalloc(&ctx->gemm_part, ctx->gemm_part_floats * sizeof(float)) != DF_OK)
    return fail(DF_ERR_OOM);
  const size_t xw = std::max({c.d_model, c.ffn_hidden, qd});
  const size_t raw_n = std::max({qkv_n, 2 * c.ffn_hidden, c.d_model, c.vocab, qd});
  if (dalloc(&ctx->h, (size_t)MB * c.d_model * sizeof(float)) != DF_OK) return fail(DF_ERR_OOM);
  if (dalloc(&ctx->x, (size_t)MB * xw * es) != DF_OK) return fail(DF_ERR_OOM);
  if (dalloc(&ctx->q, (size_t)MB * qd * es) != DF_OK) return fail(DF_ERR_OOM);
  if (dalloc(&ctx->o, (size_t)MB * qd * es) != DF_OK) return fail(DF_ERR_OOM);
  if (dalloc(&ctx->u, (size_t)MB * std::max(c.ffn_hidden, 1) * es) != DF_OK) return fail(DF_ERR_OOM);
  if (c.dtype == DF_DTYPE_F32 && dalloc(&ctx->raw, (size_t)MB * raw_n * sizeof(float)) != DF_OK)
    return fail(DF_ERR_OOM);
  ctx->ss_ld = 8 * ((c.d_model + kGemmTileN - 1) / kGemmTileN);
  if (dalloc(&ctx->ss, (size_t)ctx->ss_ld * MB * sizeof(float)) != DF_OK) return fail(DF_ERR_OOM);
  if (c.n_experts > 0) {
    const size_t E = c.n_experts, kmax = std::max(c.topk_primary, c.topk_aux);
    if (dalloc(&ctx->rlog, (size_t)std::max(c.n_layers, 1) * MB * E * sizeof(float)) != DF_OK) return fail(DF_ERR_OOM);
    if (dalloc(&ctx->sel_pos, MB * E * sizeof(int32_t)) != DF_OK) return fail(DF_ERR_OOM);
    if (dalloc(&ctx->sel_w, MB * E * sizeof(float)) != DF_OK) return fail(DF_ERR_OOM);
    if (dalloc(&ctx->moe_u, E * MB * c.ffn_hidden * es) != DF_OK) return fail(DF_ERR_OOM);
    if (dalloc(&ctx->moe_y, E * MB * c.d_model * sizeof(float)) != DF_OK) return fail(DF_ERR_OOM);
    if (dalloc(&ctx->moe_ids, (size_t)std::max(c.n_layers, 1) * MB * kmax * sizeof(int32_t)) != DF_OK)
      return fail(DF_ERR_OOM);
    // expert intermediates of rows that did not choose an expert are read (and ignored) by that
    // expert's down projection: start them at zero
    if (cudaMemset(ctx->moe_u, 0, E * MB * c.ffn_hidden * es) != cudaSuccess) return fail(DF_ERR_CUDA);
    if (cudaMemset(ctx->moe_ids, 0xff, (size_t)std::max(c.n_layers, 1) * MB * kmax * sizeof(int32_t)) != cudaSuccess)
      return fail(DF_ERR_CUDA);
  }
  if (dalloc(&ctx->tokens_dev, (size_t)c.max_batch * sizeof(int32_t)) != DF_OK) return fail(DF_ERR_OOM);
  if (dalloc(&ctx->logits_dev, (size_t)MB * std::max(c.vocab, 1) * sizeof(float)) != DF_OK) return fail(DF_ERR_OOM);
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(DF_ERR_CUDA);
  *out = ctx;
  return DF_OK;
}

int dualflow_free(dualflow_ctx* ctx) {
  if (!ctx) return DF_OK;
  cudaDeviceSynchronize();
  drop_graphs(ctx);
  for (auto& r : ctx->prof) {
    if (r.a) cudaEventDestroy(r.a);
    if (r.b) cudaEventDestroy(r.b);
  }
  if (ctx->stamps) cudaFree(ctx->stamps);
  void* ptrs[] = {ctx->status, ctx->rope, ctx->attn_part, ctx->attn_cnt, ctx->h,
                  ctx->x,      ctx->q,    ctx->o,         ctx->u,        ctx->raw,       ctx->tokens_dev, ctx->logits_dev, ctx->ss,
                  ctx->rlog, ctx->sel_pos, ctx->sel_w, ctx->moe_u, ctx->moe_y, ctx->moe_ids, ctx->gen_tokens, ctx->gen_out_dev, ctx->gen_u_dev,
                  ctx->pf_h,   ctx->pf_x,    ctx->pf_q,      ctx->pf_o,     ctx->pf_u,     ctx->pf_ss, ctx->gemm_part};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  free_prefill_moe(ctx);
  delete ctx;
  return DF_OK;
}

int dualflow_decode_attention(dualflow_ctx* ctx, const void* q1, const void* h2, const void* Wq, const void* a,
                              const dualflow_kv* kv, int32_t layer, int32_t batch, void* o, int32_t aux_on,
                              dualflow_stream stream) {
  if (!ctx || !q1 || !o) return DF_ERR_ARG;
  if (aux_on != 0 && aux_on != 1) return DF_ERR_ARG;
  if (aux_on && (!h2 || !Wq || !a)) return DF_ERR_ARG;
  if (!aligned16(q1) || (aux_on && (!aligned16(h2) || !aligned16(Wq) || !aligned16(a)))) return DF_ERR_ARG;
  if (batch <= 0 || batch > ctx->cfg.max_batch) return DF_ERR_SHAPE;
  DF_TRY(check_kv(ctx, kv, layer));
  const dualflow_config& c = ctx->cfg;
  cudaStream_t s = S(stream);
  if (c.dtype == DF_DTYPE_BF16) {
    // On a caller's stream the attention is chained to the call's first launch by programmatic
    // dependent launch, as in the step: it requests its first K/V stages while the query
    // projection runs. The first launch itself waits for the caller's preceding work in the usual
    // way (unless the caller enabled chaining), so nothing this call reads early (weights, cached
    // K/V) can be older than that work.
    const int pdl = s != nullptr ? 1 : 0;
    if (aux_on) {
      GemmArgs g = gemm_args(ctx);
      g.pdl = ctx->chain_calls ? pdl : 0;
      g.x = h2;
      g.W = Wq;
      g.n_out = c.n_q_heads * c.head_dim;
      g.k = c.d_model;
      g.m_p = 0;
      g.m_a = batch;
      g.epi = EPI_Q2;
      g.vec = a;
      g.q_out = ctx->q;
      g.q1_in = q1;
      g.seq_len = kv->seq_len;
      DF_TRY(launch_gemm_tc(ctx, g, s));
    } else {
      DF_TRY(launch_rope_q1(ctx, q1, ctx->q, kv->seq_len, batch, s));
    }
    AttnArgs at = attn_args(ctx, kv, layer, batch, 0, aux_on);
    at.o = o;
    return launch_attention_bf16(ctx, at, s, pdl);
  }
  if (aux_on)
    DF_TRY(launch_linear_f32(ctx, (const float*)h2, batch, (const float*)Wq, c.n_q_heads * c.head_dim, c.d_model,
                             ctx->raw, 0, s));
  DF_TRY(launch_q2_post_f32(ctx, ctx->raw, (const float*)q1, batch, aux_on, (const float*)a, kv->seq_len,
                            (float*)ctx->q, s));
  return launch_attention_f32(ctx, (const float*)ctx->q, (float*)o, kv->k[layer], kv->v[layer], kv->page_table,
                              kv->seq_len, batch, 0, aux_on, s);
}

int dualflow_stacked_linear(dualflow_ctx* ctx, const void* x, int32_t m_primary, int32_t m_aux, const void* W,
                            int32_t n, int32_t k, void* y, int32_t epilogue, const void* epi_arg,
                            dualflow_stream stream) {
  if (!ctx || !x || !W || !y) return DF_ERR_ARG;
  if (m_primary < 0 || m_aux < 0 || m_primary + m_aux <= 0 || n <= 0 || k <= 0) return DF_ERR_ARG;
  if (epilogue < DF_EPI_STORE_F32 || epilogue > DF_EPI_COUPLE_ADD) return DF_ERR_ARG;
  if (epilogue == DF_EPI_COUPLE_ADD && (!epi_arg || (m_aux != 0 && m_aux != m_primary))) return DF_ERR_ARG;
  if (epilogue == DF_EPI_COUPLE_ADD && !aligned16(epi_arg)) return DF_ERR_ARG;
  const dualflow_config& c = ctx->cfg;
  cudaStream_t s = S(stream);
  if (c.dtype == DF_DTYPE_BF16) {
    if (k % 64 != 0 || m_primary + m_aux > kGemmMaxAct) return DF_ERR_SHAPE;
    GemmArgs g = gemm_args(ctx);
    g.x = x;
    g.W = W;
    g.n_out = n;
    g.k = k;
    g.m_p = m_primary;
    g.m_a = m_aux;
    g.y = y;
    g.ldy = n;
    g.vec = epi_arg;
    g.epi = epilogue == DF_EPI_STORE_F32 ? EPI_STORE_F32
            : epilogue == DF_EPI_STORE_BF16 ? EPI_STORE_BF16
            : epilogue == DF_EPI_ADD_F32 ? EPI_ADD_F32
                                          : EPI_COUPLE_ADD;
    return launch_gemm_tc(ctx, g, s);
  }
  const int M = m_primary + m_aux;
  if ((size_t)M * n > (size_t)2 * c.max_batch * std::max({(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim,
                                                            2 * c.ffn_hidden, c.d_model, c.vocab}))
    return DF_ERR_SHAPE;
  if (epilogue == DF_EPI_STORE_F32 || epilogue == DF_EPI_STORE_BF16)
    return launch_linear_f32(ctx, (const float*)x, M, (const float*)W, n, k, (float*)y, 0, s);
  if (epilogue == DF_EPI_ADD_F32) return launch_linear_f32(ctx, (const float*)x, M, (const float*)W, n, k, (float*)y, 1, s);
  DF_TRY(launch_linear_f32(ctx, (const float*)x, M, (const float*)W, n, k, ctx->raw, 0, s));
  return launch_couple_add_f32(ctx, ctx->raw, m_primary, m_aux > 0, n, (const float*)epi_arg, (float*)y, s);
}

int dualflow_coupled_mlp(dualflow_ctx* ctx, float* h, const dualflow_weights* w, int32_t layer, int32_t batch,
                         int32_t aux_on, int32_t* expert_ids_out, dualflow_stream stream) {
  if (!ctx || !h || !w || !aligned16(h)) return DF_ERR_ARG;
  if (aux_on != 0 && aux_on != 1) return DF_ERR_ARG;
  if (batch <= 0 || batch > ctx->cfg.max_batch) return DF_ERR_SHAPE;
  if (layer < 0 || layer >= ctx->cfg.n_layers) return DF_ERR_ARG;
  DF_TRY(check_weights(ctx, w));
  DF_TRY(reset_counts(ctx, S(stream)));
  DF_TRY(run_mlp(ctx, h, w, layer, batch, aux_on, S(stream)));
  const dualflow_config& c = ctx->cfg;
  if (expert_ids_out && c.n_experts > 0) {
    const size_t kmax = std::max(c.topk_primary, c.topk_aux), n = 2 * (size_t)batch * kmax;
    if (cudaMemcpyAsync(expert_ids_out, ctx->moe_ids + (size_t)layer * n, n * sizeof(int32_t),
                        cudaMemcpyDeviceToDevice, S(stream)) != cudaSuccess)
      return DF_ERR_CUDA;
  }
  return DF_OK;
}

int dualflow_expert_ids(dualflow_ctx* ctx, int32_t* ids, int32_t batch, dualflow_stream stream) {
  if (!ctx || !ids) return DF_ERR_ARG;
  const dualflow_config& c = ctx->cfg;
  if (c.n_experts == 0) return DF_ERR_UNSUPPORTED;
  if (batch <= 0 || batch > c.max_batch) return DF_ERR_SHAPE;
  const size_t kmax = std::max(c.topk_primary, c.topk_aux);
  const size_t n = (size_t)c.n_layers * 2 * batch * kmax;
  if (n == 0) return DF_OK;
  return cudaMemcpyAsync(ids, ctx->moe_ids, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, S(stream)) == cudaSuccess
             ? DF_OK
             : DF_ERR_CUDA;
}

int dualflow_mixture_head(dualflow_ctx* ctx, const float* logits, int32_t batch, const float* u, float* alpha,
                          float* p_mix, int32_t* token, dualflow_stream stream) {
  if (!ctx || !logits) return DF_ERR_ARG;
  if (batch <= 0 || batch > ctx->cfg.max_batch) return DF_ERR_SHAPE;
  return launch_mixture_head(logits, batch, ctx->cfg.vocab, u, alpha, p_mix, token, nullptr, 1, S(stream));
}

static int generate_loop(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv, int32_t batch,
                         int32_t n_steps, const float* u, int32_t* tokens_out, float* logits, float* logits_all,
                         int32_t* free_pages, int32_t* n_free, int32_t aux_on, dualflow_stream stream);

int dualflow_generate(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv, const int32_t* tokens,
                      int32_t batch, int32_t n_steps, const float* u, int32_t* tokens_out, float* logits,
                      float* logits_all, int32_t* free_pages, int32_t* n_free, int32_t aux_on,
                      dualflow_stream stream) {
  if (!ctx || !tokens || !tokens_out || !logits || !kv || !kv->seq_len) return DF_ERR_ARG;
  if (aux_on != 0 && aux_on != 1) return DF_ERR_ARG;
  if (batch <= 0 || batch > ctx->cfg.max_batch || n_steps < 0) return DF_ERR_SHAPE;
  if (n_steps == 0) return DF_OK;
  // the loop's own token buffer (the host variant copies the first tokens there directly)
  if (tokens != ctx->gen_tokens &&
      cudaMemcpyAsync(ctx->gen_tokens, tokens, (size_t)batch * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      S(stream)) != cudaSuccess)
    return DF_ERR_CUDA;
  return generate_loop(ctx, w, kv, batch, n_steps, u, tokens_out, logits, logits_all, free_pages, n_free, aux_on,
                       stream);
}

// The decode loop on the tokens already in ctx->gen_tokens.
static int generate_loop(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv, int32_t batch,
                         int32_t n_steps, const float* u, int32_t* tokens_out, float* logits, float* logits_all,
                         int32_t* free_pages, int32_t* n_free, int32_t aux_on, dualflow_stream stream) {
  const dualflow_config& c = ctx->cfg;
  cudaStream_t s = S(stream);
  const size_t per_step = (size_t)2 * batch * c.vocab;
  // the step reads the loop's own token buffer, so every step replays the same captured graph
  for (int t = 0; t < n_steps; ++t) {
    DF_TRY(dualflow_step(ctx, w, kv, ctx->gen_tokens, batch, logits, aux_on, stream));
    if (logits_all && cudaMemcpyAsync(logits_all + (size_t)t * per_step, logits, per_step * sizeof(float),
                                      cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return DF_ERR_CUDA;
    DF_TRY(launch_mixture_head(logits, batch, c.vocab, u ? u + (size_t)t * batch : nullptr, nullptr, nullptr,
                               tokens_out + (size_t)t * batch, ctx->gen_tokens, aux_on, s));
    DF_TRY(launch_gen_advance(c, const_cast<int32_t*>(kv->seq_len), batch, const_cast<int32_t*>(kv->page_table),
                              free_pages, n_free, ctx->status, s));
  }
  return DF_OK;
}

int dualflow_step(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv, const int32_t* tokens,
                  int32_t batch, float* logits, int32_t aux_on, dualflow_stream stream) {
  if (!ctx || !tokens || !logits) return DF_ERR_ARG;
  if (aux_on != 0 && aux_on != 1) return DF_ERR_ARG;
  if (batch <= 0 || batch > ctx->cfg.max_batch) return DF_ERR_SHAPE;
  DF_TRY(check_weights(ctx, w));
  if (!kv || kv->n_layers != ctx->cfg.n_layers) return DF_ERR_ARG;
  for (int l = 0; l < ctx->cfg.n_layers; ++l) DF_TRY(check_kv(ctx, kv, l));
  cudaStream_t s = S(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (s != nullptr && cudaStreamIsCapturing(s, &cap) != cudaSuccess) return DF_ERR_CUDA;
  if (!ctx->graphs_enabled || s == nullptr || cap != cudaStreamCaptureStatusNone)
    return run_step(ctx, w, kv, tokens, batch, logits, aux_on, s);
  std::vector<uint64_t> key;
  graph_key(key, ctx, w, kv, tokens, batch, logits, aux_on, s);
  for (auto& g : ctx->graphs)
    if (g.key == key) return cudaGraphLaunch(g.exec, s) == cudaSuccess ? DF_OK : DF_ERR_CUDA;
  cudaGraph_t graph = nullptr;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return DF_ERR_CUDA;
  const int rc = run_step(ctx, w, kv, tokens, batch, logits, aux_on, s);
  const cudaError_t ec = cudaStreamEndCapture(s, &graph);
  if (rc != DF_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (ec != cudaSuccess) return DF_ERR_CUDA;
  GraphEntry e;
  e.key = std::move(key);
  const cudaError_t ei = cudaGraphInstantiate(&e.exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess) return DF_ERR_CUDA;
  if (ctx->graphs.size() >= 16) {
    cudaGraphExecDestroy(ctx->graphs.front().exec);
    ctx->graphs.erase(ctx->graphs.begin());
  }
  ctx->graphs.push_back(std::move(e));
  return cudaGraphLaunch(ctx->graphs.back().exec, s) == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int dualflow_step_host(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv, const int32_t* tokens_host,
                       int32_t batch, float* logits_host, int32_t aux_on, dualflow_stream stream) {
  if (!ctx || !tokens_host || !logits_host) return DF_ERR_ARG;
  if (batch <= 0 || batch > ctx->cfg.max_batch) return DF_ERR_SHAPE;
  cudaStream_t s = S(stream);
  if (cudaMemcpyAsync(ctx->tokens_dev, tokens_host, (size_t)batch * sizeof(int32_t), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return DF_ERR_CUDA;
  DF_TRY(dualflow_step(ctx, w, kv, ctx->tokens_dev, batch, ctx->logits_dev, aux_on, stream));
  const size_t rows = aux_on ? 2 : 1;
  if (cudaMemcpyAsync(logits_host, ctx->logits_dev, rows * batch * ctx->cfg.vocab * sizeof(float),
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DF_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int dualflow_prefill_reserve(dualflow_ctx* ctx, int32_t max_rows) {
  if (!ctx || max_rows < 0) return DF_ERR_ARG;
  const dualflow_config& c = ctx->cfg;
  if (c.dtype != DF_DTYPE_BF16) return DF_ERR_UNSUPPORTED;
  if (c.n_experts > 32) return DF_ERR_UNSUPPORTED;
  if (max_rows <= ctx->pf_rows) return DF_OK;
  free_prefill_moe(ctx);
  for (void* p : {(void*)ctx->pf_h, ctx->pf_x, ctx->pf_q, ctx->pf_o, ctx->pf_u, (void*)ctx->pf_ss})
    if (p) cudaFree(p);
  ctx->pf_h = nullptr;
  ctx->pf_x = ctx->pf_q = ctx->pf_o = ctx->pf_u = nullptr;
  ctx->pf_ss = nullptr;
  ctx->pf_rows = 0;
  const size_t R = (size_t)max_rows, qd = (size_t)c.n_q_heads * c.head_dim;
  void* h = nullptr;
  void* ss = nullptr;
  if (dalloc(&h, R * c.d_model * 4) != DF_OK || dalloc(&ctx->pf_x, R * c.d_model * 2) != DF_OK ||
      dalloc(&ctx->pf_q, R * qd * 2) != DF_OK || dalloc(&ctx->pf_o, R * qd * 2) != DF_OK ||
      dalloc(&ctx->pf_u, R * c.ffn_hidden * 2) != DF_OK || dalloc(&ss, R * ctx->ss_ld * 4) != DF_OK) {
    for (void* p : {h, ctx->pf_x, ctx->pf_q, ctx->pf_o, ctx->pf_u, ss})
      if (p) cudaFree(p);
    ctx->pf_x = ctx->pf_q = ctx->pf_o = ctx->pf_u = nullptr;
    return DF_ERR_OOM;
  }
  ctx->pf_h = static_cast<float*>(h);
  ctx->pf_ss = static_cast<float*>(ss);
  if (c.n_experts > 0) {
    // the MoE rows: routing of every row, then each row once per chosen expert, gathered
    const size_t E = c.n_experts, RK = R * c.topk_primary, d = c.d_model, F = c.ffn_hidden;
    if (dalloc(&ctx->pf_rlog, R * E * 4) != DF_OK || dalloc(&ctx->pf_sel_pos, R * E * 4) != DF_OK ||
        dalloc(&ctx->pf_sel_w, R * E * 4) != DF_OK || dalloc(&ctx->pf_perm, RK * 4) != DF_OK ||
        dalloc(&ctx->pf_pos, RK * 4) != DF_OK || dalloc(&ctx->pf_xg, RK * d * 2) != DF_OK ||
        dalloc(&ctx->pf_ssg, RK * ctx->ss_ld * 4) != DF_OK || dalloc(&ctx->pf_ug, RK * F * 2) != DF_OK ||
        dalloc(&ctx->pf_yg, RK * d * 4) != DF_OK || dalloc(&ctx->pf_blk, ((RK + 255) / 256 + E) * sizeof(int4)) != DF_OK ||
        dalloc(&ctx->pf_nblk, 4) != DF_OK) {
      free_prefill_moe(ctx);
      for (void* p : {(void*)ctx->pf_h, ctx->pf_x, ctx->pf_q, ctx->pf_o, ctx->pf_u, (void*)ctx->pf_ss})
        if (p) cudaFree(p);
      ctx->pf_h = nullptr;
      ctx->pf_x = ctx->pf_q = ctx->pf_o = ctx->pf_u = nullptr;
      ctx->pf_ss = nullptr;
      return DF_ERR_OOM;
    }
  }
  ctx->pf_rows = max_rows;
  return DF_OK;
}

int dualflow_prefill(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv, const int32_t* tokens,
                     int32_t batch, int32_t n_tok, dualflow_stream stream) {
  return dualflow_prefill_slots(ctx, w, kv, tokens, nullptr, batch, n_tok, nullptr, nullptr, stream);
}

int dualflow_prefill_slots(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv,
                           const int32_t* tokens, const int32_t* slots, int32_t n_seq, int32_t n_tok,
                           int32_t* free_pages, int32_t* n_free, dualflow_stream stream) {
  if (!ctx || !tokens) return DF_ERR_ARG;
  const dualflow_config& c = ctx->cfg;
  if (c.dtype != DF_DTYPE_BF16 || c.n_experts > 32) return DF_ERR_UNSUPPORTED;
  const int G = c.n_q_heads / c.n_kv_heads;
  if (G != 1 && G != 2 && G != 4) return DF_ERR_UNSUPPORTED;
  if ((free_pages == nullptr) != (n_free == nullptr)) return DF_ERR_ARG;
  if (!c.paged && free_pages) return DF_ERR_ARG;
  if (n_seq <= 0 || n_seq > c.max_batch || n_tok < 0) return DF_ERR_SHAPE;
  if (n_tok == 0) return DF_OK;
  if ((long long)n_seq * n_tok > ctx->pf_rows) return DF_ERR_SHAPE;
  DF_TRY(check_weights(ctx, w));
  if (!kv || kv->n_layers != c.n_layers) return DF_ERR_ARG;
  for (int l = 0; l < c.n_layers; ++l) DF_TRY(check_kv(ctx, kv, l));
  cudaStream_t s = S(stream);
  const int R = n_seq * n_tok;
  int32_t* table = const_cast<int32_t*>(kv->page_table);
  if (free_pages)
    DF_TRY(launch_prefill_pages(c, kv->seq_len, slots, n_seq, n_tok, table, free_pages, n_free, ctx->status, s));
  const int qkv_n = (c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim, qd = c.n_q_heads * c.head_dim;
  const int d_tiles = (c.d_model + kGemmTileN - 1) / kGemmTileN;
  // the decode step's kernels on the prefill rows: the context's activation buffers point at the
  // prefill workspace for the duration of the call
  struct Swap {
    dualflow_ctx* c;
    float* h;
    void *x, *q, *o, *u;
    float* ss;
    ~Swap() {
      c->h = h;
      c->x = x;
      c->q = q;
      c->o = o;
      c->u = u;
      c->ss = ss;
    }
  } keep{ctx, ctx->h, ctx->x, ctx->q, ctx->o, ctx->u, ctx->ss};
  ctx->h = ctx->pf_h;
  ctx->x = ctx->pf_x;
  ctx->q = ctx->pf_q;
  ctx->o = ctx->pf_o;
  ctx->u = ctx->pf_u;
  ctx->ss = ctx->pf_ss;
  DF_TRY(launch_embed_prep(ctx, w->E1, w->E1, tokens, w->g_attn[0], R, 0, s));
  int ss_parts = 1;
  auto rows = [&](GemmArgs& g) {
    g.m_p = R;
    g.m_a = 0;
    g.row_blocked = 1;
    g.seq_rows = n_tok;
    g.slots = slots;
    g.max_batch = c.max_batch;
  };
  auto normed_input = [&](GemmArgs& g) {
    g.ss_in = ctx->ss;
    g.ss_parts = ss_parts;
    g.ss_ld = ctx->ss_ld;
    g.inv_d = 1.0f / (float)c.d_model;
    g.eps = c.rms_eps;
  };
  auto norm_output = [&](GemmArgs& g, const void* g_next) {
    g.g_next = g_next;
    g.x_next = ctx->x;
    g.ss_out = ctx->ss;
    g.ss_ld = ctx->ss_ld;
  };
  for (int l = 0; l < c.n_layers; ++l) {
    GemmArgs g = gemm_args(ctx);
    g.x = ctx->x;
    g.W = w->Wqkv[l];
    g.n_out = qkv_n;
    g.k = c.d_model;
    rows(g);
    g.epi = EPI_PREFILL_QKV;
    g.q_out = ctx->q;
    g.seq_len = kv->seq_len;
    g.k_cache = kv->k[l];
    g.v_cache = kv->v[l];
    g.page_table = kv->page_table;
    normed_input(g);
    DF_TRY(launch_gemm_tc(ctx, g, s));
    DF_TRY(launch_attention_prefill(c, ctx->q, ctx->o, kv->k[l], kv->v[l], kv->seq_len, kv->page_table, slots, n_seq,
                                    n_tok, ctx->status, s));
    GemmArgs o = gemm_args(ctx);
    o.x = ctx->o;
    o.W = w->Wo[l];
    o.n_out = c.d_model;
    o.k = qd;
    rows(o);
    o.epi = EPI_ADD_F32;
    o.y = ctx->h;
    o.ldy = c.d_model;
    norm_output(o, w->g_mlp[l]);
    DF_TRY(launch_gemm_tc(ctx, o, s));
    ss_parts = d_tiles;
    if (c.n_experts > 0) {
      DF_TRY(prefill_moe(ctx, w, l, R, ss_parts, s));
      ss_parts = (c.d_model + 511) / 512;
      continue;
    }
    GemmArgs gu = gemm_args(ctx);
    gu.x = ctx->x;
    gu.W = w->Wgu[l];
    gu.n_out = c.ffn_hidden;
    gu.k = c.d_model;
    rows(gu);
    gu.epi = EPI_SWIGLU;
    gu.y = ctx->u;
    gu.ldy = c.ffn_hidden;
    gu.vec = w->b[l];
    normed_input(gu);
    DF_TRY(launch_gemm_tc(ctx, gu, s));
    GemmArgs dn = gemm_args(ctx);
    dn.x = ctx->u;
    dn.W = w->Wd[l];
    dn.n_out = c.d_model;
    dn.k = c.ffn_hidden;
    rows(dn);
    dn.epi = EPI_COUPLE_ADD;
    dn.y = ctx->h;
    dn.ldy = c.d_model;
    dn.vec = w->c[l];
    if (l + 1 < c.n_layers) norm_output(dn, w->g_attn[l + 1]);
    DF_TRY(launch_gemm_tc(ctx, dn, s));
    ss_parts = d_tiles;
  }
  return launch_seq_advance(const_cast<int32_t*>(kv->seq_len), slots, n_seq, c.max_batch, n_tok, s);
}

int dualflow_release_slots(dualflow_ctx* ctx, const dualflow_kv* kv, const int32_t* slots, int32_t n_slots,
                           int32_t* free_pages, int32_t* n_free, dualflow_stream stream) {
  if (!ctx || !kv || !kv->seq_len || !slots) return DF_ERR_ARG;
  const dualflow_config& c = ctx->cfg;
  if (n_slots < 0 || n_slots > c.max_batch) return DF_ERR_SHAPE;
  if (c.paged && (!kv->page_table || !free_pages || !n_free)) return DF_ERR_ARG;
  if (!c.paged && (free_pages || n_free)) return DF_ERR_ARG;
  if (n_slots == 0) return DF_OK;
  return launch_release_slots(c, const_cast<int32_t*>(kv->seq_len), slots, n_slots,
                              const_cast<int32_t*>(kv->page_table), free_pages, n_free, ctx->status, S(stream));
}

int dualflow_generate_host(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv,
                           const int32_t* tokens_host, int32_t batch, int32_t n_steps, const float* u_host,
                           int32_t* tokens_out_host, int32_t aux_on, dualflow_stream stream) {
  if (!ctx || !tokens_host || !tokens_out_host) return DF_ERR_ARG;
  if (batch <= 0 || batch > ctx->cfg.max_batch || n_steps < 0 || n_steps > kGenHostMaxSteps) return DF_ERR_SHAPE;
  if (n_steps == 0) return DF_OK;
  cudaStream_t s = S(stream);
  const size_t nb = (size_t)batch * sizeof(int32_t), total = (size_t)n_steps * batch;
  if (!kv || !kv->seq_len || (aux_on != 0 && aux_on != 1)) return DF_ERR_ARG;
  // the first tokens go straight into the loop's own token buffer
  if (cudaMemcpyAsync(ctx->gen_tokens, tokens_host, nb, cudaMemcpyHostToDevice, s) != cudaSuccess) return DF_ERR_CUDA;
  if (u_host && cudaMemcpyAsync(ctx->gen_u_dev, u_host, total * sizeof(float), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DF_ERR_CUDA;
  DF_TRY(generate_loop(ctx, w, kv, batch, n_steps, u_host ? ctx->gen_u_dev : nullptr, ctx->gen_out_dev,
                       ctx->logits_dev, nullptr, nullptr, nullptr, aux_on, stream));
  if (cudaMemcpyAsync(tokens_out_host, ctx->gen_out_dev, total * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return DF_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int dualflow_set_graphs(dualflow_ctx* ctx, int32_t enabled) {
  if (!ctx || (enabled != 0 && enabled != 1)) return DF_ERR_ARG;
  ctx->graphs_enabled = enabled;
  if (!enabled) drop_graphs(ctx);
  return DF_OK;
}

int dualflow_set_profiling(dualflow_ctx* ctx, int32_t mode) {
  if (!ctx || mode < 0 || mode > 2) return DF_ERR_ARG;
  if (mode == 2 && ctx->cfg.dtype != DF_DTYPE_BF16) return DF_ERR_UNSUPPORTED;
  const int n = 8 * std::max(ctx->cfg.n_layers, 1) + 16;
  if (mode == 1 && ctx->prof.empty()) {
    ctx->prof.resize(n);
    for (auto& r : ctx->prof)
      if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return DF_ERR_CUDA;
  }
  if (mode == 2 && ctx->stamps == nullptr) {
    if (dalloc(&ctx->stamps, (size_t)(n + 1) * sizeof(unsigned long long)) != DF_OK) return DF_ERR_OOM;
    if (cudaMemset(ctx->stamps, 0, (size_t)(n + 1) * sizeof(unsigned long long)) != cudaSuccess) return DF_ERR_CUDA;
    ctx->prof_fam.assign(n, 0);
  }
  if (ctx->profiling != mode) drop_graphs(ctx);
  ctx->profiling = mode;
  return DF_OK;
}

int dualflow_profile_read(dualflow_ctx* ctx, float* ms, int32_t* launches, int32_t n_families) {
  if (!ctx || n_families < 0) return DF_ERR_ARG;
  const int n = std::min<int>(n_families, DF_PROF_FAMILIES);
  if (cudaDeviceSynchronize() != cudaSuccess) return DF_ERR_CUDA;
  if (launches)
    for (int f = 0; f < n; ++f) launches[f] = ctx->step_launches[f];
  if (ms) {
    for (int f = 0; f < n; ++f) ms[f] = 0.f;
    if (ctx->profiling == 1)
      for (int i = 0; i < ctx->prof_n; ++i) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, ctx->prof[i].a, ctx->prof[i].b) != cudaSuccess) return DF_ERR_CUDA;
        if (ctx->prof[i].fam < n) ms[ctx->prof[i].fam] += t;
      }
    if (ctx->profiling == 2 && ctx->prof_n > 0) {
      // each launch's share of the step: from the end of the launch before it (the step's start
      // for the first) to its own end
      std::vector<unsigned long long> st((size_t)ctx->prof_n + 1);
      if (cudaMemcpy(st.data(), ctx->stamps, st.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost) !=
          cudaSuccess)
        return DF_ERR_CUDA;
      unsigned long long prev = st[0];
      for (int i = 0; i < ctx->prof_n; ++i) {
        const unsigned long long e = st[1 + (size_t)i];
        const double dt = e > prev ? (double)(e - prev) * 1e-6 : 0.0;
        if (ctx->prof_fam[i] < n) ms[ctx->prof_fam[i]] += (float)dt;
        prev = e > prev ? e : prev;
      }
    }
  }
  return DF_OK;
}

int dualflow_set_call_chaining(dualflow_ctx* ctx, int32_t enabled) {
  if (!ctx || (enabled != 0 && enabled != 1)) return DF_ERR_ARG;
  ctx->chain_calls = enabled;
  return DF_OK;
}

int dualflow_set_nvtx(dualflow_ctx* ctx, int32_t enabled) {
  if (!ctx || (enabled != 0 && enabled != 1)) return DF_ERR_ARG;
  ctx->nvtx = enabled;
  return DF_OK;
}

int dualflow_set_wait_limit(dualflow_ctx* ctx, int64_t limit_ns) {
  if (!ctx || limit_ns < 0) return DF_ERR_ARG;
  if ((unsigned long long)limit_ns != ctx->wait_ns) drop_graphs(ctx);
  ctx->wait_ns = (unsigned long long)limit_ns;
  return DF_OK;
}

int dualflow_router_logits(dualflow_ctx* ctx, float* logits, int32_t batch, dualflow_stream stream) {
  if (!ctx || !logits) return DF_ERR_ARG;
  const dualflow_config& c = ctx->cfg;
  if (c.n_experts == 0 || c.dtype != DF_DTYPE_BF16) return DF_ERR_UNSUPPORTED;
  if (batch <= 0 || batch > c.max_batch) return DF_ERR_SHAPE;
  if (c.n_layers == 0) return DF_OK;
  const size_t row = (size_t)2 * batch * c.n_experts * sizeof(float);
  const size_t pitch = (size_t)2 * c.max_batch * c.n_experts * sizeof(float);
  return cudaMemcpy2DAsync(logits, row, ctx->rlog, pitch, row, (size_t)c.n_layers, cudaMemcpyDeviceToDevice,
                           S(stream)) == cudaSuccess
             ? DF_OK
             : DF_ERR_CUDA;
}

int dualflow_sync_status(dualflow_ctx* ctx, dualflow_stream stream) {
  if (!ctx) return DF_ERR_ARG;
  cudaStream_t s = S(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DF_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, ctx->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DF_ERR_CUDA;
  if (v != 0 && cudaMemset(ctx->status, 0, sizeof(v)) != cudaSuccess) return DF_ERR_CUDA;
  // a kernel that gave up on a wait may have left the attention's merge counters behind
  if (v == DF_ERR_TIMEOUT && ctx->attn_cnt &&
      cudaMemset(ctx->attn_cnt, 0, (size_t)ctx->cfg.max_batch * ctx->cfg.n_kv_heads * sizeof(int32_t)) != cudaSuccess)
    return DF_ERR_CUDA;
  return v;
}

}  // extern "C"
