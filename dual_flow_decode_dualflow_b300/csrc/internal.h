// Internal declarations shared by the library's translation units: the context, the argument
// blocks of every kernel family and their host launchers.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/dualflow.h"

namespace df {

// ---- bf16 kernel constraints --------------------------------------------------------------
constexpr int kHeadDim = 128;       // bf16 attention and QKV epilogue assume D = 128
constexpr int kMaxGroupRows = 8;    // 2 flows x G query heads per KV head share one mma n-tile
constexpr int kAttnTileKeys = 64;   // keys per pipeline stage of the decode-attention kernel
constexpr int kGemmTileN = 128;     // weight rows (output features) per tcgen05 tile
constexpr int kGemmTileK = 64;      // reduction elements per pipeline stage (128-byte rows)
constexpr int kGenHostMaxSteps = 256;  // steps of one dualflow_generate_host call
constexpr int kGemmMaxAct = 256;    // activation rows (both flows) per tcgen05 tile

// Partial result of one attention segment: 8 query rows x (D values + running max + sum).
constexpr int kAttnPartFloats = kMaxGroupRows * (kHeadDim + 2);

// ---- epilogues of the tcgen05 stacked linear ------------------------------------------------
enum GemmEpi : int {
  EPI_STORE_F32 = 0,  // y fp32
  EPI_STORE_BF16 = 1, // y bf16
  EPI_ADD_F32 = 2,    // y fp32 +=
  EPI_COUPLE_ADD = 3, // z2 += c (*) z1; y fp32 += z
  EPI_QKV = 4,        // query coupling a, RoPE, q store, primary K/V append
  EPI_Q2 = 5,         // attention-only: q2 = acc + a (*) q1, RoPE of q1 and q2
  EPI_SWIGLU = 6,     // u = silu(gate) (*) up, u2 += b (*) u1, bf16 store
  EPI_MOE_GATEUP = 7, // per expert: SWIGLU for the rows that selected it, u2 += b (*) u1 if both did
  EPI_MOE_DOWN = 8,   // per expert: fp32 store of the rows that selected it
  EPI_PREFILL_QKV = 9, // prefill (primary only): RoPE at seq_len[b] + t, q store, K/V into the cache
};

struct GemmArgs {
  // operands
  const void* x;   // [m_p + m_a, k] bf16 (activations, both flows stacked)
  const void* W;   // [n_rows, k] bf16
  int n_out;       // output features (for EPI_SWIGLU: hidden units F, W has 2F rows)
  int k;
  int m_p, m_a;    // primary / auxiliary activation rows
  int epi;
  // epilogue operands
  void* y;             // STORE/ADD/COUPLE: [m, n_out] ; SWIGLU: u [m, F] bf16
  int ldy;             // leading dimension of y in elements
  const void* vec;     // COUPLE: c ; QKV/Q2: a ; SWIGLU: b   (bf16 [n_out])
  // QKV / Q2
  void* q_out;             // [2, B, Hq, D] bf16
  const void* q1_in;       // Q2: q1 [B, Hq, D] bf16
  int n_q_heads, n_kv_heads;
  const int32_t* seq_len;  // [B] device
  const float2* rope;      // [max_ctx + 1][D/2] (cos, sin)
  void* k_cache;
  void* v_cache;
  const int32_t* page_table;
  int paged, page_size, max_ctx, max_pages, pages_per_seq;
  // RMSNorm carried across kernels (decode step). When ss_in is set, the rows of x hold h (*) g
  // and each output row is scaled by 1 / sqrt(sum_p ss_in[row * ss_ld + p] * inv_d + eps),
  // p = 0 .. ss_parts - 1 in order.
  const float* ss_in;
  int ss_parts, ss_ld;
  float inv_d, eps;
  // Residual epilogues (ADD_F32, COUPLE_ADD) with g_next set also write the next norm's input
  // x_next[row] = bf16(h_new (*) g_next) ([m, n_out]) and ss_out[row * ss_ld + tile * S + split] =
  // the sum of h_new^2 over that CTA's features (n_tiles * S partials per row).
  const void* g_next;
  void* x_next;
  float* ss_out;
  int pdl;  // launch with programmatic dependent launch (weights prefetched before the wait)
  // Grouped (MoE) launch: grid z = n_groups experts. Expert e's weight rows start at row
  // e * w_group_rows of W, its activation rows at row e * x_group_rows of x (0: shared x), its
  // output at y + e * y_group_stride elements; sel_pos[row * n_groups + e] >= 0 when row uses e.
  int n_groups, w_group_rows, x_group_rows;
  size_t y_group_stride;
  const int32_t* sel_pos;
  // L2 prefetch of the next projection's weights: once its last tiles are requested, each CTA asks
  // L2 for the first pf_depth k-blocks of its share of the next launch's (tile, split) CTAs, so the
  // next launch starts on L2-resident weights. pf_W = nullptr: none.
  const void* pf_W;
  int pf_k, pf_rows, pf_tiles, pf_splits, pf_tile_rows, pf_half, pf_depth;
  // Prefill: more activation rows than one tile holds. The rows are cut into blocks of 256
  // (grid y), each CTA offsets y / x_next / ss_in / ss_out by its block; row_base is the block's
  // first row, seq_rows the prompt positions per sequence (row r = i * seq_rows + t). m_a = 0.
  // Prompt sequence i lives in cache slot slots[i] (slots = nullptr: slot i), 0 <= slot < max_batch.
  int row_blocked, seq_rows, row_base;
  const int32_t* slots;
  int max_batch;
  // Gathered expert rows (row-blocked grouped launch, prefill MoE): row block g of the grid is
  // expert blk_info[g].x's rows [blk_info[g].y, + blk_info[g].z) of x / y / ss_in; blocks g >=
  // *n_blk do nothing. m_p is the capacity in rows (the x tensor map's extent).
  const int4* blk_info;
  const int32_t* n_blk;
  // In-graph timing (profiling mode 2): the CTAs raise *stamp to the globaltimer value at their end
  // (nullable).
  unsigned long long* stamp;
};

struct AttnArgs {
  const void* q;            // [2, B, Hq, D] bf16, post-RoPE
  void* o;                  // [2, B, Hq, D] bf16
  const void* k_cache;
  const void* v_cache;
  const int32_t* seq_len;   // [B] device
  const int32_t* page_table;
  int batch, n_q_heads, n_kv_heads;
  int paged, page_size, max_ctx, max_pages, pages_per_seq;
  int extra;                // 1 when the step appended slot seq_len[b] (attend 0..seq_len[b])
  int aux_on;
  unsigned long long* stamp;  // in-graph timing: raised to the globaltimer value at the end (nullable)
};

struct ProfRec {
  int fam = 0;
  cudaEvent_t a = nullptr, b = nullptr;
};

struct GraphEntry {
  std::vector<uint64_t> key;
  cudaGraphExec_t exec = nullptr;
};

}  // namespace df

struct dualflow_ctx {
  dualflow_config cfg;
  int device = 0;
  int num_sms = 148;
  int32_t* status = nullptr;       // device status word
  float2* rope = nullptr;          // [max_ctx + 1][head_dim / 2]
  // decode-attention split workspace
  float* attn_part = nullptr;
  int32_t* attn_cnt = nullptr;
  int attn_ctas = 0;               // persistent grid size of the attention kernel
  int attn_slots = 0;
  // step activations
  float* h = nullptr;              // [2, max_batch, d] fp32 residual
  void* x = nullptr;               // [2 * max_batch, max(d, F)] storage dtype (normed input)
  void* q = nullptr;               // [2, max_batch, Hq, D]
  void* o = nullptr;               // [2, max_batch, Hq * D]
  void* u = nullptr;               // [2 * max_batch, F]
  float* raw = nullptr;            // fp32 path: [2 * max_batch, max_n] projection scratch
  float* ss = nullptr;             // [2 * max_batch][ss_ld] per-row partial sums of squares (bf16)
  // MoE (bf16): router logits, routing decision, expert intermediates and outputs, expert ids
  float* rlog = nullptr;           // [2 * max_batch][E]
  int32_t* sel_pos = nullptr;      // [2 * max_batch][E] position in the row's expert set, -1 if unused
  float* sel_w = nullptr;          // [2 * max_batch][E] mixing weight
  void* moe_u = nullptr;           // [E][2 * max_batch][F] bf16
  float* moe_y = nullptr;          // [E][2 * max_batch][d]
  int32_t* moe_ids = nullptr;      // [n_layers][2][max_batch][kmax] experts chosen by the last step
  // prefill workspace (dualflow_prefill_reserve): rows = prompt tokens of all sequences
  int pf_rows = 0;
  float* pf_h = nullptr;           // [pf_rows][d] residual
  void* pf_x = nullptr;            // [pf_rows][d] bf16 norm operand
  void* pf_q = nullptr;            // [pf_rows][Hq * D] bf16
  void* pf_o = nullptr;            // [pf_rows][Hq * D] bf16
  void* pf_u = nullptr;            // [pf_rows][F] bf16
  float* pf_ss = nullptr;          // [pf_rows][ss_ld]
  // prefill MoE (pf_rows rows R, k = topk_primary): routing, the rows gathered per expert
  float* pf_rlog = nullptr;        // [R][E] router logits
  int32_t* pf_sel_pos = nullptr;   // [R][E] position of e in the row's expert set, -1 if unused
  float* pf_sel_w = nullptr;       // [R][E]
  int32_t* pf_perm = nullptr;      // [R k] source row of gathered row q (expert-major, rows in order)
  int32_t* pf_pos = nullptr;       // [R][k] gathered row of the row's j-th expert
  void* pf_xg = nullptr;           // [R k][d] bf16 gathered norm operand
  float* pf_ssg = nullptr;         // [R k][ss_ld] gathered sums of squares
  void* pf_ug = nullptr;           // [R k][F] bf16 expert intermediates
  float* pf_yg = nullptr;          // [R k][d] expert outputs
  int4* pf_blk = nullptr;          // [R k / 256 + E] row blocks of the gathered rows
  int32_t* pf_nblk = nullptr;      // [1]
  float* gemm_part = nullptr;      // split-K partials exchanged through L2 (gemm_part_floats)
  size_t gemm_part_floats = 0;
  int32_t* gen_tokens = nullptr;   // [max_batch] input tokens of the generation loop's next step
  int32_t* gen_out_dev = nullptr;  // [kGenHostMaxSteps][max_batch] dualflow_generate_host staging
  float* gen_u_dev = nullptr;      // [kGenHostMaxSteps][max_batch]
  int ss_ld = 0;                   // ceil(d / 128) tiles x 8 splits
  int32_t* tokens_dev = nullptr;   // dualflow_step_host staging
  float* logits_dev = nullptr;
  int graphs_enabled = 1;
  std::vector<df::GraphEntry> graphs;
  // per-kernel timing of the step (events reused across steps)
  int profiling = 0;
  std::vector<df::ProfRec> prof;
  int prof_n = 0;
  int step_launches[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  // in-graph timing (profiling mode 2): stamps[0] = start of the step's first kernel, stamps[1 + i]
  // = end of its i-th launch; prof_fam[i] = that launch's family
  unsigned long long* stamps = nullptr;
  std::vector<int> prof_fam;
  unsigned long long* cur_stamp = nullptr;  // the slot of the launch being recorded (nullptr: none)
  // limit of the bounded pipeline waits (ns); 0 = the library default. Failure-path tests only.
  unsigned long long wait_ns = 0;
  int nvtx = 0;  // NVTX ranges around the step's layers and launches
  int chain_calls = 0;  // dualflow_set_call_chaining
};

namespace df {

// Tensor-map encoding through the driver entry point (no link-time libcuda dependency).
int encode_map_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                       uint32_t box_inner, uint32_t box_rows);
int encode_map_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                       uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);

// Launchers (return dualflow_status).
int launch_gemm_tc(dualflow_ctx* ctx, const GemmArgs& a, cudaStream_t s);
int gemm_splits(const dualflow_ctx* ctx, int n_out, int k, int epi, int groups = 1);
int gemm_tiles(int n_out, int epi);
size_t gemm_part_floats(const dualflow_ctx* ctx);
// Fills cur's L2-prefetch fields from the (ungrouped) projection `next` that follows it.
void gemm_prefetch_next(const dualflow_ctx* ctx, GemmArgs& cur, const GemmArgs& next);
int launch_attention_bf16(dualflow_ctx* ctx, const AttnArgs& a, cudaStream_t s, int pdl = 0);
// The same kernel with caller-chosen workspace: split partials (>= pairs + ctas slots of
// kAttnPartFloats), per-pair merge counters (zero on entry), the status word, and a grid of `ctas`
// CTAs; cache geometry is taken from `cfg`; wait_ns = limit of the pipeline waits (0: default).
// Used by the allocation-free entry point and, with the context's workspace, by the one above.
int launch_attention_bf16_ws(const dualflow_config& cfg, const AttnArgs& a, float* part, int32_t* cnt,
                             int32_t* status, int ctas, cudaStream_t s, int pdl = 0,
                             unsigned long long wait_ns = 0);
// Sets a kernel's shared-memory attributes once per device: the device's largest opt-in dynamic
// shared memory and the full shared-memory carveout. Launches never change them again, so
// concurrent launches of the same kernel with different sizes cannot race on a process-wide
// attribute. Thread-safe.
int set_smem_attrs_once(const void* kernel);

int launch_embed_rmsnorm(dualflow_ctx* ctx, const void* E1, const void* E2, const int32_t* tokens, const void* g,
                         int batch, int aux_on, cudaStream_t s);
// Decode step (bf16): h = E_f[token]; x = bf16(h (*) g); ss[row] = sum h^2 (one partial).
int launch_embed_prep(dualflow_ctx* ctx, const void* E1, const void* E2, const int32_t* tokens, const void* g,
                      int batch, int aux_on, cudaStream_t s);
// The same from the residual h (bf16): x = bf16(h (*) g); ss[row] = sum h^2 (one partial).
int launch_norm_prep(dualflow_ctx* ctx, float* h, const void* g, int batch, int aux_on, cudaStream_t s);
// MoE: routing decision from ctx->rlog (ids [2][batch][kmax], nullable), and the combine of the
// experts' outputs with output coupling and residual (g_next set: also the next norm's operand,
// ceil(d / 512) partial sums of squares per row).
int launch_moe_route(dualflow_ctx* ctx, const float* rlog, int batch, int aux_on, int32_t* ids, cudaStream_t s,
                     int pdl);
int launch_moe_plan(const dualflow_config& c, int R, const int32_t* sel_pos, int32_t* perm, int32_t* pos, int4* blk,
                    int32_t* n_blk, int32_t* status, cudaStream_t s);
int launch_moe_gather(int rows, int R, int d, const void* x, const float* ss, int ss_ld, const int32_t* perm, void* xg,
                      float* ssg, int32_t* status, cudaStream_t s);
int launch_moe_combine_rows(const dualflow_config& c, int R, const float* yg, const int32_t* sel_pos,
                            const float* sel_w, const int32_t* pos, float* h, const void* g_next, void* x_next,
                            float* ss, int ss_ld, int32_t* status, cudaStream_t s);
int launch_moe_route_rows(const dualflow_config& c, const float* rlog, int R, int32_t* sel_pos, float* sel_w,
                          cudaStream_t s);
int launch_moe_combine(dualflow_ctx* ctx, float* h, int batch, int aux_on, const void* c_vec, const void* g_next,
                       cudaStream_t s, int pdl);
int launch_mixture_head(const float* logits, int batch, int vocab, const float* u, float* alpha, float* p_mix,
                        int32_t* token, int32_t* token2, int aux_on, cudaStream_t s);
int launch_attention_prefill(const dualflow_config& c, const void* q, void* o, const void* k_cache,
                             const void* v_cache, const int32_t* seq_len, const int32_t* page_table,
                             const int32_t* slots, int n_seq, int n_tok, int32_t* status, cudaStream_t s);
int launch_seq_advance(int32_t* seq_len, const int32_t* slots, int n_seq, int max_batch, int n, cudaStream_t s);
int launch_prefill_pages(const dualflow_config& c, const int32_t* seq_len, const int32_t* slots, int n_seq, int n,
                         int32_t* table, int32_t* free_pages, int32_t* n_free, int32_t* status, cudaStream_t s);
int launch_release_slots(const dualflow_config& c, int32_t* seq_len, const int32_t* slots, int n_slots, int32_t* table,
                         int32_t* free_pages, int32_t* n_free, int32_t* status, cudaStream_t s);
int launch_gen_advance(const dualflow_config& c, int32_t* seq_len, int batch, int32_t* table, int32_t* free_pages,
                       int32_t* n_free, int32_t* status, cudaStream_t s);
int launch_rmsnorm(dualflow_ctx* ctx, const float* h, const void* g, void* x, int batch, int aux_on, cudaStream_t s);
int launch_rope_q1(dualflow_ctx* ctx, const void* q1, void* q, const int32_t* seq_len, int batch, cudaStream_t s);

// fp32 (CUDA-core) path
int launch_linear_f32(dualflow_ctx* ctx, const float* x, int m, const float* W, int n, int k, float* y, int accumulate,
                      cudaStream_t s);
int launch_qkv_post_f32(dualflow_ctx* ctx, const float* raw, int batch, int aux_on, const float* a, void* k_cache,
                        void* v_cache, const int32_t* page_table, const int32_t* seq_len, float* q, cudaStream_t s);
int launch_q2_post_f32(dualflow_ctx* ctx, const float* raw, const float* q1, int batch, int aux_on, const float* a,
                       const int32_t* seq_len, float* q, cudaStream_t s);
int launch_attention_f32(dualflow_ctx* ctx, const float* q, float* o, const void* k_cache, const void* v_cache,
                         const int32_t* page_table, const int32_t* seq_len, int batch, int extra, int aux_on,
                         cudaStream_t s);
int launch_swiglu_f32(dualflow_ctx* ctx, const float* raw, int batch, int aux_on, const float* b, float* u,
                      cudaStream_t s);
int launch_couple_add_f32(dualflow_ctx* ctx, const float* raw, int batch, int aux_on, int n, const float* c, float* h,
                          cudaStream_t s);

}  // namespace df
