/*
 * dualflow.h -- C ABI of the B300 (sm_103a) Dual-Flow Transformer decode library.
 *
 * The method ("Resumo Tecnico: Dual-Flow Transformers", gist.science, sections "Arquitetura
 * Central" and "Mecanismos Chave"): a primary flow and an auxiliary flow share every attention,
 * MLP and output matrix and the single persistent KV cache, which only the primary flow writes;
 * the auxiliary flow has its own token embedding, is coupled one way to the primary flow by the
 * learned vectors a_l (query), b_l (MLP intermediate) and c_l (MLP output), and never feeds back.
 * The pages give no coupling equations; this library fixes them as
 *     q2 = Wq.x2 + a_l (*) q1      u2 += b_l (*) u1      y2 += c_l (*) y1
 * Decode is memory-bound (same page, "Declaracao do Problema"), and grouping both flows lets one
 * read of each weight tile and each K1/V1 tile serve both ("Custos de Inferencia vs. Treinamento").
 *
 * Conventions for every call
 *  - Pointers named "device" are CUDA device addresses; all others are host addresses.
 *  - The caller owns every tensor (weights, cache, page table, free list, inputs, outputs). A
 *    context owns only its workspace, sized at dualflow_init from the config's max_* fields, plus
 *    the prefill workspace that dualflow_prefill_reserve allocates (a cold call). Hot calls never
 *    allocate.
 *  - Every compute call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns a dualflow_status. Argument and shape errors are detected on the host
 *    before any launch and leave every buffer untouched. Errors found on the device (an out-of-
 *    range page id, token or cache slot; an expired bounded wait) are latched in a device status
 *    word and reported by dualflow_sync_status.
 *  - Activations of the two flows are stacked flow-major: row r = f * batch + b, f = 0 primary,
 *    f = 1 auxiliary. With aux_on = 0 only the primary rows are computed and written, and the
 *    primary results are bit-identical to those of a call with aux_on = 1.
 *  - Storage dtype (config.dtype): DF_DTYPE_BF16 stores weights, embeddings, norm gains, coupling
 *    vectors and the KV cache as bf16 (round to nearest even); the residual stream, logits and all
 *    accumulations are fp32. DF_DTYPE_F32 stores everything as fp32 (no TF32 anywhere).
 *  - Matrices are row-major [out_features, in_features]; y = x . W^T.
 *  - A context's workspace (activations, split-KV partials and merge counters, the split-K
 *    exchange area, the prefill buffers) is shared by all of its calls: calls on one context must
 *    not overlap on the GPU (issue them on one stream, or order the streams). Independent
 *    contexts may run concurrently: apart from the static scratch of the context-free attention
 *    call (end of this header), every buffer a call writes belongs to its context or its caller.
 */
#ifndef DUALFLOW_H
#define DUALFLOW_H

#include <stdint.h>

#if defined(__GNUC__)
#define DF_API __attribute__((visibility("default")))
#else
#define DF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dualflow_ctx dualflow_ctx; /* opaque; owns workspace only */
typedef void* dualflow_stream;            /* cudaStream_t */

typedef enum {
  DF_OK = 0,
  DF_ERR_ARG = 1,            /* null pointer, negative or zero size, bad flag */
  DF_ERR_SHAPE = 2,          /* sizes inconsistent with the config or beyond its max_* fields */
  DF_ERR_DTYPE = 3,          /* unknown storage dtype */
  DF_ERR_UNSUPPORTED = 4,    /* a valid config this library has no kernel for (see dualflow_init) */
  DF_ERR_CUDA = 5,           /* a CUDA runtime call failed */
  DF_ERR_OOM = 6,            /* workspace allocation failed (dualflow_init, dualflow_prefill_reserve) */
  DF_ERR_DEVICE_BOUNDS = 7,  /* device-side check failed: page id, token id or cache slot out of range */
  DF_ERR_TIMEOUT = 8         /* a bounded device wait expired; the kernel returned early */
} dualflow_status;

enum { DF_DTYPE_F32 = 0, DF_DTYPE_BF16 = 1 };

/* Model and capacity description. */
typedef struct {
  int32_t n_layers;
  int32_t d_model;
  int32_t n_q_heads;   /* Hq */
  int32_t n_kv_heads;  /* Hkv; GQA group G = Hq / Hkv, query head h reads KV head h / G */
  int32_t head_dim;    /* D */
  int32_t ffn_hidden;  /* SwiGLU hidden F (dense) or per-expert hidden (MoE) */
  int32_t vocab;
  int32_t n_experts;   /* 0 = dense MLP */
  int32_t topk_primary;
  int32_t topk_aux;
  int32_t dtype;       /* DF_DTYPE_* */
  int32_t paged;       /* 0 = contiguous cache, 1 = paged cache */
  int32_t page_size;   /* positions per page (paged only) */
  int32_t max_batch;
  int32_t max_ctx;     /* cache capacity in positions per sequence (also the contiguous stride) */
  int32_t max_pages;   /* physical pages per layer (paged only) */
  float rope_base;     /* RoPE rotate-half pairs (i, i + D/2), theta_i = base^(-2i/D) */
  float rms_eps;       /* RMSNorm x = h / sqrt(mean(h^2) + eps) * g */
} dualflow_config;

/* Per-layer device pointers are passed as host arrays of n_layers device pointers.
 *   E1, E2   [vocab, d]       token embeddings of the primary / auxiliary flow
 *   W_lm     [vocab, d]       shared LM head;      g_final [d] shared final-norm gain
 *   g_attn, g_mlp [d]         shared pre-attention / pre-MLP RMSNorm gains
 *   Wqkv     [(Hq + 2 Hkv) D, d]   rows: Wq (Hq*D), then Wk (Hkv*D), then Wv (Hkv*D)
 *   Wo       [d, Hq D]
 *   Wgu      [2F, d]          rows: gate (F), then up (F)        (dense only)
 *   Wd       [d, F]                                              (dense only)
 *   Wr       [E, d]           shared router                      (MoE only)
 *   We_gu    [E, 2F, d]       per expert: gate rows then up rows (MoE only)
 *   We_d     [E, d, F]                                           (MoE only)
 *   a [Hq D], b [F], c [d]    coupling vectors of each layer
 */
typedef struct {
  const void* E1;
  const void* E2;
  const void* W_lm;
  const void* g_final;
  const void* const* g_attn;
  const void* const* g_mlp;
  const void* const* Wqkv;
  const void* const* Wo;
  const void* const* Wgu;
  const void* const* Wd;
  const void* const* Wr;
  const void* const* We_gu;
  const void* const* We_d;
  const void* const* a;
  const void* const* b;
  const void* const* c;
  int32_t n_layers;
} dualflow_weights;

/* The primary flow's persistent KV cache ("Arquitetura Central": only the primary writes it).
 *   k[l], v[l]  device; contiguous: [max_batch, Hkv, max_ctx, D]
 *                        paged:      [max_pages, Hkv, page_size, D]
 *   page_table  device int32 [max_batch, ceil(max_ctx / page_size)]; entry j of row b is the
 *               physical page holding positions [j*page_size, (j+1)*page_size); -1 = unused
 *   seq_len     device int32 [batch]: positions cached BEFORE the call. A step writes the new
 *               primary key/value at slot seq_len[b] and both flows attend positions
 *               0..seq_len[b]; the caller advances seq_len afterwards (dualflow_generate and the
 *               prefill calls advance it themselves). Calls that take cache slots
 *               (dualflow_prefill_slots, dualflow_release_slots) index it by slot: [max_batch]. */
typedef struct {
  void* const* k;
  void* const* v;
  const int32_t* page_table;
  const int32_t* seq_len;
  int32_t n_layers;
} dualflow_kv;

/* Creates a context for `cfg` on the current CUDA device and allocates its workspace.
 * Host-validates the config (DF_ERR_ARG / DF_ERR_SHAPE / DF_ERR_DTYPE before touching the GPU).
 * bf16 kernels need head_dim == 128, Hq / Hkv <= 4, d_model, ffn_hidden and Hq*head_dim
 * multiples of 64, max_batch <= 128 and n_experts <= 32 (else DF_ERR_UNSUPPORTED); MoE models
 * need bf16 storage. On failure *out is set to NULL. */
DF_API int dualflow_init(const dualflow_config* cfg, dualflow_ctx** out);

/* Releases the context and its workspace. NULL-safe. Synchronizes the device first. */
DF_API int dualflow_free(dualflow_ctx* ctx);

/* Static description of a status code; never NULL. */
DF_API const char* dualflow_status_string(int status);

/* Description of the last CUDA error that a call of this library met in the calling host thread: a
 * pending CUDA runtime error of the library's own runtime state, else the last failed driver call
 * of the library (tensor-map encoding), else "no error". Meant for diagnosing a DF_ERR_CUDA status
 * right after the call that returned it. Never fails; the string is static or thread-local. */
DF_API const char* dualflow_cuda_error_string(void);

/* Attention-only dual-flow decode of one layer ("Atencao de KV Compartilhada Assimetrica"):
 *   q2 = Wq . h2 + a (*) q1;  RoPE(q1), RoPE(q2) at position seq_len[b];
 *   o_f = softmax(q_f K1^T / sqrt(D)) V1 over the cached positions 0..seq_len[b]-1 of layer `layer`.
 * Nothing is appended. q1 [batch, Hq, D] (raw primary query projection), h2 [batch, d]
 * (auxiliary flow's normed input), Wq [Hq D, d], a [Hq D]: device, storage dtype.
 * o: device [2, batch, Hq, D], storage dtype (aux rows written only when aux_on).
 * seq_len[b] == 0 yields o = 0 for that row. Every K1/V1 tile is read once for both flows.
 * The call's first kernel waits for the caller's preceding work on the stream in the usual way
 * (unless dualflow_set_call_chaining enabled chaining); its second is chained to its first. */
DF_API int dualflow_decode_attention(dualflow_ctx* ctx, const void* q1, const void* h2, const void* Wq, const void* a,
                              const dualflow_kv* kv, int32_t layer, int32_t batch, void* o, int32_t aux_on,
                              dualflow_stream stream);

/* Epilogues of dualflow_stacked_linear. */
enum {
  DF_EPI_STORE_F32 = 0,   /* y fp32 [M, n] = x W^T */
  DF_EPI_STORE_BF16 = 1,  /* y storage-dtype [M, n] (bf16 rounding for bf16 contexts) */
  DF_EPI_ADD_F32 = 2,     /* y fp32 [M, n] += x W^T (residual update) */
  DF_EPI_COUPLE_ADD = 3   /* z = x W^T; z[aux rows] += c (*) z[primary rows]; y fp32 += z.
                             epi_arg: device c [n], storage dtype; needs m_aux == m_primary */
};

/* Stacked-activation linear: rows 0..m_primary-1 of x are the primary flow, the next m_aux rows
 * the auxiliary flow; one read of W serves all of them. x: device [m_primary + m_aux, k] storage
 * dtype; W: device [n, k] storage dtype; y per `epilogue`. For bf16 contexts k must be a multiple
 * of 64, m_primary + m_aux <= 2 * max_batch (<= 256), x, W and epi_arg 16-byte aligned; each row's
 * result does not depend on the other rows present. */
DF_API int dualflow_stacked_linear(dualflow_ctx* ctx, const void* x, int32_t m_primary, int32_t m_aux, const void* W,
                            int32_t n, int32_t k, void* y, int32_t epilogue, const void* epi_arg,
                            dualflow_stream stream);

/* The MLP block of layer `layer` for both flows ("Acoplamento Leve"), in place on the fp32
 * residual h: device [2, batch, d] (flow-major). x_f = RMSNorm(h_f, g_mlp); dense:
 * u_f = silu(Wg x_f) (*) (Wu x_f), u2 += b (*) u1, y_f = Wd u_f; MoE ("Replay de Roteador"):
 * the primary picks its top-k_primary experts from its router logits, the auxiliary flow uses the
 * top-k_aux experts of the PRIMARY logits with softmax weights from its own logits, b couples an
 * expert's intermediate when both flows use it; then y2 += c (*) y1 and h_f += y_f.
 * expert_ids_out (MoE only, nullable): device int32 [2, batch, max(k_primary, k_aux)], experts of
 * each row in descending router logit order (ties to the lower index), -1 padded. */
DF_API int dualflow_coupled_mlp(dualflow_ctx* ctx, float* h, const dualflow_weights* w, int32_t layer, int32_t batch,
                         int32_t aux_on, int32_t* expert_ids_out, dualflow_stream stream);

/* Experts chosen in every layer by the last dualflow_step of this context (MoE models only, else
 * DF_ERR_UNSUPPORTED): copies [n_layers, 2, batch, max(k_primary, k_aux)] int32 into the device
 * buffer ids (row order as expert_ids_out of dualflow_coupled_mlp; flow-1 rows are -1 when the
 * step ran with aux_on = 0). batch must equal the step's batch. Asynchronous on `stream`. */
DF_API int dualflow_expert_ids(dualflow_ctx* ctx, int32_t* ids, int32_t batch, dualflow_stream stream);

/* Mixture head and token choice ("Objetivo de Mistura", gist.science technical summary, "Mecanismos
 * Chave": the two flows' next-token distributions are mixed with a weight on the primary that
 * grows with its confidence and is at least one half). Reading of this library:
 *   p_f = softmax(logits_f), alpha = 1/2 + 1/2 * sum_i p1_i^2, p_mix = alpha p1 + (1 - alpha) p2;
 *   token = argmax_i p_mix_i (ties to the lower index) when u is NULL, else the smallest i with
 *   p_mix_0 + ... + p_mix_i > u[b] (inverse-transform sampling; the last i with p_mix_i > 0 if
 *   rounding leaves no partial sum above u[b]).
 *   logits  device fp32 [2, batch, vocab] (flow-major, as written by dualflow_step), finite
 *   u       device fp32 [batch] uniforms in [0, 1), or NULL for greedy choice
 *   alpha   device fp32 [batch] or NULL;  p_mix  device fp32 [batch, vocab] or NULL
 *   token   device int32 [batch] or NULL
 * vocab is the context's. One launch on `stream`, nothing allocated, graph-capturable; fp32
 * arithmetic with every reduction in a fixed order (the outputs do not depend on scheduling).
 * Returns DF_ERR_ARG for a NULL context or logits, DF_ERR_SHAPE for batch outside
 * 1..max_batch; non-finite logits give unspecified (but in-bounds) tokens. */
DF_API int dualflow_mixture_head(dualflow_ctx* ctx, const float* logits, int32_t batch, const float* u, float* alpha,
                                 float* p_mix, int32_t* token, dualflow_stream stream);

/* The decode loop: n_steps decode steps in which each step's chosen token is the next step's input
 * (the technical summary's decode phase, "Custos de Inferencia vs. Treinamento": the auxiliary flow
 * is on at every generated token). Step t runs dualflow_step on the loop's token buffer, then the
 * mixture head and token choice of dualflow_mixture_head (from the primary's distribution alone
 * when aux_on = 0), then advances the cache: seq_len[b] += 1 and, for a paged cache, when the next
 * slot seq_len[b] opens a logical page whose table entry is -1, the top entry of the free-page
 * list is popped into the table (sequences in order b = 0, 1, ...). Everything stays on the GPU.
 *   tokens      device int32 [batch]: the first step's input tokens
 *   u           device fp32 [n_steps, batch] uniforms in [0, 1) (sampling), or NULL (argmax)
 *   tokens_out  device int32 [n_steps, batch]: token chosen after each step
 *   logits      device fp32 [2, batch, vocab]: workspace, holds the last step's logits on return
 *   logits_all  device fp32 [n_steps, 2, batch, vocab] or NULL: every step's logits
 *   free_pages  device int32 [*n_free], n_free device int32 (paged caches; NULL: no new pages)
 * kv->seq_len (device) is advanced in place by n_steps and kv->page_table written as above; the
 * first step's slot must already be mapped, as for dualflow_step. Asynchronous on `stream`;
 * nothing is allocated. A length reaching max_ctx, a page slot beyond the table or an empty free
 * list latches DF_ERR_DEVICE_BOUNDS and that sequence stops advancing (its later steps overwrite
 * the same slot). Host errors as for dualflow_step; n_steps < 0 is DF_ERR_SHAPE, 0 does nothing. */
DF_API int dualflow_generate(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv,
                             const int32_t* tokens, int32_t batch, int32_t n_steps, const float* u,
                             int32_t* tokens_out, float* logits, float* logits_all, int32_t* free_pages,
                             int32_t* n_free, int32_t aux_on, dualflow_stream stream);

/* Workspace for dualflow_prefill / dualflow_prefill_slots: room for max_rows = prompt sequences *
 * prompt tokens activation rows (about (4 d + 4 Hq D + 2 F + 4 ss) bytes per row; a MoE context
 * adds about k (6 d + 2 F + 4 ss + 8) + 12 E bytes per row, k = topk_primary). Allocates (cold
 * call, not for a hot loop); a smaller request than the current room does nothing. bf16 contexts,
 * dense or MoE with at most 32 experts (DF_ERR_UNSUPPORTED otherwise); DF_ERR_OOM leaves no
 * prefill room. */
DF_API int dualflow_prefill_reserve(dualflow_ctx* ctx, int32_t max_rows);

/* Primary-only prefill ("Custos de Inferencia vs. Treinamento", gist.science technical summary: the
 * auxiliary flow is off while a prompt is processed and on from the decode phase). tokens: device
 * int32 [batch, n_tok] row-major, token t of sequence b at position seq_len[b] + t. In one pass per
 * layer the primary flow's projections run on all batch * n_tok rows (tcgen05 tiles of 256 rows),
 * the keys/values of every prompt position are written into the cache, and each position attends
 * the cached positions 0 .. itself (causal). Then seq_len[b] += n_tok (device). No logits: the
 * caller runs the prompt's last token as the first decode step (dualflow_step / dualflow_generate),
 * where the auxiliary flow joins. A MoE layer routes every prompt row (top-k of its router
 * logits, the decode step's rule for the primary flow), gathers each expert's rows and runs that
 * expert's projections on them only. Needs dualflow_prefill_reserve(ctx, >= batch * n_tok)
 * (DF_ERR_SHAPE otherwise); bf16 contexts (dense, or MoE with at most 32 experts) with
 * G = Hq / Hkv in {1, 2, 4} (DF_ERR_UNSUPPORTED otherwise). A position seq_len[b] + t >= max_ctx latches
 * DF_ERR_DEVICE_BOUNDS; so does, with a paged cache, a prompt position whose page the table does
 * not map (this call takes no free list: see dualflow_prefill_slots). Asynchronous on `stream`,
 * launched eagerly (no graph). Same as dualflow_prefill_slots(ctx, w, kv, tokens, NULL, batch,
 * n_tok, NULL, NULL, stream). */
DF_API int dualflow_prefill(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv,
                            const int32_t* tokens, int32_t batch, int32_t n_tok, dualflow_stream stream);

/* Continuous batching, admission: the primary-only prefill of dualflow_prefill for n_seq prompts
 * (device int32 tokens [n_seq, n_tok]) into chosen cache slots: prompt i goes to slot slots[i]
 * (device int32 [n_seq], distinct values in [0, max_batch); NULL: slot i), at positions
 * seq_len[slots[i]] + t, and afterwards seq_len[slots[i]] += n_tok. The other slots' cache
 * entries, lengths and table rows are not touched. A new sequence enters a slot whose length is
 * 0 (dualflow_release_slots). Paged contexts: with a free list (free_pages: device int32 array of
 * free physical page ids, *n_free of them in use, the top at free_pages[*n_free - 1]; both NULL or
 * both set), first every page that positions seq_len[b] .. seq_len[b] + n_tok of a slot touch
 * (the prompt and the slot the next decode step writes, below max_ctx) and that the table does
 * not map yet is popped from the top of the free list, prompt by prompt in page order, on the
 * device; without one the table must already map the prompt's pages. An empty free list, a slot
 * outside [0, max_batch) or an unmapped page latches DF_ERR_DEVICE_BOUNDS and the affected
 * writes are skipped. Contiguous contexts take no free list (DF_ERR_ARG). n_seq in [1, max_batch]
 * and n_seq * n_tok <= the reserved rows (DF_ERR_SHAPE otherwise). Asynchronous on `stream`. */
DF_API int dualflow_prefill_slots(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv,
                                  const int32_t* tokens, const int32_t* slots, int32_t n_seq, int32_t n_tok,
                                  int32_t* free_pages, int32_t* n_free, dualflow_stream stream);

/* Continuous batching, retirement: ends the sequences held by the cache slots slots[0 .. n_slots)
 * (device int32, distinct values in [0, max_batch)). Every listed slot's length becomes 0; in a
 * paged context its mapped pages are pushed on top of the free list in page order
 * (free_pages[(*n_free)++] = page; the array must hold max_pages entries) and its table row is
 * set to -1. Cache contents are left as they are (a new sequence overwrites them). A slot outside
 * [0, max_batch), or a free list already holding max_pages entries, latches DF_ERR_DEVICE_BOUNDS.
 * Paged contexts need free_pages and n_free, contiguous ones take neither (DF_ERR_ARG);
 * 0 <= n_slots <= max_batch (DF_ERR_SHAPE). One device thread, asynchronous on `stream`. */
DF_API int dualflow_release_slots(dualflow_ctx* ctx, const dualflow_kv* kv, const int32_t* slots, int32_t n_slots,
                                  int32_t* free_pages, int32_t* n_free, dualflow_stream stream);

/* dualflow_generate with HOST buffers, for contiguous caches: copies tokens_host [batch] (and
 * u_host [n_steps, batch] if not NULL) to the device, runs n_steps of the decode loop (step, mixture
 * head, token choice, length advance), copies the chosen tokens back to tokens_out_host
 * [n_steps, batch] and synchronizes `stream`. 0 <= n_steps <= 256 (DF_ERR_SHAPE otherwise); the
 * context's own buffers hold the logits. Pinned host memory gives asynchronous copies. */
DF_API int dualflow_generate_host(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv,
                                  const int32_t* tokens_host, int32_t batch, int32_t n_steps, const float* u_host,
                                  int32_t* tokens_out_host, int32_t aux_on, dualflow_stream stream);

/* One whole decode step of both flows: embeddings E1[tok], E2[tok] -> n_layers x {RMSNorm,
 * QKV with query coupling, RoPE and primary-only KV append, shared-KV attention, O projection,
 * coupled MLP} -> final RMSNorm -> shared LM head.
 * tokens: device int32 [batch]; logits: device fp32 [2, batch, vocab] (aux rows written only
 * when aux_on). Writes slot seq_len[b] of every layer's K1/V1 and nothing else of the cache.
 * On a non-default stream the first call for a given set of arguments captures the step into a
 * CUDA graph and later identical calls replay it (see dualflow_set_graphs). */
DF_API int dualflow_step(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv, const int32_t* tokens,
                  int32_t batch, float* logits, int32_t aux_on, dualflow_stream stream);

/* dualflow_step with HOST token and logit buffers: copies tokens_host [batch] to the device,
 * runs the step, copies logits [2, batch, vocab] back to logits_host and synchronizes `stream`.
 * Pinned host memory gives asynchronous copies. */
DF_API int dualflow_step_host(dualflow_ctx* ctx, const dualflow_weights* w, const dualflow_kv* kv,
                       const int32_t* tokens_host, int32_t batch, float* logits_host, int32_t aux_on,
                       dualflow_stream stream);

/* Enables (1, default) or disables (0) CUDA-graph capture and replay in dualflow_step. */
DF_API int dualflow_set_graphs(dualflow_ctx* ctx, int32_t enabled);

/* Kernel families reported by dualflow_profile_read. */
enum {
  DF_PROF_NORM = 0,      /* embedding gather and RMSNorm */
  DF_PROF_QKV = 1,       /* QKV projection with query coupling, RoPE and KV append */
  DF_PROF_ATTN = 2,      /* shared-KV decode attention */
  DF_PROF_OPROJ = 3,     /* O projection and residual */
  DF_PROF_GATEUP = 4,    /* gate/up projection with SwiGLU and b coupling */
  DF_PROF_DOWN = 5,      /* down projection with c coupling and residual */
  DF_PROF_LMHEAD = 6,    /* shared LM head */
  DF_PROF_OTHER = 7,     /* fp32-path helpers */
  DF_PROF_FAMILIES = 8
};

/* Per-kernel timing of dualflow_step (mode 0: off, the default).
 *   mode 1: every kernel the step launches is bracketed by a CUDA event pair on the launching
 *           stream (captured into the step's CUDA graph when graphs are on). The event records
 *           serialise the launches, so a kernel's time includes its full start-up: a stand-alone
 *           duration, not its share of the pipelined step.
 *   mode 2: every kernel raises a per-launch device slot to the globaltimer value at which its
 *           CTAs finish (the step's first kernel also records the step's start); nothing is
 *           serialised. A launch's time is then its share of the step: from the end of the launch
 *           before it to its own end, and the shares of one step add up to the step. bf16 storage
 *           only (DF_ERR_UNSUPPORTED for fp32).
 * Changing the mode drops the cached graphs. DF_ERR_ARG for another mode. */
DF_API int dualflow_set_profiling(dualflow_ctx* ctx, int32_t mode);

/* Synchronizes the device and reports the last dualflow_step: launches[f] = kernels of family f
 * it launched (always available) and ms[f] = their summed time in the current profiling mode
 * (all 0 in mode 0). Either array may be NULL; n_families entries are written (at most
 * DF_PROF_FAMILIES). With graphs on, the last step is the last replay of the last captured graph. */
DF_API int dualflow_profile_read(dualflow_ctx* ctx, float* ms, int32_t* launches, int32_t n_families);

/* Enables (1) or disables (0, default) chaining of dualflow_decode_attention's first kernel to the
 * kernel that precedes the call on a non-NULL stream, by programmatic dependent launch: the call
 * then starts while that kernel finishes, and may read Wq and the cached K/V of positions below
 * seq_len[b] before that kernel's writes are visible. Only for callers whose preceding kernel
 * writes none of them (back-to-back calls of this library qualify: they write o only). */
DF_API int dualflow_set_call_chaining(dualflow_ctx* ctx, int32_t enabled);

/* Enables (1) or disables (0, default) NVTX ranges: one per layer of dualflow_step and one per
 * kernel launch, named after the families above. They are host-side ranges around the launches,
 * so they show up for eager launches (dualflow_set_graphs(ctx, 0)) and for the capture of a step's
 * graph, not for its replays. */
DF_API int dualflow_set_nvtx(dualflow_ctx* ctx, int32_t enabled);

/* Limit, in nanoseconds, of the kernels' bounded pipeline waits (0 restores the default of one
 * second). Meant for tests of the failure path only: with a limit far below a copy's latency the
 * waits expire, the step reports DF_ERR_TIMEOUT through dualflow_sync_status and its outputs are
 * garbage, while every asynchronous copy a kernel issued is still awaited (with the default limit)
 * before its CTA exits. Changing the limit drops the cached graphs. DF_ERR_ARG if negative. */
DF_API int dualflow_set_wait_limit(dualflow_ctx* ctx, int64_t limit_ns);

/* Router logits of the context's last MoE computation ("Replay de Roteador", gist.science technical
 * summary, "Mecanismos Chave": the shared router scores every expert for both flows; the primary
 * flow's scores choose the experts). Copies device fp32 [n_layers, 2, batch, n_experts] (flow-major
 * rows as in the step) into the device buffer `logits`: layer l of the last dualflow_step, or of
 * the last dualflow_coupled_mlp call on layer l. The flow-1 rows of a layer are stale when that
 * layer last ran with aux_on = 0. batch must equal the one of those calls. DF_ERR_UNSUPPORTED for
 * dense configurations. Asynchronous on `stream`. */
DF_API int dualflow_router_logits(dualflow_ctx* ctx, float* logits, int32_t batch, dualflow_stream stream);

/* Synchronizes `stream`, then returns and clears the device status word: DF_OK, or the first
 * DF_ERR_DEVICE_BOUNDS / DF_ERR_TIMEOUT latched by a kernel since the last call. After
 * DF_ERR_TIMEOUT it also clears the attention kernel's merge counters, which a kernel that stopped
 * early may have left behind, so the context is usable again (the outputs of the failed calls are
 * not). */
DF_API int dualflow_sync_status(dualflow_ctx* ctx, dualflow_stream stream);

/* Largest batch * n_kv_heads that dualflow_decode_attention_noalloc accepts. */
#define DF_NOALLOC_MAX_PAIRS 512

/* Shared-KV decode attention (the attention kernel of dualflow_decode_attention) that allocates
 * nothing. The pages describe no such call: it exists for callers that may not call cudaMalloc --
 * an application whose own pool owns all device memory, a plugin restricted to the buffers it is
 * handed, or a latency-critical program that cannot accept cudaMalloc's implicit device-wide
 * synchronisation -- and so cannot create a context (dualflow_init allocates its workspace).
 *
 * It takes no context. The attention's scratch (split-KV partials, merge counters, a status word;
 * about 3.4 MB) lives in one statically sized device array of the library, which every device
 * that loads the library holds until the process exits. Limits: batch * cfg->n_kv_heads <=
 * DF_NOALLOC_MAX_PAIRS, else DF_ERR_SHAPE before any launch; bf16 storage only, with the same
 * head_dim / group / page-size limits as dualflow_init (DF_ERR_UNSUPPORTED otherwise).
 *   cfg     host; n_q_heads, n_kv_heads, head_dim, dtype, paged, page_size, max_batch, max_ctx,
 *           max_pages describe the cache layout exactly as for dualflow_init (other fields unused)
 *   q       device bf16 [2, batch, Hq, D], 16-byte aligned: both flows' queries, already coupled
 *           and rotated (the queries dualflow_decode_attention forms internally); flow 1 rows read
 *           only if aux_on
 *   kv      host struct of device pointers, as for dualflow_decode_attention; layer selects k/v
 *   o       device bf16 [2, batch, Hq, D]: o_f = softmax(q_f K1^T / sqrt(D)) V1 over the cached
 *           positions 0..seq_len[b]-1; seq_len[b] == 0 gives o = 0; flow 1 written only if aux_on
 *   status  device int32 or NULL: a device-side bounds error (out-of-range page id or length) or
 *           an expired bounded wait is latched there (set only if it holds 0; the caller clears
 *           it). With NULL the code is latched in the library's array, where the caller cannot
 *           read it.
 * The first call on a device (with that device current) looks up the array's device address;
 * make that first call before any stream capture. The address is kept for the life of the
 * process: after cudaDeviceReset (or any reset of the device's primary context) the array is
 * loaded anew, so this call must not be used across such a reset. Every call clears the merge counters it uses
 * with cudaMemsetAsync on `stream`, then launches one kernel there. All calls on a device share
 * the one array, so calls that may overlap on the GPU (other streams, other host threads) race on
 * it and must be serialised by the caller. */
DF_API int dualflow_decode_attention_noalloc(const dualflow_config* cfg, const void* q, const dualflow_kv* kv,
                                             int32_t layer, int32_t batch, void* o, int32_t aux_on,
                                             int32_t* status, dualflow_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* DUALFLOW_H */
