// Allocation-free entry point for the shared-KV decode attention kernel.
//
// dualflow_decode_attention needs a context, and dualflow_init allocates the context's workspace
// with cudaMalloc. Some callers cannot do that: a host application that hands every byte of device
// memory to its own pool, a plugin that may only use the buffers it is given, or a latency-critical
// multi-stream program for which cudaMalloc's implicit device-wide synchronisation is not
// acceptable. For them this file keeps the attention kernel's scratch (split-KV partials, merge
// counters, a status word) in one file-scope device array, sized for a stated maximum problem, so
// a call launches the kernel on buffers the caller already owns and allocates nothing.
#include <string.h>

#include <mutex>

#include "internal.h"

using namespace df;

namespace {

constexpr int kMaxPairs = DF_NOALLOC_MAX_PAIRS;  // batch * n_kv_heads per call
constexpr int kMaxCtas = 320;                    // persistent grid: 2 CTAs per SM, capped
constexpr size_t kPartBytes = (size_t)(kMaxPairs + kMaxCtas) * kAttnPartFloats * sizeof(float);
constexpr size_t kCntOffset = kPartBytes;                                   // int32 [kMaxPairs]
constexpr size_t kStatusOffset = kCntOffset + (size_t)kMaxPairs * sizeof(int32_t);  // int32
constexpr size_t kScratchBytes = kStatusOffset + 256;
constexpr int kMaxDevices = 64;

// About 3.4 MB, held on every device that loads the library until the process exits.
static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

struct DeviceScratch {
  unsigned char* base = nullptr;  // device address of g_attn_scratch on this device
  int ctas = 0;
};

std::mutex g_mu;
DeviceScratch g_scratch[kMaxDevices];

// First call on a device (made with that device current): look up the array's device address
// and the SM count. The host-side symbol is only a stand-in and is never passed to a kernel.
int scratch_for_current_device(DeviceScratch* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DF_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DF_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceScratch& d = g_scratch[dev];
  if (d.base == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_attn_scratch) != cudaSuccess || ptr == nullptr) return DF_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return DF_ERR_CUDA;
    d.ctas = 2 * sms < kMaxCtas ? 2 * sms : kMaxCtas;
    d.base = static_cast<unsigned char*>(ptr);
  }
  *out = d;
  return DF_OK;
}

}  // namespace

extern "C" int dualflow_decode_attention_noalloc(const dualflow_config* cfg, const void* q, const dualflow_kv* kv,
                                                 int32_t layer, int32_t batch, void* o, int32_t aux_on,
                                                 int32_t* status, dualflow_stream stream) {
  if (!cfg || !q || !o || !kv || !kv->k || !kv->v || !kv->seq_len) return DF_ERR_ARG;
  if (aux_on != 0 && aux_on != 1) return DF_ERR_ARG;
  if (layer < 0 || layer >= kv->n_layers || !kv->k[layer] || !kv->v[layer]) return DF_ERR_ARG;
  if (cfg->dtype != DF_DTYPE_BF16) return cfg->dtype == DF_DTYPE_F32 ? DF_ERR_UNSUPPORTED : DF_ERR_DTYPE;
  if (cfg->n_q_heads <= 0 || cfg->n_kv_heads <= 0 || cfg->max_batch <= 0 || cfg->max_ctx <= 0) return DF_ERR_ARG;
  if (cfg->n_q_heads % cfg->n_kv_heads != 0) return DF_ERR_SHAPE;
  if (cfg->head_dim != kHeadDim || 2 * (cfg->n_q_heads / cfg->n_kv_heads) > kMaxGroupRows) return DF_ERR_UNSUPPORTED;
  if (cfg->paged) {
    if (!kv->page_table || cfg->max_pages <= 0) return DF_ERR_ARG;
    if (cfg->page_size != 16 && cfg->page_size != 32 && cfg->page_size != 64) return DF_ERR_UNSUPPORTED;
  }
  if (batch <= 0 || batch > cfg->max_batch) return DF_ERR_SHAPE;
  if ((long long)batch * cfg->n_kv_heads > kMaxPairs) return DF_ERR_SHAPE;

  DeviceScratch d;
  int rc = scratch_for_current_device(&d);
  if (rc != DF_OK) return rc;
  float* part = reinterpret_cast<float*>(d.base);
  int32_t* cnt = reinterpret_cast<int32_t*>(d.base + kCntOffset);
  int32_t* st = status ? status : reinterpret_cast<int32_t*>(d.base + kStatusOffset);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The merge counters must start at zero; a call that stopped early could have left some behind.
  const size_t pairs = (size_t)batch * cfg->n_kv_heads;
  if (cudaMemsetAsync(cnt, 0, pairs * sizeof(int32_t), s) != cudaSuccess) return DF_ERR_CUDA;
  if (!status && cudaMemsetAsync(st, 0, sizeof(int32_t), s) != cudaSuccess) return DF_ERR_CUDA;

  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.o = o;
  a.k_cache = kv->k[layer];
  a.v_cache = kv->v[layer];
  a.seq_len = kv->seq_len;
  a.page_table = kv->page_table;
  a.batch = batch;
  a.n_q_heads = cfg->n_q_heads;
  a.n_kv_heads = cfg->n_kv_heads;
  a.paged = cfg->paged;
  a.page_size = cfg->paged ? cfg->page_size : 1;
  a.max_ctx = cfg->max_ctx;
  a.max_pages = cfg->max_pages;
  a.pages_per_seq = cfg->paged ? (cfg->max_ctx + cfg->page_size - 1) / cfg->page_size : 0;
  a.extra = 0;
  a.aux_on = aux_on;
  return launch_attention_bf16_ws(*cfg, a, part, cnt, st, d.ctas, s);
}
