"""Python binding of libdualflow.so (B300 Dual-Flow Transformer decode step).

Argument marshalling only: every step of the decode path runs in the library's CUDA kernels.
The functions carry the C ABI's names (include/dualflow.h); tensors are passed as raw device
pointers (torch tensors are accepted and converted with .data_ptr()), streams as cudaStream_t
handles (torch streams are accepted). A missing or unloadable library raises immediately:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int32, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdualflow.so")

DF_OK, DF_ERR_ARG, DF_ERR_SHAPE, DF_ERR_DTYPE, DF_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
DF_ERR_CUDA, DF_ERR_OOM, DF_ERR_DEVICE_BOUNDS, DF_ERR_TIMEOUT = 5, 6, 7, 8
DF_DTYPE_F32, DF_DTYPE_BF16 = 0, 1
DF_EPI_STORE_F32, DF_EPI_STORE_BF16, DF_EPI_ADD_F32, DF_EPI_COUPLE_ADD = 0, 1, 2, 3

C_FUNCTIONS = ("dualflow_init", "dualflow_free", "dualflow_status_string", "dualflow_decode_attention",
               "dualflow_stacked_linear", "dualflow_coupled_mlp", "dualflow_step", "dualflow_step_host",
               "dualflow_set_graphs", "dualflow_set_profiling", "dualflow_profile_read", "dualflow_sync_status",
               "dualflow_decode_attention_noalloc", "dualflow_expert_ids", "dualflow_mixture_head",
               "dualflow_generate", "dualflow_generate_host", "dualflow_prefill_reserve", "dualflow_prefill",
               "dualflow_prefill_slots", "dualflow_release_slots", "dualflow_set_nvtx", "dualflow_set_call_chaining",
               "dualflow_set_wait_limit", "dualflow_router_logits", "dualflow_cuda_error_string")
DF_PROF_FAMILIES = 8
DF_NOALLOC_MAX_PAIRS = 512  # the header's limit of batch * n_kv_heads for the context-free attention
PROF_NAMES = ("norm", "qkv", "attention", "o_proj", "gate_up", "down", "lm_head", "other")


class dualflow_config(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in ("n_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim", "ffn_hidden",
                                       "vocab", "n_experts", "topk_primary", "topk_aux", "dtype", "paged",
                                       "page_size", "max_batch", "max_ctx", "max_pages")] + [
        ("rope_base", c_float), ("rms_eps", c_float)]


_PP = POINTER(c_void_p)


class dualflow_weights(ctypes.Structure):
    _fields_ = [("E1", c_void_p), ("E2", c_void_p), ("W_lm", c_void_p), ("g_final", c_void_p),
                ("g_attn", _PP), ("g_mlp", _PP), ("Wqkv", _PP), ("Wo", _PP), ("Wgu", _PP), ("Wd", _PP),
                ("Wr", _PP), ("We_gu", _PP), ("We_d", _PP), ("a", _PP), ("b", _PP), ("c", _PP),
                ("n_layers", c_int32)]


class dualflow_kv(ctypes.Structure):
    _fields_ = [("k", _PP), ("v", _PP), ("page_table", c_void_p), ("seq_len", c_void_p), ("n_layers", c_int32)]


class DualFlowError(RuntimeError):
    def __init__(self, fn: str, code: int):
        detail = f": {dualflow_cuda_error_string()}" if code == DF_ERR_CUDA else ""
        super().__init__(f"{fn}: {dualflow_status_string(code)} (status {code}){detail}")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH):
    """Loads libdualflow.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libdualflow.so not found at {path}: run __graft_entry__.build() "
                          "(the decode path has no fallback without its CUDA library)")
    lib = ctypes.CDLL(path)
    i32, vp = c_int32, c_void_p
    sig = {
        "dualflow_init": ([POINTER(dualflow_config), POINTER(vp)], i32),
        "dualflow_free": ([vp], i32),
        "dualflow_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "dualflow_decode_attention": ([vp, vp, vp, vp, vp, POINTER(dualflow_kv), i32, i32, vp, i32, vp], i32),
        "dualflow_stacked_linear": ([vp, vp, i32, i32, vp, i32, i32, vp, i32, vp, vp], i32),
        "dualflow_coupled_mlp": ([vp, vp, POINTER(dualflow_weights), i32, i32, i32, vp, vp], i32),
        "dualflow_step": ([vp, POINTER(dualflow_weights), POINTER(dualflow_kv), vp, i32, vp, i32, vp], i32),
        "dualflow_step_host": ([vp, POINTER(dualflow_weights), POINTER(dualflow_kv), vp, i32, vp, i32, vp], i32),
        "dualflow_set_graphs": ([vp, i32], i32),
        "dualflow_set_profiling": ([vp, i32], i32),
        "dualflow_profile_read": ([vp, POINTER(c_float), POINTER(i32), i32], i32),
        "dualflow_sync_status": ([vp, vp], i32),
        "dualflow_decode_attention_noalloc": ([POINTER(dualflow_config), vp, POINTER(dualflow_kv), i32, i32, vp, i32,
                                               vp, vp], i32),
        "dualflow_expert_ids": ([vp, vp, i32, vp], i32),
        "dualflow_mixture_head": ([vp, vp, i32, vp, vp, vp, vp, vp], i32),
        "dualflow_generate": ([vp, POINTER(dualflow_weights), POINTER(dualflow_kv), vp, i32, i32, vp, vp, vp, vp, vp, vp,
                               i32, vp], i32),
        "dualflow_prefill_reserve": ([vp, i32], i32),
        "dualflow_prefill": ([vp, POINTER(dualflow_weights), POINTER(dualflow_kv), vp, i32, i32, vp], i32),
        "dualflow_prefill_slots": ([vp, POINTER(dualflow_weights), POINTER(dualflow_kv), vp, vp, i32, i32, vp, vp, vp],
                                   i32),
        "dualflow_release_slots": ([vp, POINTER(dualflow_kv), vp, i32, vp, vp, vp], i32),
        "dualflow_generate_host": ([vp, POINTER(dualflow_weights), POINTER(dualflow_kv), vp, i32, i32, vp, vp, i32, vp],
                                   i32),
        "dualflow_set_nvtx": ([vp, i32], i32),
        "dualflow_set_call_chaining": ([vp, i32], i32),
        "dualflow_set_wait_limit": ([vp, ctypes.c_int64], i32),
        "dualflow_router_logits": ([vp, vp, i32, vp], i32),
        "dualflow_cuda_error_string": ([], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a device pointer or a tensor, got {type(x)}")


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _check(fn: str, rc: int) -> None:
    if rc != DF_OK:
        raise DualFlowError(fn, rc)


def dualflow_status_string(code: int) -> str:
    return load_library().dualflow_status_string(code).decode()


def dualflow_cuda_error_string() -> str:
    """The last CUDA runtime error the library met in this host thread (diagnoses DF_ERR_CUDA)."""
    return load_library().dualflow_cuda_error_string().decode()


def dualflow_init(cfg: dualflow_config) -> int:
    lib = load_library()
    h = c_void_p()
    _check("dualflow_init", lib.dualflow_init(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def dualflow_init_status(cfg: dualflow_config) -> tuple[int, int | None]:
    """dualflow_init returning (status, handle) instead of raising."""
    lib = load_library()
    h = c_void_p()
    rc = lib.dualflow_init(ctypes.byref(cfg), ctypes.byref(h))
    return rc, h.value


def dualflow_free(ctx: int) -> None:
    _check("dualflow_free", load_library().dualflow_free(ctx))


def dualflow_decode_attention(ctx, q1, h2, Wq, a, kv: "dualflow_kv", layer: int, batch: int, o, aux_on: int,
                              stream=None) -> None:
    rc = load_library().dualflow_decode_attention(ctx, _ptr(q1), _ptr(h2), _ptr(Wq), _ptr(a), ctypes.byref(kv),
                                                  layer, batch, _ptr(o), aux_on, _stream(stream))
    _check("dualflow_decode_attention", rc)


def dualflow_stacked_linear(ctx, x, m_primary: int, m_aux: int, W, n: int, k: int, y, epilogue: int, epi_arg=None,
                            stream=None) -> None:
    rc = load_library().dualflow_stacked_linear(ctx, _ptr(x), m_primary, m_aux, _ptr(W), n, k, _ptr(y), epilogue,
                                                _ptr(epi_arg), _stream(stream))
    _check("dualflow_stacked_linear", rc)


def dualflow_coupled_mlp(ctx, h, w: "dualflow_weights", layer: int, batch: int, aux_on: int, expert_ids_out=None,
                         stream=None) -> None:
    rc = load_library().dualflow_coupled_mlp(ctx, _ptr(h), ctypes.byref(w), layer, batch, aux_on,
                                             _ptr(expert_ids_out), _stream(stream))
    _check("dualflow_coupled_mlp", rc)


def dualflow_step(ctx, w: "dualflow_weights", kv: "dualflow_kv", tokens, batch: int, logits, aux_on: int,
                  stream=None) -> None:
    rc = load_library().dualflow_step(ctx, ctypes.byref(w), ctypes.byref(kv), _ptr(tokens), batch, _ptr(logits),
                                      aux_on, _stream(stream))
    _check("dualflow_step", rc)


def dualflow_step_host(ctx, w: "dualflow_weights", kv: "dualflow_kv", tokens_host, batch: int, logits_host,
                       aux_on: int, stream=None) -> None:
    """tokens_host / logits_host: host pointers or pinned CPU tensors."""
    rc = load_library().dualflow_step_host(ctx, ctypes.byref(w), ctypes.byref(kv), _ptr(tokens_host), batch,
                                           _ptr(logits_host), aux_on, _stream(stream))
    _check("dualflow_step_host", rc)


def dualflow_set_graphs(ctx, enabled: int) -> None:
    _check("dualflow_set_graphs", load_library().dualflow_set_graphs(ctx, enabled))


def dualflow_set_profiling(ctx, mode: int) -> None:
    """0: off; 1: CUDA event pair around every launch (serialising); 2: in-graph end stamps, each
    launch's share of the step (no serialisation)."""
    _check("dualflow_set_profiling", load_library().dualflow_set_profiling(ctx, mode))


def dualflow_set_call_chaining(ctx, enabled: int) -> None:
    """Chains dualflow_decode_attention's first kernel to the caller's preceding kernel (see the header)."""
    _check("dualflow_set_call_chaining", load_library().dualflow_set_call_chaining(ctx, enabled))


def dualflow_set_nvtx(ctx, enabled: int) -> None:
    _check("dualflow_set_nvtx", load_library().dualflow_set_nvtx(ctx, enabled))


def dualflow_set_wait_limit(ctx, limit_ns: int) -> None:
    """Limit of the kernels' bounded pipeline waits in ns (0: default); failure-path tests only."""
    _check("dualflow_set_wait_limit", load_library().dualflow_set_wait_limit(ctx, limit_ns))


def dualflow_router_logits(ctx, logits, batch: int, stream=None) -> None:
    """Router logits of the last MoE computation: device fp32 [n_layers, 2, batch, n_experts]."""
    _check("dualflow_router_logits", load_library().dualflow_router_logits(ctx, _ptr(logits), batch,
                                                                            _stream(stream)))


def dualflow_profile_read(ctx) -> tuple[list[float], list[int]]:
    """(ms per kernel family, launches per kernel family) of the last dualflow_step."""
    ms = (c_float * DF_PROF_FAMILIES)()
    n = (c_int32 * DF_PROF_FAMILIES)()
    _check("dualflow_profile_read", load_library().dualflow_profile_read(ctx, ms, n, DF_PROF_FAMILIES))
    return list(ms), list(n)


def dualflow_decode_attention_noalloc(cfg: dualflow_config, q, kv: "dualflow_kv", layer: int, batch: int, o,
                                      aux_on: int, status=None, stream=None) -> None:
    """Decode attention without a context and without any device allocation (the library keeps
    the kernel's scratch in a static device array). q: both flows' coupled, rotated queries."""
    rc = load_library().dualflow_decode_attention_noalloc(ctypes.byref(cfg), _ptr(q), ctypes.byref(kv), layer, batch,
                                                          _ptr(o), aux_on, _ptr(status), _stream(stream))
    _check("dualflow_decode_attention_noalloc", rc)


def dualflow_expert_ids(ctx, ids, batch: int, stream=None) -> None:
    """Experts of every layer chosen by the last step: device int32 [n_layers, 2, batch, kmax]."""
    _check("dualflow_expert_ids", load_library().dualflow_expert_ids(ctx, _ptr(ids), batch, _stream(stream)))


def dualflow_mixture_head(ctx, logits, batch: int, u=None, alpha=None, p_mix=None, token=None, stream=None) -> None:
    """Mixture of both flows' next-token distributions and the token choice: logits device fp32
    [2, batch, vocab]; u device fp32 [batch] (sampling) or None (argmax); outputs nullable."""
    rc = load_library().dualflow_mixture_head(ctx, _ptr(logits), batch, _ptr(u), _ptr(alpha), _ptr(p_mix),
                                              _ptr(token), _stream(stream))
    _check("dualflow_mixture_head", rc)


def dualflow_generate(ctx, w: "dualflow_weights", kv: "dualflow_kv", tokens, batch: int, n_steps: int, tokens_out,
                      logits, u=None, logits_all=None, free_pages=None, n_free=None, aux_on: int = 1,
                      stream=None) -> None:
    """The decode loop: n_steps steps, each step's chosen token feeding the next (see the header)."""
    rc = load_library().dualflow_generate(ctx, ctypes.byref(w), ctypes.byref(kv), _ptr(tokens), batch, n_steps, _ptr(u),
                                          _ptr(tokens_out), _ptr(logits), _ptr(logits_all), _ptr(free_pages),
                                          _ptr(n_free), aux_on, _stream(stream))
    _check("dualflow_generate", rc)


def dualflow_generate_host(ctx, w: "dualflow_weights", kv: "dualflow_kv", tokens_host, batch: int, n_steps: int,
                           tokens_out_host, u_host=None, aux_on: int = 1, stream=None) -> None:
    """The decode loop with host token buffers (pinned CPU tensors): n_steps <= 256."""
    rc = load_library().dualflow_generate_host(ctx, ctypes.byref(w), ctypes.byref(kv), _ptr(tokens_host), batch,
                                               n_steps, _ptr(u_host), _ptr(tokens_out_host), aux_on, _stream(stream))
    _check("dualflow_generate_host", rc)


def dualflow_prefill_reserve(ctx, max_rows: int) -> None:
    """Allocates the prefill workspace for batch * prompt-token rows (cold call)."""
    _check("dualflow_prefill_reserve", load_library().dualflow_prefill_reserve(ctx, max_rows))


def dualflow_prefill(ctx, w: "dualflow_weights", kv: "dualflow_kv", tokens, batch: int, n_tok: int,
                     stream=None) -> None:
    """Primary-only prefill of tokens [batch, n_tok] at positions seq_len[b] + t (see the header)."""
    rc = load_library().dualflow_prefill(ctx, ctypes.byref(w), ctypes.byref(kv), _ptr(tokens), batch, n_tok,
                                         _stream(stream))
    _check("dualflow_prefill", rc)


def dualflow_prefill_slots(ctx, w: "dualflow_weights", kv: "dualflow_kv", tokens, slots, n_seq: int, n_tok: int,
                           free_pages=None, n_free=None, stream=None) -> None:
    """Primary-only prefill of tokens [n_seq, n_tok] into cache slots slots[i] (device int32, or
    None for 0 .. n_seq - 1); paged contexts may pass a free list to map the prompts' pages."""
    rc = load_library().dualflow_prefill_slots(ctx, ctypes.byref(w), ctypes.byref(kv), _ptr(tokens), _ptr(slots),
                                               n_seq, n_tok, _ptr(free_pages), _ptr(n_free), _stream(stream))
    _check("dualflow_prefill_slots", rc)


def dualflow_release_slots(ctx, kv: "dualflow_kv", slots, n_slots: int, free_pages=None, n_free=None,
                           stream=None) -> None:
    """Ends the sequences of cache slots slots[0 .. n_slots): lengths to 0, a paged slot's pages
    back on the free list."""
    rc = load_library().dualflow_release_slots(ctx, ctypes.byref(kv), _ptr(slots), n_slots, _ptr(free_pages),
                                               _ptr(n_free), _stream(stream))
    _check("dualflow_release_slots", rc)


def dualflow_sync_status(ctx, stream=None) -> int:
    """Returns (and clears) the device status word; raises only when the call itself fails."""
    rc = load_library().dualflow_sync_status(ctx, _stream(stream))
    if rc == DF_ERR_CUDA:
        raise DualFlowError("dualflow_sync_status", rc)
    return rc


# ---- struct builders (keep the returned objects alive while the library may read them) --------

def _arr(ptrs):
    n = len(ptrs)
    return (c_void_p * max(n, 1))(*[_ptr(p) for p in ptrs])


def make_weights(n_layers: int, E1, E2, W_lm, g_final, layers: list[dict]) -> dualflow_weights:
    """layers[l]: dict with g_attn, g_mlp, Wqkv, Wo, a, b, c and Wgu, Wd (dense) or Wr, We_gu, We_d (MoE)."""
    w = dualflow_weights()
    w.E1, w.E2, w.W_lm, w.g_final = _ptr(E1), _ptr(E2), _ptr(W_lm), _ptr(g_final)
    keep = []
    for name in ("g_attn", "g_mlp", "Wqkv", "Wo", "Wgu", "Wd", "Wr", "We_gu", "We_d", "a", "b", "c"):
        vals = [L.get(name) for L in layers]
        if all(v is None for v in vals):
            setattr(w, name, None)
            continue
        arr = _arr(vals)
        keep.append(arr)
        setattr(w, name, ctypes.cast(arr, _PP))
    w.n_layers = n_layers
    w._keep = keep
    return w


def make_kv(k_layers: list, v_layers: list, seq_len, page_table=None) -> dualflow_kv:
    kv = dualflow_kv()
    ka, va = _arr(k_layers), _arr(v_layers)
    kv.k, kv.v = ctypes.cast(ka, _PP), ctypes.cast(va, _PP)
    kv.page_table = _ptr(page_table)
    kv.seq_len = _ptr(seq_len)
    kv.n_layers = len(k_layers)
    kv._keep = (ka, va)
    return kv


def make_config(**kw) -> dualflow_config:
    c = dualflow_config()
    defaults = dict(n_experts=0, topk_primary=0, topk_aux=0, paged=0, page_size=16, max_pages=0, rope_base=10000.0,
                    rms_eps=1e-6)
    defaults.update(kw)
    for k, v in defaults.items():
        setattr(c, k, v)
    return c
