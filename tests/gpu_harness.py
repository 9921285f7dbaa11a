"""Builds the same seeded workload twice: on the device for the CUDA path (filled in place by the
generator's device fill) and lazily on the host, widened to fp64, for the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import dfsynth
import dual_flow_decode_dualflow_b300 as dfl
import oracle as O
from dfsynth import workloads as W

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _host_to_torch(host: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(host).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(host, dtype=np.float32))


def device_tensor(w: W.Workload, spec: W.TensorSpec, dev) -> torch.Tensor:
    t = torch.empty(spec.shape, dtype=TORCH_DT[w.dtype], device=dev)
    if spec.dist == "gain" or spec.numel < 4096:
        t.copy_(_host_to_torch(W.host_tensor(w, spec), w.dtype).reshape(spec.shape))
    else:
        dfsynth.cuda_normal_(t.data_ptr(), w.seed, spec.name, spec.numel, spec.sigma, w.dtype)
    return t


def config_for(w: W.Workload) -> dfl.dualflow_config:
    paged = int(w.paged)
    max_pages = w.page_table()[1] if w.paged else 0
    return dfl.make_config(
        n_layers=w.n_layers if w.kind == "step" else 1, d_model=w.d_model, n_q_heads=w.n_q_heads,
        n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, ffn_hidden=w.ffn_hidden, vocab=w.vocab,
        n_experts=w.n_experts, topk_primary=w.topk_primary, topk_aux=w.topk_aux,
        dtype=dfl.DF_DTYPE_BF16 if w.dtype == "bf16" else dfl.DF_DTYPE_F32, paged=paged, page_size=w.page_size,
        max_batch=w.batch, max_ctx=w.max_ctx, max_pages=max_pages, rope_base=w.rope_base, rms_eps=w.rms_eps)


class DeviceRun:
    """Device tensors, library context and C structs of one workload."""

    def __init__(self, w: W.Workload, dev, overrides: dict | None = None):
        self.w, self.dev = w, dev
        self.t = {}
        for spec in W.all_specs(w):
            self.t[spec.name] = device_tensor(w, spec, dev)
        for k, v in (overrides or {}).items():
            self.t[k] = v
        self.seq_len_np = w.seq_lens()
        self.seq_len = torch.from_numpy(self.seq_len_np).to(dev)
        self.table = None
        if w.paged:
            self.table_np, _ = w.page_table()
            self.table = torch.from_numpy(self.table_np).to(dev)
        self.ctx = dfl.dualflow_init(config_for(w))
        if w.kind == "step":
            self.tokens_np = w.tokens()
            self.tokens = torch.from_numpy(self.tokens_np).to(dev)
            self.rebuild_structs()
            self.logits = torch.full((2, w.batch, w.vocab), float("nan"), device=dev)
        else:
            self.kv = dfl.make_kv([self.t["K"]], [self.t["V"]], self.seq_len, self.table)
            self.o = torch.full((2, w.batch, w.n_q_heads, w.head_dim), float("nan"), dtype=TORCH_DT[w.dtype],
                                device=dev)

    def rebuild_structs(self):
        w, t = self.w, self.t
        layers = []
        for l in range(w.n_layers):
            names = ["g_attn", "g_mlp", "Wqkv", "Wo", "a", "b", "c"] + (
                ["Wgu", "Wd"] if w.n_experts == 0 else ["Wr", "We_gu", "We_d"])
            layers.append({n: t[f"L{l}.{n}"] for n in names})
        self.weights = dfl.make_weights(w.n_layers, t["E1"], t["E2"], t["W_lm"], t["g_final"], layers)
        self.kv = dfl.make_kv([t[f"L{l}.K"] for l in range(w.n_layers)], [t[f"L{l}.V"] for l in range(w.n_layers)],
                              self.seq_len, self.table)

    def step(self, aux_on=1, stream=None):
        dfl.dualflow_step(self.ctx, self.weights, self.kv, self.tokens, self.w.batch, self.logits, aux_on, stream)

    def attention(self, aux_on=1, stream=None):
        t = self.t
        dfl.dualflow_decode_attention(self.ctx, t["q1"], t["h2"], t["Wq"], t["a"], self.kv, 0, self.w.batch, self.o,
                                      aux_on, stream)

    def status(self):
        return dfl.dualflow_sync_status(self.ctx)

    def close(self):
        if self.ctx:
            dfl.dualflow_free(self.ctx)
            self.ctx = None


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


# ---------------------------------------------------------------------------------------------
# oracle-side inputs (host generator, widened lazily)
# ---------------------------------------------------------------------------------------------

def hparams(w: W.Workload) -> O.HParams:
    return O.HParams(d_model=w.d_model, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                     ffn_hidden=w.ffn_hidden, vocab=w.vocab, dtype=w.dtype, rope_base=w.rope_base,
                     rms_eps=w.rms_eps, n_experts=w.n_experts, topk_primary=w.topk_primary, topk_aux=w.topk_aux)


def _spec(w, name):
    for s in W.all_specs(w) if w.kind == "step" else W.global_specs(w):
        if s.name == name:
            return s
    raise KeyError(name)


def host_f64(w: W.Workload, name: str, overrides: dict | None = None) -> np.ndarray:
    if overrides and name in overrides:
        return overrides[name]
    spec = _spec(w, name)
    return O.widen(W.host_tensor(w, spec), w.dtype).reshape(spec.shape)


class LazyRows:
    """rows[i] of a [n, d] tensor, drawn on demand."""

    def __init__(self, w, name):
        self.w, self.spec = w, _spec(w, name)
        self.d = self.spec.shape[-1]

    def __getitem__(self, i):
        return O.widen(W.host_tensor(self.w, self.spec, offset=int(i) * self.d, count=self.d), self.w.dtype)


class LazyLayers:
    def __init__(self, w, overrides=None):
        self.w, self.overrides = w, overrides or {}
        self._cache = (None, None)

    def __len__(self):
        return self.w.n_layers

    def __getitem__(self, l):
        if self._cache[0] == l:
            return self._cache[1]
        names = [s.name for s in W.layer_specs(self.w, l) if not s.name.endswith((".K", ".V"))]
        d = {n.split(".", 1)[1]: host_f64(self.w, n, self.overrides) for n in names}
        self._cache = (l, d)
        return d


class LazySeqCache:
    """K[b] / V[b] of a contiguous [B, Hkv, cap, D] cache tensor, drawn per sequence."""

    def __init__(self, w, name):
        self.w, self.spec = w, _spec(w, name)
        self.per = int(np.prod(self.spec.shape[1:]))

    def __getitem__(self, b):
        x = W.host_tensor(self.w, self.spec, offset=int(b) * self.per, count=self.per)
        return O.widen(x, self.w.dtype).reshape(self.spec.shape[1:])


class LazyPages:
    """Physical page pid of a paged [P, Hkv, page, D] cache tensor."""

    def __init__(self, w, name):
        self.w, self.spec = w, _spec(w, name)
        self.per = int(np.prod(self.spec.shape[1:]))

    def __getitem__(self, pid):
        x = W.host_tensor(self.w, self.spec, offset=int(pid) * self.per, count=self.per)
        return O.widen(x, self.w.dtype).reshape(self.spec.shape[1:])


def oracle_cache(w: W.Workload, layer: int | None):
    kn = "K" if layer is None else f"L{layer}.K"
    vn = "V" if layer is None else f"L{layer}.V"
    if w.paged:
        table, _ = w.page_table()
        return O.PagedCache(LazyPages(w, kn), LazyPages(w, vn), table, w.page_size)
    return O.DenseCache(LazySeqCache(w, kn), LazySeqCache(w, vn))


class LazyCaches:
    def __init__(self, w):
        self.w = w

    def __len__(self):
        return self.w.n_layers

    def __getitem__(self, l):
        return oracle_cache(self.w, l)


def oracle_step(w: W.Workload, rows=None, aux_on=True, mirror=True, overrides=None, ids_override=None):
    glob = {"E1": LazyRows(w, "E1"), "E2": LazyRows(w, "E2"), "W_lm": host_f64(w, "W_lm", overrides),
            "g_final": host_f64(w, "g_final", overrides)}
    for k in ("E1", "E2"):
        if overrides and k in overrides:
            glob[k] = overrides[k]
    return O.decode_step(hparams(w), glob, LazyLayers(w, overrides), LazyCaches(w), w.tokens(), w.seq_lens(),
                         aux_on=aux_on, mirror=mirror, rows=rows, ids_override=ids_override)


def oracle_attention(w: W.Workload, rows=None, aux_on=True, mirror=True):
    q1 = host_f64(w, "q1")
    h2 = host_f64(w, "h2")
    return O.attention_only_step(hparams(w), q1, h2, host_f64(w, "Wq"), host_f64(w, "a"), oracle_cache(w, None),
                                 w.seq_lens(), aux_on=aux_on, mirror=mirror, rows=rows)


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max_i |g_i - r_i| / max_i |r_i| over one output tensor."""
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))
