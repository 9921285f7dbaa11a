"""The synthetic decode workloads and the recipe that draws each of their tensors.

A workload fixes shapes, storage dtype, seed and the distribution of every input;
`tensor_specs` lists the tensors a run needs (name, shape, distribution), and the
fill helpers produce them on the host (numpy) or on the device (in place). No
arithmetic of the Dual-Flow method lives here.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

from . import host_gain, host_normal, host_permutation, host_uniform_int


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "step": the whole model's decode step; "attention": one attention-only layer call
    dtype: str  # storage dtype of weights, embeddings and cache: "f32" or "bf16"
    seed: int
    n_layers: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_hidden: int  # SwiGLU hidden (dense) or per-expert hidden (MoE)
    vocab: int
    batch: int
    ctx_len: int = 0  # every sequence's cached length; 0 means ragged lengths in [ctx_lo, ctx_hi]
    ctx_lo: int = 0
    ctx_hi: int = 0
    paged: bool = False
    page_size: int = 16
    n_experts: int = 0
    topk_primary: int = 0
    topk_aux: int = 0
    w_sigma: float = 0.02
    emb_sigma: float = 0.02
    kv_sigma: float = 1.0
    coup_sigma: float = 0.1
    act_sigma: float = 1.0
    gain_sigma: float = 0.0
    rope_base: float = 10000.0
    rms_eps: float = 1e-6

    # ---- derived sizes ----
    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def appends(self) -> bool:
        """The full step appends the new primary key/value at slot L_b; the attention-only call does not."""
        return self.kind == "step"

    def seq_lens(self) -> np.ndarray:
        if self.ctx_len > 0:
            return np.full(self.batch, self.ctx_len, dtype=np.int32)
        return host_uniform_int(self.seed, "seq_len", self.batch, self.ctx_lo, self.ctx_hi)

    @property
    def max_ctx(self) -> int:
        """Capacity (positions) of the contiguous cache: room for the appended slot, rounded up to 64."""
        longest = self.ctx_len if self.ctx_len > 0 else self.ctx_hi
        need = longest + (1 if self.appends else 0)
        return ((need + 63) // 64) * 64

    def pages_per_seq(self, lens: np.ndarray) -> np.ndarray:
        held = lens + (1 if self.appends else 0)
        return (held + self.page_size - 1) // self.page_size

    def page_table(self) -> tuple[np.ndarray, int]:
        """Shuffled page table int32[B, max_pages] (-1 = unused) and the number of physical pages."""
        lens = self.seq_lens()
        npg = self.pages_per_seq(lens)
        total = int(npg.sum())
        perm = host_permutation(self.seed, "pages", total)
        max_pages = (self.max_ctx + self.page_size - 1) // self.page_size
        table = np.full((self.batch, max_pages), -1, dtype=np.int32)
        off = 0
        for b in range(self.batch):
            table[b, : npg[b]] = perm[off : off + npg[b]]
            off += int(npg[b])
        return table, total

    def cache_shape(self) -> tuple[int, ...]:
        if self.paged:
            _, total = self.page_table()
            return (total, self.n_kv_heads, self.page_size, self.head_dim)
        return (self.batch, self.n_kv_heads, self.max_ctx, self.head_dim)

    def tokens(self) -> np.ndarray:
        return host_uniform_int(self.seed, "tokens", self.batch, 0, self.vocab - 1)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    dist: str  # "normal" or "gain"
    sigma: float

    @property
    def numel(self) -> int:
        return int(np.prod(self.shape))


def layer_specs(w: Workload, layer: int) -> list[TensorSpec]:
    d, F, E = w.d_model, w.ffn_hidden, w.n_experts
    p = f"L{layer}."
    out = [
        TensorSpec(p + "g_attn", (d,), "gain", w.gain_sigma),
        TensorSpec(p + "g_mlp", (d,), "gain", w.gain_sigma),
        TensorSpec(p + "Wqkv", (w.q_dim + 2 * w.kv_dim, d), "normal", w.w_sigma),
        TensorSpec(p + "Wo", (d, w.q_dim), "normal", w.w_sigma),
        TensorSpec(p + "a", (w.q_dim,), "normal", w.coup_sigma),
        TensorSpec(p + "b", (F,), "normal", w.coup_sigma),
        TensorSpec(p + "c", (d,), "normal", w.coup_sigma),
    ]
    if E == 0:
        out += [TensorSpec(p + "Wgu", (2 * F, d), "normal", w.w_sigma),
                TensorSpec(p + "Wd", (d, F), "normal", w.w_sigma)]
    else:
        out += [TensorSpec(p + "Wr", (E, d), "normal", w.w_sigma),
                TensorSpec(p + "We_gu", (E, 2 * F, d), "normal", w.w_sigma),
                TensorSpec(p + "We_d", (E, d, F), "normal", w.w_sigma)]
    out += [TensorSpec(p + "K", w.cache_shape(), "normal", w.kv_sigma),
            TensorSpec(p + "V", w.cache_shape(), "normal", w.kv_sigma)]
    return out


def global_specs(w: Workload) -> list[TensorSpec]:
    if w.kind == "attention":
        B, d = w.batch, w.d_model
        return [
            TensorSpec("q1", (B, w.n_q_heads, w.head_dim), "normal", w.act_sigma),
            TensorSpec("h2", (B, d), "normal", w.act_sigma),
            TensorSpec("Wq", (w.q_dim, d), "normal", w.w_sigma),
            TensorSpec("a", (w.q_dim,), "normal", w.coup_sigma),
            TensorSpec("K", w.cache_shape(), "normal", w.kv_sigma),
            TensorSpec("V", w.cache_shape(), "normal", w.kv_sigma),
        ]
    d, V = w.d_model, w.vocab
    return [
        TensorSpec("E1", (V, d), "normal", w.emb_sigma),
        TensorSpec("E2", (V, d), "normal", w.emb_sigma),
        TensorSpec("W_lm", (V, d), "normal", w.w_sigma),
        TensorSpec("g_final", (d,), "gain", w.gain_sigma),
    ]


def all_specs(w: Workload) -> list[TensorSpec]:
    out = global_specs(w)
    if w.kind == "step":
        for layer in range(w.n_layers):
            out += layer_specs(w, layer)
    return out


def host_tensor(w: Workload, spec: TensorSpec, offset: int = 0, count: int | None = None) -> np.ndarray:
    """Draw a tensor (or the flat slice [offset, offset+count)) on the host.

    bf16 storage comes back as uint16 bit patterns; f32 as float32.
    """
    if spec.dist == "gain":
        return host_gain(w.seed, spec.name, spec.shape, spec.sigma, w.dtype)
    if count is None:
        return host_normal(w.seed, spec.name, spec.shape, spec.sigma, w.dtype)
    return host_normal(w.seed, spec.name, (count,), spec.sigma, w.dtype, offset=offset)


# ---- the five decode workloads ------------------------------------------------------------

TINY_F32 = Workload(
    name="tiny_f32_1layer", kind="step", dtype="f32", seed=1001, n_layers=1, d_model=256, n_q_heads=4,
    n_kv_heads=4, head_dim=64, ffn_hidden=1024, vocab=512, batch=1, ctx_len=128,
    w_sigma=0.02, emb_sigma=0.1, kv_sigma=0.02, coup_sigma=0.1)

ATTN_B8_L2048 = Workload(
    name="attn_b8_l2048_bf16", kind="attention", dtype="bf16", seed=1002, n_layers=1, d_model=2048,
    n_q_heads=16, n_kv_heads=4, head_dim=128, ffn_hidden=0, vocab=0, batch=8, ctx_len=2048,
    w_sigma=0.02, kv_sigma=1.0, coup_sigma=0.1, act_sigma=1.0)

DENSE_24L_B32_L4096 = Workload(
    name="dense_24l_d2048_b32_l4096_bf16", kind="step", dtype="bf16", seed=1003, n_layers=24, d_model=2048,
    n_q_heads=16, n_kv_heads=4, head_dim=128, ffn_hidden=8192, vocab=32000, batch=32, ctx_len=4096,
    w_sigma=0.02, emb_sigma=0.02, kv_sigma=1.0, coup_sigma=0.1)

PAGED_RAGGED_B64 = Workload(
    name="attn_paged_ragged_b64_l1k-32k_bf16", kind="attention", dtype="bf16", seed=1004, n_layers=1,
    d_model=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, ffn_hidden=0, vocab=0, batch=64, ctx_len=0,
    ctx_lo=1024, ctx_hi=32768, paged=True, page_size=16, w_sigma=0.02, kv_sigma=1.0, coup_sigma=0.1)

# config 3's model on config 4's cache layout: pages of 16, shuffled, ragged lengths
DENSE_PAGED_RAGGED_B32 = DENSE_24L_B32_L4096.replace(
    name="dense_24l_d2048_b32_paged_l1k-32k_bf16", seed=1006, ctx_len=0, ctx_lo=1024, ctx_hi=32768, paged=True,
    page_size=16)

MOE_16L_B64 = Workload(
    name="moe_16l_e16_top2_top4_b64_l4096_bf16", kind="step", dtype="bf16", seed=1005, n_layers=16,
    d_model=2048, n_q_heads=16, n_kv_heads=4, head_dim=128, ffn_hidden=1408, vocab=32000, batch=64,
    ctx_len=4096, n_experts=16, topk_primary=2, topk_aux=4, w_sigma=0.02, emb_sigma=0.02, kv_sigma=1.0,
    coup_sigma=0.1)

WORKLOADS = {w.name: w for w in (TINY_F32, ATTN_B8_L2048, DENSE_24L_B32_L4096, PAGED_RAGGED_B64, MOE_16L_B64,
                                  DENSE_PAGED_RAGGED_B32)}
