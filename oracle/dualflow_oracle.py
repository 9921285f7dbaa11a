"""Dual-Flow Transformer decode step: plain, slow CPU oracle in fp64.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the benchmark's
CPU-baseline / reference legs may import this module; the library's product path
never does, and this module imports nothing from the library. It shares no code
with the CUDA path: the only common piece is the seeded input generator (dfsynth),
which the callers use to draw inputs and which holds none of the method's arithmetic.

What it computes: one decode step of both flows, written out as the plain definition
(loops over batch rows, flows, heads and layers; explicit softmax over every key;
numpy's float64 matmul as the only library primitive). Sources, by page and section:

  [T1] "Resumo Tecnico: Dual-Flow Transformers" (gist.science, pt), section
       "Arquitetura Central" -- primary flow is a full causal transformer that writes the
       persistent KV cache and never depends on the auxiliary flow; the auxiliary flow reads
       the primary state and cache, never writes the cache, never feeds back; it is off in
       prefill and on from the last prompt position; both flows share every attention, MLP
       and output matrix; each flow has its own token embedding; light learned coupling.
  [T2] same page, "Mecanismos Chave", "Atencao de KV Compartilhada Assimetrica" -- the
       auxiliary query Q2 is coupled to the primary query Q1 through a_l and attends to the
       primary's K1, V1; "Acoplamento Leve" -- one-way coupling a_l, b_l, c_l at the query,
       the MLP intermediate and the MLP output; "Objetivo de Mistura" -- p_mix; "Replay de
       Roteador" -- the auxiliary flow reuses the primary router's experts with its own
       mixing weights.
  [T3] same page, "Custos de Inferencia vs. Treinamento" -- the only extra parameters are
       the embeddings and the coupling vectors (so norm gains and the LM head are shared).
  [T4] same page, "Contribuicoes Principais" -- Dense LLaMA and sparse LLaMA-style MoE
       model families (read as pre-RMSNorm, RoPE, SwiGLU, no biases); independent expert
       fan-outs for the two flows.

The pages name the coupling vectors but give no equations; this implementation fixes them as
    q2 = Wq.x2 + a (*) q1        u2 += b (*) u1        y2 += c (*) y1
(parity unpinned against the pages: no page states them). Readings taken where the pages
are silent, each one a choice of this implementation:
  R1 coupling acts on raw projections, before RoPE; q1, q2 share the position L_b.
  R2 u is the SwiGLU product (input of the down projection); y is the down-projection
     output before the residual; no coupling at the attention output.
  R3 the auxiliary flow attends K1/V1 at positions 0..L_b, including the entry the primary
     flow appends at L_b in this step (attention-only calls append nothing: 0..L_b-1).
  R4 RoPE rotate-half pairs (i, i + D/2), theta_i = base^(-2i/D), 0-based positions.
  R5 scale 1/sqrt(D); GQA maps query head h to KV head floor(h / G); no biases.
  R6 RMSNorm x = h / sqrt(mean(h^2) + eps) * g with eps = 1e-6; gains shared by the flows.
  R7 silu(z) = z * sigmoid(z); shared, untied LM head; shared final norm.
  R8 MoE: top-k by largest router logit, ties to the lower expert index; weights are the
     softmax over the selected k. The auxiliary set is the top-k_aux of the PRIMARY logits
     (replay, widened) and its weights the softmax of its own logits r2 over that set.
     b couples an expert's intermediate only when the expert is in both flows' sets.
  R9 mixture head: alpha = 1/2 + 1/2 * sum_i p1_i^2 (collision probability mapped to [1/2, 1]).
  R10 an attention-only call on a sequence with nothing cached (L_b = 0) returns o = 0 (softmax
     over an empty set is undefined; the step itself always attends at least its own new entry).
  R11 token choice after the mixture head: greedy = argmax of p_mix (ties to the lower index), or
     inverse-transform sampling with a supplied uniform u in [0, 1): the smallest i whose
     cumulative probability exceeds u (the last i with p_i > 0 when rounding leaves none).
  R13 prefill: the primary flow alone processes a prompt's tokens in one pass, each position
     attending every earlier cached position and itself, and writes their keys/values into the
     cache; the auxiliary flow is turned on at the last prompt position, which the caller runs as
     the first decode step. Computed here as one primary-only decode step per prompt position (the
     plain definition: a causal pass computes exactly what a step at each position computes).
  R12 generation loop: each decode step appends the primary's k1/v1 at position seq_len[b] (the
     entry the step attended), seq_len[b] grows by one, and the token chosen from that step's
     mixture (R11) is the next step's input. With the auxiliary flow off the choice is made from
     the primary's distribution softmax(logits_1) alone.

Precision: inputs arrive as the stored values widened to fp64. With mirror=True and a bf16
workload the oracle rounds (to nearest bf16, ties to even) exactly where the GPU path stores
bf16: the operand of each norm-fed projection (the gain-scaled row g (*) h, whose product is
then scaled by 1/rms -- an exact rewriting of RMSNorm(h).W^T), the post-RoPE queries, the
appended k1/v1, the attention output o and the SwiGLU output u (after coupling); router logits
are rounded to fp32 before the top-k decision, the precision in which the GPU takes it.
Everything else is fp64. With mirror=False every step is the plain fp64 definition.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, Sequence

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------------------------

def widen(stored: np.ndarray, dtype: str) -> np.ndarray:
    """Stored tensor -> fp64 values. bf16 arrives as uint16 bit patterns, f32 as float32."""
    if dtype == "bf16":
        return (np.asarray(stored, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(F64)
    return np.asarray(stored, dtype=np.float32).astype(F64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (8 significant bits), ties to even."""
    x = np.asarray(x, dtype=F64)
    m, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)


def round_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=F64).astype(np.float32).astype(F64)


# ---------------------------------------------------------------------------------------------
# building blocks
# ---------------------------------------------------------------------------------------------

def rms_scale(h: np.ndarray, eps: float) -> np.ndarray:
    """1 / sqrt(mean(h^2) + eps) of each row of h (R6)."""
    return 1.0 / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)


def rmsnorm(h: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of each row of h with gain g (R6; LLaMA family of [T4], gains shared per [T3])."""
    return h * rms_scale(h, eps) * g


def rope(x: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotary embedding of vectors x[..., D] at position pos (R4: rotate-half pairs (i, i+D/2))."""
    D = x.shape[-1]
    half = D // 2
    theta = base ** (-2.0 * np.arange(half, dtype=F64) / D)
    ang = pos * theta
    cos, sin = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :half], x[..., half:]
    return np.concatenate([lo * cos - hi * sin, hi * cos + lo * sin], axis=-1)


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """Softmax attention of query rows q[R, D] over keys K[L, D] and values V[L, D] (R5).

    Scores s = q.k / sqrt(D) for every key; p = exp(s - max s) / sum; o = sum_j p_j v_j.
    """
    D = q.shape[-1]
    s = (q @ K.T) / np.sqrt(F64(D))
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ V


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def topk_lower_index(r: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries of r, largest first; equal values go to the lower index (R8)."""
    order = sorted(range(len(r)), key=lambda i: (-r[i], i))
    return np.array(order[:k], dtype=np.int64)


def softmax(z: np.ndarray) -> np.ndarray:
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


# ---------------------------------------------------------------------------------------------
# caches: the primary flow's single persistent K1/V1 store [T1]
# ---------------------------------------------------------------------------------------------

@dataclass
class DenseCache:
    """K[b] and V[b] give [Hkv, capacity, D] fp64 arrays (a full array or a dict of rows)."""
    K: object
    V: object

    def seq(self, b: int, L: int):
        return np.asarray(self.K[b], dtype=F64)[:, :L, :], np.asarray(self.V[b], dtype=F64)[:, :L, :]


@dataclass
class PagedCache:
    """Physical pages K[pid], V[pid] -> [Hkv, page_size, D]; table[b, j] = physical id of the
    sequence's j-th logical page. Positions are read in logical order."""
    K: object
    V: object
    table: np.ndarray
    page_size: int

    def seq(self, b: int, L: int):
        n = (L + self.page_size - 1) // self.page_size
        ks = [np.asarray(self.K[int(self.table[b, j])], dtype=F64) for j in range(n)]
        vs = [np.asarray(self.V[int(self.table[b, j])], dtype=F64) for j in range(n)]
        return np.concatenate(ks, axis=1)[:, :L, :], np.concatenate(vs, axis=1)[:, :L, :]


# ---------------------------------------------------------------------------------------------
# the decode step
# ---------------------------------------------------------------------------------------------

@dataclass
class HParams:
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_hidden: int
    vocab: int
    dtype: str
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    n_experts: int = 0
    topk_primary: int = 0
    topk_aux: int = 0


def _store(x, hp: HParams, mirror: bool):
    """The value the GPU path keeps at a bf16 storage point (identity otherwise)."""
    return round_bf16(x) if (mirror and hp.dtype == "bf16") else x


def _normed(h, g, hp: HParams, mirror: bool):
    """RMSNorm(h) with gain g as the input of a linear layer.

    RMSNorm(h).W^T = (1/rms(h)) ((g (*) h).W^T). The bf16 GPU path stores the gain-scaled row
    g (*) h as the product's operand and scales the fp32 product by 1/rms; mirror mode rounds at
    that storage point (the scale commutes with the product, so it is applied to the operand here).
    """
    if mirror and hp.dtype == "bf16":
        return round_bf16(h * g) * rms_scale(h, hp.rms_eps)
    return rmsnorm(h, g, hp.rms_eps)


def _attention_block(hp, P, x, cache, b, L, pos, aux_on, mirror, append):
    """Shared QKV, query coupling, RoPE, KV append and asymmetric shared-KV attention ([T2]).

    x: normed inputs of this batch row, x[0] primary, x[1] auxiliary. Returns (o[2, Hq*D],
    k_new[Hkv, D], v_new[Hkv, D]) where o[1] is NaN when the auxiliary flow is off.
    """
    Hq, Hkv, D = hp.n_q_heads, hp.n_kv_heads, hp.head_dim
    qd, kd = Hq * D, Hkv * D
    Wq, Wk, Wv = P["Wqkv"][:qd], P["Wqkv"][qd:qd + kd], P["Wqkv"][qd + kd:]
    q1 = Wq @ x[0]
    k1 = (Wk @ x[0]).reshape(Hkv, D)
    v1 = (Wv @ x[0]).reshape(Hkv, D)
    q = [rope(q1.reshape(Hq, D), pos, hp.rope_base)]
    if aux_on:
        q2 = Wq @ x[1] + P["a"] * q1  # query coupling, before RoPE (R1)
        q.append(rope(q2.reshape(Hq, D), pos, hp.rope_base))
    q = [_store(qf, hp, mirror) for qf in q]
    k_new = _store(rope(k1, pos, hp.rope_base), hp, mirror)
    v_new = _store(v1, hp, mirror)
    Kc, Vc = cache.seq(b, L)
    if append:  # the primary writes slot L; both flows attend it (R3)
        Kc = np.concatenate([Kc, k_new[:, None, :]], axis=1)
        Vc = np.concatenate([Vc, v_new[:, None, :]], axis=1)
    G = Hq // Hkv
    o = np.full((2, Hq, D), np.nan)
    for f in range(len(q)):
        for h in range(Hq):
            g = h // G
            o[f, h] = attention(q[f][h][None, :], Kc[g], Vc[g])[0]
    o = _store(o, hp, mirror)
    return o.reshape(2, qd), k_new, v_new


def _dense_mlp(hp, P, x, aux_on, mirror):
    """Shared SwiGLU MLP with intermediate coupling b and output coupling c ([T2], R2)."""
    F = hp.ffn_hidden
    Wg, Wu = P["Wgu"][:F], P["Wgu"][F:]
    u = [silu(Wg @ x[0]) * (Wu @ x[0])]
    if aux_on:
        u.append(silu(Wg @ x[1]) * (Wu @ x[1]) + P["b"] * u[0])
    u = [_store(uf, hp, mirror) for uf in u]
    y = [P["Wd"] @ uf for uf in u]
    if aux_on:
        y[1] = y[1] + P["c"] * y[0]
    return y


def route(hp, r1, r2, aux_on):
    """Router replay ([T2] "Replay de Roteador", independent fan-outs [T4], R8).

    Returns (S1, w1, S2, w2): the primary's top-k1 experts of its own logits with softmax
    weights, and the auxiliary set = top-k2 of the PRIMARY logits with softmax weights taken
    from the auxiliary logits over that set.
    """
    S1 = topk_lower_index(r1, hp.topk_primary)
    w1 = softmax(r1[S1])
    if not aux_on:
        return S1, w1, None, None
    S2 = topk_lower_index(r1, hp.topk_aux)
    w2 = softmax(r2[S2])
    return S1, w1, S2, w2


def _moe_mlp(hp, P, x, aux_on, mirror, ids_override=None):
    """MoE SwiGLU experts shared by both flows with router replay and couplings b, c."""
    F = hp.ffn_hidden
    r1 = P["Wr"] @ x[0]
    r2 = P["Wr"] @ x[1] if aux_on else None
    if mirror:  # the top-k decision is taken on fp32 logits, as on the GPU
        r1 = round_f32(r1)
        r2 = round_f32(r2) if aux_on else None
    S1, w1, S2, w2 = route(hp, r1, r2, aux_on)
    if ids_override is not None:
        S1 = np.asarray(ids_override[0][: hp.topk_primary], dtype=np.int64)
        w1 = softmax(r1[S1])
        if aux_on:
            S2 = np.asarray(ids_override[1][: hp.topk_aux], dtype=np.int64)
            w2 = softmax(r2[S2])
    u1 = {}
    for e in S1:
        Wg, Wu = P["We_gu"][e][:F], P["We_gu"][e][F:]
        u1[int(e)] = silu(Wg @ x[0]) * (Wu @ x[0])
    y1 = np.zeros(hp.d_model)
    for e, w in zip(S1, w1):
        y1 = y1 + w * (P["We_d"][e] @ _store(u1[int(e)], hp, mirror))
    y = [y1]
    if aux_on:
        y2 = np.zeros(hp.d_model)
        for e, w in zip(S2, w2):
            Wg, Wu = P["We_gu"][e][:F], P["We_gu"][e][F:]
            u2 = silu(Wg @ x[1]) * (Wu @ x[1])
            if int(e) in u1:
                u2 = u2 + P["b"] * u1[int(e)]
            y2 = y2 + w * (P["We_d"][e] @ _store(u2, hp, mirror))
        y.append(y2 + P["c"] * y1)
    ids = np.full((2, max(hp.topk_primary, hp.topk_aux)), -1, dtype=np.int64)
    ids[0, : len(S1)] = S1
    if aux_on:
        ids[1, : len(S2)] = S2
    return y, ids, (r1, r2)


def decode_step(hp: HParams, glob: dict, layers: Sequence[dict], caches: Sequence, tokens: np.ndarray,
                seq_len: np.ndarray, aux_on: bool = True, mirror: bool = True, rows=None,
                ids_override: Callable | None = None, trace: list | None = None) -> dict:
    """One decode step of both flows for batch rows `rows` ([T1], [T2]).

    glob: E1, E2, W_lm, g_final (fp64). layers[l]: g_attn, g_mlp, Wqkv, Wo, a, b, c and either
    Wgu, Wd (dense) or Wr, We_gu, We_d (MoE). caches[l]: DenseCache or PagedCache of the
    pre-step K1/V1. seq_len[b] = cached positions before the step; the new token sits at
    position seq_len[b] and its primary key/value are appended there.

    Returns logits[2, R, V] (row 1 NaN when aux_on is False), k_new / v_new [n_layers, R, Hkv, D]
    and, for MoE, expert ids [n_layers, 2, R, max(k1, k2)] and router logits.
    """
    rows = list(range(len(tokens))) if rows is None else list(rows)
    R, nL = len(rows), len(layers)
    Hkv, D = hp.n_kv_heads, hp.head_dim
    h = np.full((2, R, hp.d_model), np.nan)
    for i, b in enumerate(rows):
        h[0, i] = glob["E1"][tokens[b]]  # separate token embeddings [T1]
        if aux_on:
            h[1, i] = glob["E2"][tokens[b]]
    k_new = np.zeros((nL, R, Hkv, D))
    v_new = np.zeros((nL, R, Hkv, D))
    kmax = max(hp.topk_primary, hp.topk_aux)
    ids = np.full((nL, 2, R, max(kmax, 1)), -1, dtype=np.int64)
    rlog = np.full((nL, 2, R, max(hp.n_experts, 1)), np.nan)
    nf = 2 if aux_on else 1
    for layer in range(nL):
        P = layers[layer]
        for i, b in enumerate(rows):
            L = int(seq_len[b])
            x = [_normed(h[f, i], P["g_attn"], hp, mirror) for f in range(nf)]
            o, k_new[layer, i], v_new[layer, i] = _attention_block(
                hp, P, x, caches[layer], b, L, L, aux_on, mirror, append=True)
            for f in range(nf):
                h[f, i] = h[f, i] + P["Wo"] @ o[f]  # shared O projection, residual
            x = [_normed(h[f, i], P["g_mlp"], hp, mirror) for f in range(nf)]
            if hp.n_experts == 0:
                y = _dense_mlp(hp, P, x, aux_on, mirror)
            else:
                ov = ids_override(layer, b) if ids_override is not None else None
                y, ids[layer, :, i], (r1, r2) = _moe_mlp(hp, P, x, aux_on, mirror, ov)
                rlog[layer, 0, i] = r1
                if aux_on:
                    rlog[layer, 1, i] = r2
            for f in range(nf):
                h[f, i] = h[f, i] + y[f]
            if trace is not None:
                trace.append(dict(layer=layer, b=b, o=o, h=h[:, i].copy()))
    logits = np.full((2, R, hp.vocab), np.nan)
    for f in range(nf):
        for i in range(R):
            xf = _normed(h[f, i], glob["g_final"], hp, mirror)
            logits[f, i] = glob["W_lm"] @ xf  # shared LM head [T1]
    return dict(logits=logits, k_new=k_new, v_new=v_new, expert_ids=ids, router_logits=rlog, h=h)


def attention_only_step(hp: HParams, q1: np.ndarray, h2: np.ndarray, Wq: np.ndarray, a: np.ndarray, cache,
                        seq_len: np.ndarray, aux_on: bool = True, mirror: bool = True, rows=None) -> np.ndarray:
    """Attention-only dual-flow decode call ([T2] asymmetric shared-KV attention).

    q1[B, Hq, D]: the primary's raw query projection; h2[B, d]: the auxiliary flow's normed
    input. q2 = Wq.h2 + a (*) q1; RoPE on q1 and q2 at position L_b; both attend the cached
    primary K1/V1 at positions 0..L_b-1 (nothing is appended). Returns o[2, R, Hq, D]
    (row 1 NaN when the auxiliary flow is off).
    """
    rows = list(range(q1.shape[0])) if rows is None else list(rows)
    Hq, Hkv, D = hp.n_q_heads, hp.n_kv_heads, hp.head_dim
    G = Hq // Hkv
    out = np.full((2, len(rows), Hq, D), np.nan)
    for i, b in enumerate(rows):
        L = int(seq_len[b])
        qs = [q1[b].reshape(-1)]
        if aux_on:
            qs.append(Wq @ h2[b] + a * q1[b].reshape(-1))
        qs = [_store(rope(qf.reshape(Hq, D), L, hp.rope_base), hp, mirror) for qf in qs]
        if L == 0:  # R10
            out[: len(qs), i] = 0.0
            continue
        Kc, Vc = cache.seq(b, L)
        for f in range(len(qs)):
            for h in range(Hq):
                out[f, i, h] = attention(qs[f][h][None, :], Kc[h // G], Vc[h // G])[0]
    return _store(out, hp, mirror)


def mixture_head(logits1: np.ndarray, logits2: np.ndarray):
    """Mixture of the two flows' next-token distributions ([T2] "Objetivo de Mistura", R9).

    p_f = softmax(logits_f); alpha = 1/2 + 1/2 * sum_i p1_i^2 (>= 1/2, grows with the primary's
    confidence); p_mix = alpha * p1 + (1 - alpha) * p2. Returns (alpha, p_mix, argmax p_mix).
    """
    p1, p2 = softmax(np.asarray(logits1, F64)), softmax(np.asarray(logits2, F64))
    alpha = 0.5 + 0.5 * float(np.sum(p1 * p1))
    pm = alpha * p1 + (1.0 - alpha) * p2
    return alpha, pm, int(np.argmax(pm))


def choice_distribution(logits1: np.ndarray, logits2: np.ndarray | None) -> np.ndarray:
    """The distribution the next token is chosen from (R11, R12): the mixture of both flows, or the
    primary's softmax alone when logits2 is None."""
    if logits2 is None:
        p = softmax(np.asarray(logits1, F64))
    else:
        _, p, _ = mixture_head(logits1, logits2)
    return p


def append_entry(cache, b: int, L: int, k: np.ndarray, v: np.ndarray) -> None:
    """Writes the primary's key/value [Hkv, D] at position L of sequence b (the cache arrays are
    written in place; a paged cache must map position L to a page)."""
    if isinstance(cache, PagedCache):
        pid = int(cache.table[b, L // cache.page_size])
        cache.K[pid][:, L % cache.page_size, :] = k
        cache.V[pid][:, L % cache.page_size, :] = v
    else:
        cache.K[b][:, L, :] = k
        cache.V[b][:, L, :] = v


def generate(hp: HParams, glob: dict, layers: Sequence[dict], caches: Sequence, tokens: np.ndarray,
             seq_len: np.ndarray, n_steps: int, u: np.ndarray | None = None, aux_on: bool = True,
             mirror: bool = True, token_override: Callable | None = None,
             ids_override: Callable | None = None) -> dict:
    """The decode loop (R12): n_steps decode steps of every sequence; after step t the appended
    entries join the caches, seq_len grows by one, and token[t, b] (R11; u[t, b] when sampling)
    feeds step t + 1. caches are written in place. token_override(t, b, token, p) may replace a
    choice made from distribution p (a caller resolving a near tie the way another implementation
    took it).

    Returns tokens [n_steps, B], logits [n_steps, 2, B, V] and the final seq_len."""
    tokens = np.array(tokens, dtype=np.int64)
    L = np.array(seq_len, dtype=np.int64)
    B = len(tokens)
    out_tok = np.zeros((n_steps, B), dtype=np.int64)
    out_logits = np.full((n_steps, 2, B, hp.vocab), np.nan)
    for t in range(n_steps):
        ov = (lambda l, b, t=t: ids_override(t, l, b)) if ids_override is not None else None
        r = decode_step(hp, glob, layers, caches, tokens, L, aux_on=aux_on, mirror=mirror, ids_override=ov)
        out_logits[t] = r["logits"]
        for layer in range(len(layers)):
            for b in range(B):
                append_entry(caches[layer], b, int(L[b]), r["k_new"][layer, b], r["v_new"][layer, b])
        for b in range(B):
            p = choice_distribution(r["logits"][0, b], r["logits"][1, b] if aux_on else None)
            tok = int(np.argmax(p)) if u is None else sample_inverse_cdf(p, float(u[t, b]))
            if token_override is not None:
                tok = int(token_override(t, b, tok, p))
            out_tok[t, b] = tok
        L = L + 1
        tokens = out_tok[t].copy()
    return dict(tokens=out_tok, logits=out_logits, seq_len=L)


def prefill(hp: HParams, glob: dict, layers: Sequence[dict], caches: Sequence, prompt: np.ndarray,
            seq_len: np.ndarray, mirror: bool = True) -> dict:
    """Primary-only prefill (R13) of prompt [B, n]: token t of sequence b sits at position
    seq_len[b] + t; its key/value enter the cache there (caches written in place). Returns the
    primary logits of every position [B, n, V], the final seq_len and, for MoE, the primary
    router logits of every position [n_layers, B, n, E]."""
    prompt = np.asarray(prompt, dtype=np.int64)
    B, n = prompt.shape
    L = np.array(seq_len, dtype=np.int64)
    logits = np.zeros((B, n, hp.vocab))
    rlog = np.full((len(layers), B, n, max(hp.n_experts, 1)), np.nan)
    for t in range(n):
        r = decode_step(hp, glob, layers, caches, prompt[:, t], L, aux_on=False, mirror=mirror)
        logits[:, t] = r["logits"][0]
        rlog[:, :, t] = r["router_logits"][:, 0]
        for layer in range(len(layers)):
            for b in range(B):
                append_entry(caches[layer], b, int(L[b]), r["k_new"][layer, b], r["v_new"][layer, b])
        L = L + 1
    return dict(logits=logits, seq_len=L, rlog=rlog)


def sample_inverse_cdf(p: np.ndarray, u: float) -> int:
    """Token drawn from the distribution p with the uniform u in [0, 1) (R11): the smallest i with
    p_0 + ... + p_i > u; if rounding leaves every partial sum <= u, the last i with p_i > 0."""
    p = np.asarray(p, F64)
    above = np.nonzero(np.cumsum(p) > u)[0]
    if len(above):
        return int(above[0])
    return int(np.nonzero(p > 0)[0][-1])
