"""Pins of the CPU oracle against things other than itself.

Each pin takes the oracle module and raises AssertionError when the oracle disagrees with a
closed form, an invariant of the method, a special case that reduces to a library routine
(torch / scipy / numpy complex arithmetic, all fp64), or brute force on a tiny input. The
same pins run against deliberately broken copies of the oracle (tests/test_oracle_pins.py)
to show that each plausible mistake is caught by at least one of them.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch
import torch.nn.functional as TF

F64 = np.float64


# ---------------------------------------------------------------------------------------------
# tiny random models (numpy RNG; the pins need no seeded workload)
# ---------------------------------------------------------------------------------------------

def tiny_hp(O, **kw):
    base = dict(d_model=16, n_q_heads=4, n_kv_heads=2, head_dim=8, ffn_hidden=24, vocab=13, dtype="f32",
                rope_base=10000.0, rms_eps=1e-6)
    base.update(kw)
    return O.HParams(**base)


def tiny_model(O, hp, n_layers=2, batch=2, ctx=(5, 3), seed=0, couple=True, tie_emb=False):
    rng = np.random.default_rng(seed)
    d, Hq, Hkv, D, F, V = hp.d_model, hp.n_q_heads, hp.n_kv_heads, hp.head_dim, hp.ffn_hidden, hp.vocab
    n = lambda *s, sd=1.0: rng.normal(0.0, sd, size=s)  # noqa: E731
    glob = dict(E1=n(V, d), W_lm=n(V, d, sd=0.3), g_final=1.0 + n(d, sd=0.1))
    glob["E2"] = glob["E1"].copy() if tie_emb else n(V, d)
    layers = []
    cap = max(ctx) + 4
    caches = []
    for _ in range(n_layers):
        P = dict(g_attn=1.0 + n(d, sd=0.1), g_mlp=1.0 + n(d, sd=0.1),
                 Wqkv=n((Hq + 2 * Hkv) * D, d, sd=0.3), Wo=n(d, Hq * D, sd=0.3),
                 a=n(Hq * D, sd=0.5) if couple else np.zeros(Hq * D),
                 b=n(F, sd=0.5) if couple else np.zeros(F),
                 c=n(d, sd=0.5) if couple else np.zeros(d))
        if hp.n_experts == 0:
            P.update(Wgu=n(2 * F, d, sd=0.3), Wd=n(d, F, sd=0.3))
        else:
            E = hp.n_experts
            P.update(Wr=n(E, d), We_gu=n(E, 2 * F, d, sd=0.3), We_d=n(E, d, F, sd=0.3))
        layers.append(P)
        caches.append(O.DenseCache(K=n(batch, Hkv, cap, D), V=n(batch, Hkv, cap, D)))
    tokens = rng.integers(0, V, size=batch)
    seq_len = np.array(ctx[:batch], dtype=np.int64)
    return glob, layers, caches, tokens, seq_len


def close(a, b, tol=1e-12, what=""):
    a, b = np.asarray(a, F64), np.asarray(b, F64)
    err = np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)
    assert err <= tol, f"{what}: relative error {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------------------------------------
# storage rounding
# ---------------------------------------------------------------------------------------------

def pin_round_bf16(O):
    import dfsynth
    rng = np.random.default_rng(1)
    x32 = (rng.normal(size=20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    want = dfsynth.bf16_bits_to_f32(dfsynth.f32_to_bf16_bits(x32)).astype(F64)
    assert np.array_equal(O.round_bf16(x32.astype(F64)), want), "round_bf16 != integer RNE on fp32 inputs"
    # ties go to the even significand: 1 + 2^-8 -> 1 ; 1 + 3*2^-8 -> 1 + 2^-6
    assert O.round_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert O.round_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert O.round_bf16(np.array([-(1 + 3 * 2.0 ** -8)]))[0] == -(1 + 2.0 ** -6)


# ---------------------------------------------------------------------------------------------
# building blocks vs library routines and closed forms
# ---------------------------------------------------------------------------------------------

def pin_rmsnorm(O):
    rng = np.random.default_rng(2)
    h, g = rng.normal(size=(5, 64)) * 3.0, 1.0 + 0.1 * rng.normal(size=64)
    lib = TF.rms_norm(torch.from_numpy(h), (64,), weight=torch.from_numpy(g), eps=1e-6).numpy()
    close(O.rmsnorm(h, g, 1e-6), lib, 1e-13, "rmsnorm vs torch rms_norm")
    # unit gain: output RMS = sqrt(ms / (ms + eps)) exactly
    eps = 0.25
    out = O.rmsnorm(h, np.ones(64), eps)
    ms = np.mean(h * h, axis=-1)
    close(np.sqrt(np.mean(out * out, axis=-1)), np.sqrt(ms / (ms + eps)), 1e-13, "rmsnorm unit-gain RMS")


def pin_rope(O):
    rng = np.random.default_rng(3)
    D, base = 16, 10000.0
    x = rng.normal(size=(3, D))
    # complex formulation: z_i = x_i + i x_{i+D/2}, rotated by pos * base^(-2i/D)
    for pos in (0, 1, 7, 4096):
        z = x[:, : D // 2] + 1j * x[:, D // 2:]
        z = z * np.exp(1j * pos * base ** (-2.0 * np.arange(D // 2) / D))
        close(O.rope(x, pos, base), np.concatenate([z.real, z.imag], axis=-1), 1e-13, f"rope pos {pos}")
    assert np.array_equal(O.rope(x, 0, base), x), "rope at position 0 is not the identity"
    # relative-position property: <R_m q, R_n k> = <R_{m-n} q, k>
    q, k = rng.normal(size=D), rng.normal(size=D)
    for m, n in ((5, 2), (100, 37), (9, 9)):
        close(O.rope(q, m, base) @ O.rope(k, n, base), O.rope(q, m - n, base) @ k, 1e-12, "rope relative")
    # hand case D=4, pos=1: theta = (1, 1/100); e_0 -> (cos 1, 0, sin 1, 0)
    out = O.rope(np.array([1.0, 0, 0, 0]), 1, base)
    close(out, [math.cos(1.0), 0.0, math.sin(1.0), 0.0], 1e-15, "rope hand case")


def pin_attention_closed_forms(O):
    rng = np.random.default_rng(4)
    D = 8
    q = rng.normal(size=(2, D))
    K, V = rng.normal(size=(1, D)), rng.normal(size=(1, D))
    close(O.attention(q, K, V), np.repeat(V, 2, axis=0), 1e-15, "L=1 gives v")
    K = np.repeat(rng.normal(size=(1, D)), 6, axis=0)
    V = rng.normal(size=(6, D))
    close(O.attention(q, K, V), np.repeat(V.mean(0, keepdims=True), 2, axis=0), 1e-14, "equal keys give mean v")
    K = np.zeros((5, D)); K[3, 0] = 1.0
    qq = np.zeros((1, D)); qq[0, 0] = 2000.0
    V = rng.normal(size=(5, D))
    close(O.attention(qq, K, V), V[3:4], 1e-12, "dominant score selects its value")
    # shift invariance: adding a constant to every score leaves the output unchanged
    K, V = rng.normal(size=(7, D)), rng.normal(size=(7, D))
    Kx = np.concatenate([K, np.ones((7, 1))], axis=1)
    qx = np.concatenate([q, 5.0 * np.ones((2, 1))], axis=1)
    close(O.attention(qx, Kx, np.concatenate([V, V[:, :1]], axis=1))[:, :D] * 1.0,
          O.attention(q * math.sqrt(D / (D + 1)), K, V), 1e-12, "score shift invariance")


def pin_attention_gqa_vs_sdpa(O):
    """Attention-only call with a = 0 and aux off reduces to torch's SDPA (GQA) on RoPE'd queries."""
    rng = np.random.default_rng(5)
    hp = tiny_hp(O, n_q_heads=8, n_kv_heads=2, head_dim=16, d_model=32)
    B, cap = 3, 40
    L = np.array([1, 17, 33])
    q1 = rng.normal(size=(B, 8, 16))
    h2 = rng.normal(size=(B, 32))
    Wq = rng.normal(size=(128, 32)) * 0.2
    a = rng.normal(size=128) * 0.3
    K, V = rng.normal(size=(B, 2, cap, 16)), rng.normal(size=(B, 2, cap, 16))
    cache = O.DenseCache(K=K, V=V)
    got = O.attention_only_step(hp, q1, h2, Wq, a, cache, L, aux_on=True, mirror=False)
    for b in range(B):
        for f, qraw in enumerate((q1[b].reshape(-1), Wq @ h2[b] + a * q1[b].reshape(-1))):
            qr = O.rope(qraw.reshape(8, 16), int(L[b]), hp.rope_base)
            z = qraw.reshape(8, 16)
            zc = (z[:, :8] + 1j * z[:, 8:]) * np.exp(1j * L[b] * 10000.0 ** (-2.0 * np.arange(8) / 16))
            close(qr, np.concatenate([zc.real, zc.imag], -1), 1e-12, "query rope")
            ref = TF.scaled_dot_product_attention(
                torch.from_numpy(qr)[None, :, None, :], torch.from_numpy(K[b, :, : L[b]])[None],
                torch.from_numpy(V[b, :, : L[b]])[None], enable_gqa=True)[0, :, 0].numpy()
            close(got[f, b], ref, 1e-12, f"attention-only vs SDPA, flow {f + 1}, row {b}")


def pin_small_ops(O):
    z = np.linspace(-30, 30, 301)
    close(O.silu(z), TF.silu(torch.from_numpy(z)).numpy(), 1e-14, "silu")
    close(O.softmax(z[:7]), scipy.special.softmax(z[:7]), 1e-14, "softmax")
    r = np.array([0.5, 2.0, -1.0, 2.0, 0.5, 3.0])
    assert list(O.topk_lower_index(r, 4)) == [5, 1, 3, 0], "top-k order / tie rule (lower index first)"


# ---------------------------------------------------------------------------------------------
# the step: the primary flow is a standard decoder; the method's invariants; coupling
# ---------------------------------------------------------------------------------------------

def _torch_rope(x, pos, base):
    D = x.shape[-1]
    th = base ** (-2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
    z = torch.complex(x[..., : D // 2], x[..., D // 2:]) * torch.polar(torch.ones_like(th), pos * th)
    return torch.cat([z.real, z.imag], dim=-1)


def torch_llama_decode(hp, glob, layers, caches, tokens, seq_len, E="E1", Wq_scale=None, Wd_pre=None,
                       Wd_post=None):
    """A textbook LLaMA-style pre-norm decode step built from torch library calls (fp64).

    Optional per-layer modifications express special cases of the coupled auxiliary flow as a plain
    decoder: Wq_scale (rows of Wq scaled), Wd_pre (columns of Wd scaled), Wd_post (rows scaled).
    """
    t = lambda a: torch.from_numpy(np.asarray(a, F64))  # noqa: E731
    Hq, Hkv, D, F = hp.n_q_heads, hp.n_kv_heads, hp.head_dim, hp.ffn_hidden
    out = []
    for b in range(len(tokens)):
        h = t(glob[E][tokens[b]])
        L = int(seq_len[b])
        for li, P in enumerate(layers):
            x = TF.rms_norm(h, (hp.d_model,), weight=t(P["g_attn"]), eps=hp.rms_eps)
            W = t(P["Wqkv"])
            Wq, Wk, Wv = W[: Hq * D], W[Hq * D: (Hq + Hkv) * D], W[(Hq + Hkv) * D:]
            if Wq_scale is not None:
                Wq = Wq * t(Wq_scale)[:, None]
            q = _torch_rope(TF.linear(x, Wq).view(Hq, D), L, hp.rope_base)
            k = _torch_rope(TF.linear(x, Wk).view(Hkv, D), L, hp.rope_base)
            v = TF.linear(x, Wv).view(Hkv, D)
            Kc, Vc = caches[li].seq(b, L)
            Kc = torch.cat([t(Kc), k[:, None]], 1)
            Vc = torch.cat([t(Vc), v[:, None]], 1)
            o = TF.scaled_dot_product_attention(q[None, :, None], Kc[None], Vc[None], enable_gqa=True)[0, :, 0]
            h = h + TF.linear(o.reshape(-1), t(P["Wo"]))
            x = TF.rms_norm(h, (hp.d_model,), weight=t(P["g_mlp"]), eps=hp.rms_eps)
            Wg, Wu = t(P["Wgu"][:F]), t(P["Wgu"][F:])
            Wd = t(P["Wd"])
            if Wd_pre is not None:
                Wd = Wd * t(Wd_pre)[None, :]
            if Wd_post is not None:
                Wd = Wd * t(Wd_post)[:, None]
            h = h + TF.linear(TF.silu(TF.linear(x, Wg)) * TF.linear(x, Wu), Wd)
        x = TF.rms_norm(h, (hp.d_model,), weight=t(glob["g_final"]), eps=hp.rms_eps)
        out.append(TF.linear(x, t(glob["W_lm"])).numpy())
    return np.stack(out)


def pin_primary_is_standard_decoder(O):
    hp = tiny_hp(O)
    glob, layers, caches, tokens, L = tiny_model(O, hp, n_layers=2)
    got = O.decode_step(hp, glob, layers, caches, tokens, L, aux_on=True, mirror=False)
    close(got["logits"][0], torch_llama_decode(hp, glob, layers, caches, tokens, L), 1e-11,
          "primary flow vs torch LLaMA decode")
    # the appended entry is the RoPE'd primary key and the raw value of the new token
    P = layers[0]
    x = O.rmsnorm(glob["E1"][tokens[0]], P["g_attn"], hp.rms_eps)
    kd = hp.n_kv_heads * hp.head_dim
    qd = hp.n_q_heads * hp.head_dim
    k = _torch_rope(torch.from_numpy(P["Wqkv"][qd: qd + kd] @ x).view(hp.n_kv_heads, -1), int(L[0]),
                    hp.rope_base).numpy()
    close(got["k_new"][0, 0], k, 1e-12, "appended key")
    close(got["v_new"][0, 0], (P["Wqkv"][qd + kd:] @ x).reshape(hp.n_kv_heads, -1), 1e-12, "appended value")


def pin_flow_invariants(O):
    hp = tiny_hp(O)
    glob, layers, caches, tokens, L = tiny_model(O, hp, n_layers=2, seed=7)
    for mirror in (False, True):
        hpm = tiny_hp(O, dtype="bf16") if mirror else hp
        on = O.decode_step(hpm, glob, layers, caches, tokens, L, aux_on=True, mirror=mirror)
        off = O.decode_step(hpm, glob, layers, caches, tokens, L, aux_on=False, mirror=mirror)
        # (i) the primary flow never depends on the auxiliary flow
        assert np.array_equal(on["logits"][0], off["logits"][0]), "primary logits change with aux_on"
        # (ii) the auxiliary flow writes nothing into the cache
        assert np.array_equal(on["k_new"], off["k_new"]) and np.array_equal(on["v_new"], off["v_new"])
        assert np.all(np.isnan(off["logits"][1])) and np.all(np.isfinite(on["logits"][1]))
    # (iii) a = b = c = 0 and E2 = E1: the flows coincide exactly
    glob0, layers0, caches0, tokens0, L0 = tiny_model(O, hp, n_layers=2, seed=8, couple=False, tie_emb=True)
    r = O.decode_step(hp, glob0, layers0, caches0, tokens0, L0, aux_on=True, mirror=False)
    assert np.array_equal(r["logits"][0], r["logits"][1]), "uncoupled tied flows differ"
    # (iv) perturbing E2, a, b or c leaves the primary bitwise unchanged, and changes the auxiliary
    base = O.decode_step(hp, glob, layers, caches, tokens, L, aux_on=True, mirror=False)
    for key in ("E2", "a", "b", "c"):
        g2 = dict(glob)
        l2 = [dict(P) for P in layers]
        if key == "E2":
            g2["E2"] = glob["E2"] + 0.5
        else:
            l2[0][key] = layers[0][key] + 0.5
        r = O.decode_step(hp, g2, l2, caches, tokens, L, aux_on=True, mirror=False)
        assert np.array_equal(r["logits"][0], base["logits"][0]), f"primary depends on {key}"
        assert np.max(np.abs(r["logits"][1] - base["logits"][1])) > 1e-6, f"auxiliary ignores {key}"


def pin_coupling_special_cases(O):
    """With E2 = E1 in a one-layer model the auxiliary flow is a plain decoder with modified weights:
    a -> Wq rows scaled by (1 + a) (coupling before RoPE); b -> Wd columns scaled by (1 + b);
    c -> Wd rows scaled by (1 + c)."""
    hp = tiny_hp(O)
    glob, layers, caches, tokens, L = tiny_model(O, hp, n_layers=1, seed=9, couple=False, tie_emb=True)
    rng = np.random.default_rng(10)
    for key in ("a", "b", "c"):
        l2 = [dict(layers[0])]
        vec = rng.normal(size=l2[0][key].shape) * 0.5
        l2[0][key] = vec
        got = O.decode_step(hp, glob, l2, caches, tokens, L, aux_on=True, mirror=False)["logits"][1]
        kw = {"a": dict(Wq_scale=1 + vec), "b": dict(Wd_pre=1 + vec), "c": dict(Wd_post=1 + vec)}[key]
        close(got, torch_llama_decode(hp, glob, l2, caches, tokens, L, **kw), 1e-11, f"coupling {key}")


def pin_query_coupling_source(O):
    """E2 = 0 makes the auxiliary input zero, so its first-layer query is exactly a (*) q1: its
    attention output must equal SDPA of RoPE(a (*) q1) over the cache plus the appended entry."""
    hp = tiny_hp(O)
    glob, layers, caches, tokens, L = tiny_model(O, hp, n_layers=1, seed=17)
    glob = dict(glob, E2=np.zeros_like(glob["E2"]))
    tr = []
    r = O.decode_step(hp, glob, layers, caches, tokens, L, aux_on=True, mirror=False, trace=tr)
    P = layers[0]
    Hq, Hkv, D = hp.n_q_heads, hp.n_kv_heads, hp.head_dim
    for e in tr:
        b = e["b"]
        x1 = O.rmsnorm(glob["E1"][tokens[b]], P["g_attn"], hp.rms_eps)
        q2 = (P["a"] * (P["Wqkv"][: Hq * D] @ x1)).reshape(Hq, D)
        q2 = _torch_rope(torch.from_numpy(q2), int(L[b]), hp.rope_base)
        Kc, Vc = caches[0].seq(b, int(L[b]))
        Kc = np.concatenate([Kc, r["k_new"][0, b][:, None]], 1)
        Vc = np.concatenate([Vc, r["v_new"][0, b][:, None]], 1)
        ref = TF.scaled_dot_product_attention(q2[None, :, None], torch.from_numpy(Kc)[None],
                                              torch.from_numpy(Vc)[None], enable_gqa=True)[0, :, 0].numpy()
        close(e["o"][1].reshape(Hq, D), ref, 1e-12, "auxiliary query = a (*) q1 when its input is zero")


def pin_paged_equals_dense(O):
    """A shuffled paged layout read through its page table gives exactly the dense-cache result."""
    rng = np.random.default_rng(18)
    hp = tiny_hp(O, n_q_heads=4, n_kv_heads=2, head_dim=8, d_model=16)
    B, ps, cap = 3, 4, 24
    L = np.array([24, 5, 13])
    K, V = rng.normal(size=(B, 2, cap, 8)), rng.normal(size=(B, 2, cap, 8))
    npg = (L + ps - 1) // ps
    perm = rng.permutation(int(npg.sum()))
    table = np.full((B, cap // ps), -1)
    pk = np.zeros((int(npg.sum()), 2, ps, 8))
    pv = np.zeros_like(pk)
    off = 0
    for b in range(B):
        for j in range(npg[b]):
            pid = perm[off + j]
            table[b, j] = pid
            pk[pid] = K[b, :, j * ps:(j + 1) * ps]
            pv[pid] = V[b, :, j * ps:(j + 1) * ps]
        off += npg[b]
    q1, h2 = rng.normal(size=(B, 4, 8)), rng.normal(size=(B, 16))
    Wq, a = rng.normal(size=(32, 16)), rng.normal(size=32)
    dense = O.attention_only_step(hp, q1, h2, Wq, a, O.DenseCache(K, V), L, mirror=False)
    paged = O.attention_only_step(hp, q1, h2, Wq, a, O.PagedCache(pk, pv, table, ps), L, mirror=False)
    assert np.array_equal(dense, paged), "paged cache != dense cache"


def pin_empty_cache(O):
    """L_b = 0: the only attended entry is the one appended in this step, so o = v_new for both flows."""
    hp = tiny_hp(O, n_q_heads=2, n_kv_heads=2)
    glob, layers, caches, tokens, _ = tiny_model(O, hp, n_layers=1, seed=11)
    tr = []
    r = O.decode_step(hp, glob, layers, caches, tokens, np.array([0, 0]), aux_on=True, mirror=False, trace=tr)
    for e in tr:
        v = r["v_new"][0, e["b"]]
        for f in range(2):
            close(e["o"][f].reshape(2, -1), v, 1e-13, "empty cache attends only the new entry")


def pin_moe_special_cases(O):
    # E = 1, k = 1: the MoE layer is the dense SwiGLU layer with that expert's weights
    hpm = tiny_hp(O, n_experts=1, topk_primary=1, topk_aux=1)
    glob, layers, caches, tokens, L = tiny_model(O, hpm, n_layers=1, seed=12)
    dense = [dict(P, Wgu=P["We_gu"][0], Wd=P["We_d"][0]) for P in layers]
    got = O.decode_step(hpm, glob, layers, caches, tokens, L, mirror=False)["logits"]
    want = O.decode_step(tiny_hp(O), glob, dense, caches, tokens, L, mirror=False)["logits"]
    close(got, want, 1e-13, "MoE E=1,k=1 vs dense")
    # k = E: every expert, weighted by the full softmax of the router logits
    hpE = tiny_hp(O, n_experts=3, topk_primary=3, topk_aux=3)
    rng = np.random.default_rng(13)
    r1, r2 = rng.normal(size=3), rng.normal(size=3)
    S1, w1, S2, w2 = O.route(hpE, r1, r2, True)
    close(w1[np.argsort(S1)], scipy.special.softmax(r1), 1e-14, "k=E primary weights")
    close(w2[np.argsort(S2)], scipy.special.softmax(r2), 1e-14, "k=E auxiliary weights")
    # replay: the auxiliary set is chosen by the primary logits and contains the primary set
    hpr = tiny_hp(O, n_experts=6, topk_primary=2, topk_aux=4)
    r1 = np.array([0.1, 0.9, -0.3, 0.4, 0.8, 0.0])
    r2 = np.array([5.0, -5.0, 4.0, 0.0, 0.0, 3.0])
    S1, w1, S2, w2 = O.route(hpr, r1, r2, True)
    assert list(S1) == [1, 4] and list(S2) == [1, 4, 3, 0], "replay sets"
    close(w2, scipy.special.softmax(r2[[1, 4, 3, 0]]), 1e-14, "auxiliary weights from its own logits")
    # E2 = E1 and no coupling with k_aux = k_primary: both flows coincide
    hps = tiny_hp(O, n_experts=4, topk_primary=2, topk_aux=2)
    glob, layers, caches, tokens, L = tiny_model(O, hps, n_layers=2, seed=14, couple=False, tie_emb=True)
    r = O.decode_step(hps, glob, layers, caches, tokens, L, mirror=False)
    assert np.array_equal(r["logits"][0], r["logits"][1]) and np.array_equal(r["expert_ids"][:, 0],
                                                                              r["expert_ids"][:, 1])
    # a brute-force MoE layer on one token: sum over selected experts of w_e * Wd_e (silu(Wg_e x) * Wu_e x)
    hpb = tiny_hp(O, n_experts=5, topk_primary=2, topk_aux=3)
    glob, layers, caches, tokens, L = tiny_model(O, hpb, n_layers=1, batch=1, seed=15)
    tr = []
    res = O.decode_step(hpb, glob, layers, caches, tokens, L, mirror=False, trace=tr)
    P, F = layers[0], hpb.ffn_hidden
    h_mid = None
    # recompute the mid-layer residual from the attention output recorded in the trace
    h0 = [glob["E1"][tokens[0]], glob["E2"][tokens[0]]]
    h_mid = [h0[f] + P["Wo"] @ tr[0]["o"][f] for f in range(2)]
    x = [O.rmsnorm(h_mid[f], P["g_mlp"], hpb.rms_eps) for f in range(2)]
    r1, r2 = P["Wr"] @ x[0], P["Wr"] @ x[1]
    y = []
    for f, (rf, k) in enumerate(((r1, 2), (r2, 3))):
        sel = [i for i in np.argsort(-r1, kind="stable")[:k]]
        wts = [math.exp(rf[e]) for e in sel]
        wts = [wv / sum(wts) for wv in wts]
        acc = np.zeros(hpb.d_model)
        for e, wv in zip(sel, wts):
            u = [0.0] * F
            for j in range(F):
                gj = sum(P["We_gu"][e][j, m] * x[f][m] for m in range(hpb.d_model))
                uj = sum(P["We_gu"][e][F + j, m] * x[f][m] for m in range(hpb.d_model))
                u[j] = gj / (1 + math.exp(-gj)) * uj
                if f == 1 and e in np.argsort(-r1, kind="stable")[:2]:
                    g1 = sum(P["We_gu"][e][j, m] * x[0][m] for m in range(hpb.d_model))
                    u1 = sum(P["We_gu"][e][F + j, m] * x[0][m] for m in range(hpb.d_model))
                    u[j] += P["b"][j] * g1 / (1 + math.exp(-g1)) * u1
            acc += wv * (P["We_d"][e] @ np.array(u))
        y.append(acc)
    y[1] = y[1] + P["c"] * y[0]
    close(res["h"][0, 0], h_mid[0] + y[0], 1e-12, "brute MoE primary")
    close(res["h"][1, 0], h_mid[1] + y[1], 1e-12, "brute MoE auxiliary")


def pin_mirror_tracks_exact(O):
    """Mirror mode only rounds at the bf16 storage points: on a small bf16 model it stays within
    bf16 rounding of the exact fp64 step. Residual rows of scale ~8 and gains of spread 0.4 make a
    dropped 1/rms or a dropped gain in the mirrored norm show far above that rounding."""
    hp = tiny_hp(O, dtype="bf16")
    glob, layers, caches, tokens, L = tiny_model(O, hp, n_layers=2, seed=21)
    glob = dict(glob, E1=glob["E1"] * 8.0, E2=glob["E2"] * 8.0, g_final=1.0 + 4.0 * (glob["g_final"] - 1.0))
    layers = [dict(P, g_attn=1.0 + 4.0 * (P["g_attn"] - 1.0), g_mlp=1.0 + 4.0 * (P["g_mlp"] - 1.0)) for P in layers]
    exact = O.decode_step(hp, glob, layers, caches, tokens, L, aux_on=True, mirror=False)
    mirr = O.decode_step(hp, glob, layers, caches, tokens, L, aux_on=True, mirror=True)
    close(mirr["logits"], exact["logits"], 3e-2, "mirrored bf16 step vs exact fp64 step")
    assert not np.array_equal(mirr["logits"], exact["logits"]), "mirror mode rounds nothing"


def pin_mixture_head(O):
    V = 10
    a, pm, tok = O.mixture_head(np.zeros(V), np.arange(V, dtype=F64))
    close(a, 0.5 + 0.5 / V, 1e-15, "uniform primary: alpha = 1/2 + 1/(2V)")
    close(pm.sum(), 1.0, 1e-15, "p_mix sums to one")
    big = np.zeros(V); big[3] = 800.0
    a, pm, tok = O.mixture_head(big, np.arange(V, dtype=F64))
    close(a, 1.0, 1e-15, "confident primary: alpha = 1")
    assert tok == 3
    rng = np.random.default_rng(16)
    for _ in range(20):
        a, _, _ = O.mixture_head(rng.normal(size=V) * 3, rng.normal(size=V))
        assert 0.5 <= a <= 1.0


def pin_sampling(O):
    """Inverse-transform sampling: hand-worked cases, closed forms, and the empirical frequencies
    of a stratified grid of uniforms reproduce the distribution."""
    p = np.array([0.1, 0.0, 0.3, 0.6])
    for u, want in [(0.0, 0), (0.05, 0), (0.1, 2), (0.39, 2), (0.4, 3), (0.9999, 3)]:
        assert O.sample_inverse_cdf(p, u) == want, (u, want)
    assert O.sample_inverse_cdf(np.array([0.5, 0.5, 0.0]), 1.0) == 1  # no partial sum exceeds u
    V = 37
    for u in (0.013, 0.5 + 1e-9, 0.977):
        assert O.sample_inverse_cdf(np.full(V, 1.0 / V), u) == int(np.floor(u * V))
    one = np.zeros(V); one[11] = 1.0
    assert all(O.sample_inverse_cdf(one, u) == 11 for u in (0.0, 0.3, 0.999))
    rng = np.random.default_rng(17)
    q = rng.dirichlet(np.ones(12))
    N = 20000
    counts = np.bincount([O.sample_inverse_cdf(q, (k + 0.5) / N) for k in range(N)], minlength=12)
    assert np.all(np.abs(counts - N * q) <= 1.0 + 1e-9), (counts, N * q)


def _torch_decode_one(hp, glob, layers, tok, L, Kl, Vl, Wq_scale=None):
    """One sequence's decode step with a textbook decoder from torch calls (fp64) over explicit
    cache tensors Kl[l], Vl[l] ([Hkv, L, D]); returns the logits and each layer's new (k, v)."""
    t = lambda a: torch.from_numpy(np.asarray(a, F64))  # noqa: E731
    Hq, Hkv, D, F = hp.n_q_heads, hp.n_kv_heads, hp.head_dim, hp.ffn_hidden
    h = t(glob["E1"][tok])
    new = []
    for li, P in enumerate(layers):
        x = TF.rms_norm(h, (hp.d_model,), weight=t(P["g_attn"]), eps=hp.rms_eps)
        W = t(P["Wqkv"])
        Wq, Wk, Wv = W[: Hq * D], W[Hq * D: (Hq + Hkv) * D], W[(Hq + Hkv) * D:]
        if Wq_scale is not None:
            Wq = Wq * t(Wq_scale)[:, None]
        q = _torch_rope(TF.linear(x, Wq).view(Hq, D), L, hp.rope_base)
        k = _torch_rope(TF.linear(x, Wk).view(Hkv, D), L, hp.rope_base)
        v = TF.linear(x, Wv).view(Hkv, D)
        Kc = torch.cat([Kl[li], k[:, None]], 1)
        Vc = torch.cat([Vl[li], v[:, None]], 1)
        o = TF.scaled_dot_product_attention(q[None, :, None], Kc[None], Vc[None], enable_gqa=True)[0, :, 0]
        h = h + TF.linear(o.reshape(-1), t(P["Wo"]))
        x = TF.rms_norm(h, (hp.d_model,), weight=t(P["g_mlp"]), eps=hp.rms_eps)
        h = h + TF.linear(TF.silu(TF.linear(x, t(P["Wgu"][:F]))) * TF.linear(x, t(P["Wgu"][F:])), t(P["Wd"]))
        new.append((k, v))
    x = TF.rms_norm(h, (hp.d_model,), weight=t(glob["g_final"]), eps=hp.rms_eps)
    return TF.linear(x, t(glob["W_lm"])), new


def torch_generate(hp, glob, layers, caches, tokens, seq_len, n_steps, u=None, aux_Wq_scale=None):
    """Generation with torch calls and torch-side KV lists: the primary decoder's distribution, or
    (aux_Wq_scale given) its mixture with a second decoder whose query rows are scaled, attending
    the primary's cache; next token by torch.argmax or by torch.searchsorted of the cumulative sum."""
    B, nL = len(tokens), len(layers)
    Kl = [[torch.from_numpy(np.asarray(caches[li].seq(b, int(seq_len[b]))[0], F64)) for li in range(nL)] for b in range(B)]
    Vl = [[torch.from_numpy(np.asarray(caches[li].seq(b, int(seq_len[b]))[1], F64)) for li in range(nL)] for b in range(B)]
    toks = [int(x) for x in tokens]
    out = np.zeros((n_steps, B), dtype=np.int64)
    for st in range(n_steps):
        for b in range(B):
            L = int(seq_len[b]) + st
            l1, new = _torch_decode_one(hp, glob, layers, toks[b], L, Kl[b], Vl[b])
            p = torch.softmax(l1, 0)
            if aux_Wq_scale is not None:
                l2, _ = _torch_decode_one(hp, glob, layers, toks[b], L, Kl[b], Vl[b], Wq_scale=aux_Wq_scale)
                alpha = 0.5 + 0.5 * torch.dot(p, p)
                p = alpha * p + (1 - alpha) * torch.softmax(l2, 0)
            if u is None:
                out[st, b] = int(torch.argmax(p))
            else:
                out[st, b] = int(torch.searchsorted(torch.cumsum(p, 0), torch.tensor([float(u[st, b])], dtype=torch.float64),
                                                    right=True)[0])
            for li, (k, v) in enumerate(new):
                Kl[b][li] = torch.cat([Kl[b][li], k[:, None]], 1)
                Vl[b][li] = torch.cat([Vl[b][li], v[:, None]], 1)
        toks = [int(x) for x in out[st]]
    return out


def torch_prefill(hp, glob, layers, caches, prompt, seq_len):
    """A causal prefill with torch calls: all of a sequence's prompt positions in one pass per layer,
    scaled_dot_product_attention with a boolean mask (position L + i sees cached positions and
    prompt positions up to itself); returns the logits of every position [B, n, V]."""
    t = lambda a: torch.from_numpy(np.asarray(a, F64))  # noqa: E731
    Hq, Hkv, D, F = hp.n_q_heads, hp.n_kv_heads, hp.head_dim, hp.ffn_hidden
    B, n = prompt.shape
    out = []
    for b in range(B):
        L = int(seq_len[b])
        h = t(glob["E1"][prompt[b]])  # [n, d]
        pos = torch.arange(L, L + n, dtype=torch.float64)
        mask = torch.arange(L + n)[None, :] <= torch.arange(L, L + n)[:, None]  # [n, L + n]
        for li, P in enumerate(layers):
            x = TF.rms_norm(h, (hp.d_model,), weight=t(P["g_attn"]), eps=hp.rms_eps)
            W = t(P["Wqkv"])
            q = TF.linear(x, W[: Hq * D]).view(n, Hq, D)
            k = TF.linear(x, W[Hq * D: (Hq + Hkv) * D]).view(n, Hkv, D)
            v = TF.linear(x, W[(Hq + Hkv) * D:]).view(n, Hkv, D)
            th = hp.rope_base ** (-2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
            ang = pos[:, None, None] * th  # [n, 1, D/2]
            rot = lambda z: torch.cat([z[..., : D // 2] * torch.cos(ang) - z[..., D // 2:] * torch.sin(ang),  # noqa: E731
                                       z[..., : D // 2] * torch.sin(ang) + z[..., D // 2:] * torch.cos(ang)], -1)
            q, k = rot(q), rot(k)
            Kc, Vc = caches[li].seq(b, L)
            Kall = torch.cat([t(Kc), k.transpose(0, 1)], 1)  # [Hkv, L + n, D]
            Vall = torch.cat([t(Vc), v.transpose(0, 1)], 1)
            o = TF.scaled_dot_product_attention(q.transpose(0, 1)[None], Kall[None], Vall[None], attn_mask=mask,
                                                enable_gqa=True)[0]  # [Hq, n, D]
            h = h + TF.linear(o.transpose(0, 1).reshape(n, -1), t(P["Wo"]))
            x = TF.rms_norm(h, (hp.d_model,), weight=t(P["g_mlp"]), eps=hp.rms_eps)
            h = h + TF.linear(TF.silu(TF.linear(x, t(P["Wgu"][:F]))) * TF.linear(x, t(P["Wgu"][F:])), t(P["Wd"]))
        x = TF.rms_norm(h, (hp.d_model,), weight=t(glob["g_final"]), eps=hp.rms_eps)
        out.append(TF.linear(x, t(glob["W_lm"])).numpy())
    return np.stack(out)


def pin_prefill(O):
    """Prefill (one primary-only decode step per prompt position) equals a torch causal pass over the
    whole prompt at every position, with and without a cached prefix; decoding after it equals
    decoding after the same tokens fed one by one."""
    hp = tiny_hp(O)
    glob, layers, caches, _, L = tiny_model(O, hp, n_layers=2, seed=31)
    prompt = np.random.default_rng(32).integers(0, hp.vocab, size=(2, 4))
    for start in (np.zeros(2, dtype=np.int64), L):
        ref = torch_prefill(hp, glob, layers, caches, prompt, start)
        got = O.prefill(hp, glob, layers, _writable_caches(O, caches), prompt, start, mirror=False)
        close(got["logits"], ref, 1e-11, "prefill logits at every position")
        assert np.array_equal(got["seq_len"], start + prompt.shape[1])


def pin_prefill_moe(O):
    """Prefill of a MoE model with one expert and top-1 routing equals the torch causal pass of the
    dense model whose MLP is that expert (the routing weight of a single chosen expert is 1), at
    every position; its router logits are reported for every position and layer."""
    hp = tiny_hp(O, n_experts=1, topk_primary=1, topk_aux=1)
    glob, layers, caches, _, L = tiny_model(O, hp, n_layers=2, seed=33)
    dense = [dict({k: v for k, v in P.items() if k not in ("Wr", "We_gu", "We_d")}, Wgu=P["We_gu"][0], Wd=P["We_d"][0])
             for P in layers]
    prompt = np.random.default_rng(34).integers(0, hp.vocab, size=(2, 3))
    ref = torch_prefill(tiny_hp(O), glob, dense, caches, prompt, L)
    got = O.prefill(hp, glob, layers, _writable_caches(O, caches), prompt, L, mirror=False)
    close(got["logits"], ref, 1e-11, "one-expert MoE prefill logits")
    assert got["rlog"].shape == (2, 2, 3, 1) and np.all(np.isfinite(got["rlog"]))


def _writable_caches(O, caches):
    return [O.DenseCache(K=np.array(c.K, copy=True), V=np.array(c.V, copy=True)) for c in caches]


def pin_generate(O):
    """The decode loop against torch-built generators: greedy and sampled generation of tied,
    uncoupled flows (the mixture is the primary's distribution); the mixture of a one-layer model
    whose auxiliary flow differs only by query coupling a (a second decoder with scaled query rows
    sharing the primary's cache); and primary-only generation with coupling on."""
    hp = tiny_hp(O, vocab=11)
    n = 4
    glob, layers, caches, tokens, L = tiny_model(O, hp, n_layers=2, seed=21, couple=False, tie_emb=True)
    ref = torch_generate(hp, glob, layers, caches, tokens, L, n)
    got = O.generate(hp, glob, layers, _writable_caches(O, caches), tokens, L, n, mirror=False)
    assert np.array_equal(got["tokens"], ref), (got["tokens"], ref)
    assert np.array_equal(got["seq_len"], L + n)
    u = np.random.default_rng(22).uniform(size=(n, len(tokens)))
    ref = torch_generate(hp, glob, layers, caches, tokens, L, n, u=u)
    got = O.generate(hp, glob, layers, _writable_caches(O, caches), tokens, L, n, u=u, mirror=False)
    assert np.array_equal(got["tokens"], ref), (got["tokens"], ref)
    # the mixture matters: a one-layer model, E2 = E1, coupling a only
    glob1, layers1, caches1, tokens1, L1 = tiny_model(O, hp, n_layers=1, seed=23, couple=False, tie_emb=True,
                                                      batch=2)
    a = np.random.default_rng(24).normal(size=layers1[0]["a"].shape) * 1.5
    layers1 = [dict(layers1[0], a=a)]
    ref = torch_generate(hp, glob1, layers1, caches1, tokens1, L1, n, aux_Wq_scale=1 + a)
    got = O.generate(hp, glob1, layers1, _writable_caches(O, caches1), tokens1, L1, n, mirror=False)
    assert np.array_equal(got["tokens"], ref), (got["tokens"], ref)
    prim = torch_generate(hp, glob1, layers1, caches1, tokens1, L1, n)
    assert not np.array_equal(prim, ref), "the mixture never changes a choice here: the pin is blind"
    # auxiliary flow off: the primary's own choice, coupling or not
    got = O.generate(hp, glob1, layers1, _writable_caches(O, caches1), tokens1, L1, n, aux_on=False, mirror=False)
    assert np.array_equal(got["tokens"], prim)


def pin_generate_paged(O):
    """Generation through a shuffled paged cache (pages of 4) that holds every position the
    sequences reach, so the entries each step appends land in pages mapped ahead of time, gives the
    tokens of the torch-built generator, which keeps its own dense key/value lists; every slot the
    loop appends to holds a finite entry afterwards and every other unused slot is still unwritten."""
    hp = tiny_hp(O, vocab=11)
    n, ps = 5, 4
    glob, layers, caches, tokens, L = tiny_model(O, hp, n_layers=2, seed=25, couple=False, tie_emb=True)
    ref = torch_generate(hp, glob, layers, caches, tokens, L, n)
    B, Hkv, D = len(tokens), hp.n_kv_heads, hp.head_dim
    need = (L + n + ps - 1) // ps  # pages covering positions 0 .. L_b + n - 1
    perm = np.random.default_rng(26).permutation(int(need.sum()))
    table = np.full((B, int(need.max()) + 1), -1)
    off = 0
    for b in range(B):
        table[b, : need[b]] = perm[off: off + need[b]]
        off += int(need[b])
    paged = []
    for c in caches:
        K = np.full((int(need.sum()), Hkv, ps, D), np.nan)
        V = np.full_like(K, np.nan)
        for b in range(B):
            for pos in range(int(L[b])):
                pid = table[b, pos // ps]
                K[pid][:, pos % ps] = c.K[b][:, pos]
                V[pid][:, pos % ps] = c.V[b][:, pos]
        paged.append(O.PagedCache(K, V, table, ps))
    got = O.generate(hp, glob, layers, paged, tokens, L, n, mirror=False)
    assert np.array_equal(got["tokens"], ref), (got["tokens"], ref)
    for c in paged:
        for b in range(B):
            for pos in range(int(need[b]) * ps):
                pid = table[b, pos // ps]
                written = np.all(np.isfinite(c.K[pid][:, pos % ps])) and np.all(np.isfinite(c.V[pid][:, pos % ps]))
                assert written == (pos < L[b] + n), f"sequence {b} position {pos}: written {written}"


ALL_PINS = [pin_round_bf16, pin_rmsnorm, pin_rope, pin_attention_closed_forms, pin_attention_gqa_vs_sdpa,
            pin_small_ops, pin_primary_is_standard_decoder, pin_flow_invariants, pin_coupling_special_cases, pin_query_coupling_source,
            pin_paged_equals_dense, pin_empty_cache, pin_moe_special_cases, pin_mirror_tracks_exact, pin_mixture_head,
            pin_sampling, pin_generate, pin_generate_paged, pin_prefill, pin_prefill_moe]
