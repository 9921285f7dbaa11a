"""Primary-only prefill (dualflow_prefill) on the GPU against the oracle's prefill.

The cache rows the prefill writes (positions seq_len[b] .. seq_len[b] + n - 1 of every layer) are
compared with the oracle's at the bf16 bar, every other cache element must be unchanged bit for
bit, the lengths must advance by n, and a decode step of both flows after the prefill must give
the oracle's logits (which depend on every prefilled entry)."""
import numpy as np
import pytest
import torch

import dual_flow_decode_dualflow_b300 as dfl
import oracle as O
from dfsynth import workloads as W
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
TOL = 2e-2

SMALL = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=1, ffn_hidden=512, vocab=1000, batch=3, ctx_len=0,
             ctx_lo=5, ctx_hi=200, gain_sigma=0.1)
# (workload, prompt tokens per sequence, cached lengths before the prefill or None for the workload's)
CASES = {
    "g4_b3_n9": (W.DENSE_24L_B32_L4096.replace(**SMALL), 9, None),
    "g2_b2_n300_rowblocks": (W.DENSE_24L_B32_L4096.replace(**dict(SMALL, n_kv_heads=2, batch=2, ctx_lo=0, ctx_hi=600)),
                             300, [0, 37]),
    "g1_b2_n70": (W.DENSE_24L_B32_L4096.replace(**dict(SMALL, n_q_heads=2, n_kv_heads=2, batch=2, ctx_lo=0,
                                                       ctx_hi=100)), 70, [3, 20]),
}


def _oracle_caches(w):
    out = []
    for l in range(w.n_layers):
        K = H.host_f64(w, f"L{l}.K").reshape(w.cache_shape()).copy()
        V = H.host_f64(w, f"L{l}.V").reshape(w.cache_shape()).copy()
        out.append(O.DenseCache(K=K, V=V))
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_parity(cuda_device, name):
    w, n, lens = CASES[name]
    run = H.DeviceRun(w, cuda_device)
    try:
        if lens is not None:
            run.seq_len_np = np.array(lens, dtype=np.int32)
            run.seq_len.copy_(torch.from_numpy(run.seq_len_np))
        L = run.seq_len_np.astype(np.int64)
        assert L.max() + n < w.max_ctx
        prompt = np.random.default_rng(41).integers(0, w.vocab, size=(w.batch, n)).astype(np.int32)
        before = {k: v.clone() for k, v in run.t.items() if k.endswith((".K", ".V"))}
        dfl.dualflow_prefill_reserve(run.ctx, w.batch * n)
        dfl.dualflow_prefill(run.ctx, run.weights, run.kv, torch.from_numpy(prompt).to(cuda_device), w.batch, n)
        assert run.status() == 0
        assert np.array_equal(run.seq_len.cpu().numpy(), L + n)

        caches = _oracle_caches(w)
        glob = {"E1": H.LazyRows(w, "E1"), "E2": H.LazyRows(w, "E2"), "W_lm": H.host_f64(w, "W_lm"),
                "g_final": H.host_f64(w, "g_final")}
        layers = H.LazyLayers(w)
        O.prefill(H.hparams(w), glob, layers, caches, prompt, L, mirror=True)
        for l in range(w.n_layers):
            for kind in ("K", "V"):
                t = run.t[f"L{l}.{kind}"]
                ref = caches[l].K if kind == "K" else caches[l].V
                exp = before[f"L{l}.{kind}"].clone()
                for b in range(w.batch):
                    got = H.to_f64(t[b, :, L[b]:L[b] + n, :])
                    err = H.rel_err(got, ref[b][:, L[b]:L[b] + n, :])
                    assert err <= TOL, f"layer {l} {kind} seq {b}: rel err {err:.3e}"
                    exp[b, :, L[b]:L[b] + n, :] = t[b, :, L[b]:L[b] + n, :]
                assert torch.equal(exp, t), f"layer {l} {kind}: cache changed outside the prompt's rows"

        # the next token of every sequence as a decode step of both flows, after the prompt
        nxt = np.random.default_rng(42).integers(0, w.vocab, size=w.batch).astype(np.int32)
        run.tokens.copy_(torch.from_numpy(nxt))
        run.tokens_np = nxt
        run.step(aux_on=1)
        assert run.status() == 0
        ref = O.decode_step(H.hparams(w), glob, layers, caches, nxt, L + n, aux_on=True, mirror=True)
        got = H.to_f64(run.logits)
        for f in range(2):
            err = H.rel_err(got[f], ref["logits"][f])
            assert err <= TOL, f"decode after prefill, flow {f + 1}: rel err {err:.3e}"
    finally:
        run.close()


def test_prefill_rejects_without_room(cuda_device):
    w, n, _ = CASES["g4_b3_n9"]
    run = H.DeviceRun(w, cuda_device)
    try:
        prompt = torch.zeros((w.batch, n), dtype=torch.int32, device=cuda_device)
        with pytest.raises(dfl.DualFlowError):
            dfl.dualflow_prefill(run.ctx, run.weights, run.kv, prompt, w.batch, n)  # nothing reserved
        dfl.dualflow_prefill_reserve(run.ctx, w.batch * n - 1)
        with pytest.raises(dfl.DualFlowError):
            dfl.dualflow_prefill(run.ctx, run.weights, run.kv, prompt, w.batch, n)
        assert np.array_equal(run.seq_len.cpu().numpy(), run.seq_len_np)  # nothing ran
    finally:
        run.close()


def test_prefill_into_released_slot(cuda_device):
    """Continuous batching on a contiguous cache: the sequence of slot 1 ends (length 0) and a new
    prompt is prefilled into that slot alone. The other slots' cache entries and lengths stay bit
    for bit; the new prompt's keys/values, and a decode step of all slots after it, match the
    oracle (the new sequence prefilled from an empty cache, the others as they were)."""
    w, _, _ = CASES["g4_b3_n9"]
    n = 23
    run = H.DeviceRun(w, cuda_device)
    try:
        L = run.seq_len_np.astype(np.int64)
        slot = torch.tensor([1], dtype=torch.int32, device=cuda_device)
        before = {k: v.clone() for k, v in run.t.items() if k.endswith((".K", ".V"))}
        dfl.dualflow_release_slots(run.ctx, run.kv, slot, 1)
        assert run.status() == 0
        assert np.array_equal(run.seq_len.cpu().numpy(), [L[0], 0, L[2]])
        prompt = np.random.default_rng(43).integers(0, w.vocab, size=(1, n)).astype(np.int32)
        dfl.dualflow_prefill_reserve(run.ctx, n)
        dfl.dualflow_prefill_slots(run.ctx, run.weights, run.kv, torch.from_numpy(prompt).to(cuda_device), slot, 1, n)
        assert run.status() == 0
        L2 = np.array([L[0], n, L[2]])
        assert np.array_equal(run.seq_len.cpu().numpy(), L2)

        caches = _oracle_caches(w)
        glob = {"E1": H.LazyRows(w, "E1"), "E2": H.LazyRows(w, "E2"), "W_lm": H.host_f64(w, "W_lm"),
                "g_final": H.host_f64(w, "g_final")}
        layers = H.LazyLayers(w)
        O.prefill(H.hparams(w), glob, layers, [O.DenseCache(K=c.K[1:2], V=c.V[1:2]) for c in caches], prompt,
                  np.array([0]), mirror=True)
        for l in range(w.n_layers):
            for kind in ("K", "V"):
                t = run.t[f"L{l}.{kind}"]
                ref = caches[l].K if kind == "K" else caches[l].V
                err = H.rel_err(H.to_f64(t[1, :, :n, :]), ref[1][:, :n, :])
                assert err <= TOL, f"layer {l} {kind}: rel err {err:.3e}"
                exp = before[f"L{l}.{kind}"].clone()
                exp[1, :, :n, :] = t[1, :, :n, :]
                assert torch.equal(exp, t), f"layer {l} {kind}: cache changed outside the new prompt's rows"

        nxt = np.random.default_rng(44).integers(0, w.vocab, size=w.batch).astype(np.int32)
        run.tokens.copy_(torch.from_numpy(nxt))
        run.step(aux_on=1)
        assert run.status() == 0
        ref = O.decode_step(H.hparams(w), glob, layers, caches, nxt, L2, aux_on=True, mirror=True)
        got = H.to_f64(run.logits)
        for f in range(2):
            err = H.rel_err(got[f], ref["logits"][f])
            assert err <= TOL, f"decode after the slot prefill, flow {f + 1}: rel err {err:.3e}"
    finally:
        run.close()


MOE_SMALL = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=1, ffn_hidden=128, vocab=1000, batch=2,
                 n_experts=6, topk_primary=2, topk_aux=3, ctx_len=0, ctx_lo=5, ctx_hi=200, gain_sigma=0.1)
# The expert choice is an integer decided by floating point. The GPU's router logits differ from
# the oracle's (mirror mode) by far less than 5e-3 of their largest magnitude, so where every
# top-2 decision of the prompt has gaps above that (set and order), the choice is unique and must
# match; this prompt seed is such a case, and the test checks the premise on the oracle's logits.
MOE_TIE = 5e-3
MOE_PROMPT_SEED = 40


def test_prefill_moe_parity(cuda_device):
    """Primary-only prefill of a MoE model (router, top-k, each expert's gate/up + SwiGLU and
    down on the rows that chose it, mixed in set order) against the oracle's prefill, then a
    decode step of both flows after it."""
    w = W.MOE_16L_B64.replace(**MOE_SMALL)
    n = 7
    run = H.DeviceRun(w, cuda_device)
    try:
        L = run.seq_len_np.astype(np.int64)
        prompt = np.random.default_rng(MOE_PROMPT_SEED).integers(0, w.vocab, size=(w.batch, n)).astype(np.int32)
        before = {k: v.clone() for k, v in run.t.items() if k.endswith((".K", ".V"))}
        dfl.dualflow_prefill_reserve(run.ctx, w.batch * n)
        dfl.dualflow_prefill(run.ctx, run.weights, run.kv, torch.from_numpy(prompt).to(cuda_device), w.batch, n)
        assert run.status() == 0
        assert np.array_equal(run.seq_len.cpu().numpy(), L + n)

        caches = _oracle_caches(w)
        glob = {"E1": H.LazyRows(w, "E1"), "E2": H.LazyRows(w, "E2"), "W_lm": H.host_f64(w, "W_lm"),
                "g_final": H.host_f64(w, "g_final")}
        layers = H.LazyLayers(w)
        ref_pf = O.prefill(H.hparams(w), glob, layers, caches, prompt, L, mirror=True)
        rl = ref_pf["rlog"]
        s = -np.sort(-rl, axis=-1)
        m = np.abs(rl).max(axis=-1)
        assert np.all(s[..., 0] - s[..., 1] > MOE_TIE * m) and np.all(s[..., 1] - s[..., 2] > MOE_TIE * m)
        for l in range(w.n_layers):
            for kind in ("K", "V"):
                t = run.t[f"L{l}.{kind}"]
                ref = caches[l].K if kind == "K" else caches[l].V
                exp = before[f"L{l}.{kind}"].clone()
                for b in range(w.batch):
                    err = H.rel_err(H.to_f64(t[b, :, L[b]:L[b] + n, :]), ref[b][:, L[b]:L[b] + n, :])
                    assert err <= TOL, f"layer {l} {kind} seq {b}: rel err {err:.3e}"
                    exp[b, :, L[b]:L[b] + n, :] = t[b, :, L[b]:L[b] + n, :]
                assert torch.equal(exp, t), f"layer {l} {kind}: cache changed outside the prompt's rows"

        nxt = np.random.default_rng(42).integers(0, w.vocab, size=w.batch).astype(np.int32)
        run.tokens.copy_(torch.from_numpy(nxt))
        run.tokens_np = nxt
        run.step(aux_on=1)
        assert run.status() == 0
        ref = O.decode_step(H.hparams(w), glob, layers, caches, nxt, L + n, aux_on=True, mirror=True)
        got = H.to_f64(run.logits)
        for f in range(2):
            err = H.rel_err(got[f], ref["logits"][f])
            assert err <= TOL, f"decode after the MoE prefill, flow {f + 1}: rel err {err:.3e}"
    finally:
        run.close()


def test_prefill_moe_matches_decode_steps(cuda_device):
    """A longer MoE prompt (several 256-row blocks per expert after gathering) against the same
    prompt fed as primary-only decode steps, one position at a time, on the GPU: the cache entries
    both write and the logits of a decode step of both flows after them agree at the bf16 bar.
    Every row takes all experts (top-k = E): the two paths' router logits differ by rounding, so
    with a smaller k a near tie could hand a row different experts on each path; with k = E only
    the mixing order can differ, which changes nothing beyond rounding."""
    w = W.MOE_16L_B64.replace(**dict(MOE_SMALL, batch=3, ctx_lo=0, ctx_hi=700, topk_primary=6, topk_aux=6))
    n = 300
    runs = [H.DeviceRun(w, cuda_device) for _ in range(2)]
    try:
        lens = np.array([0, 41, 300], dtype=np.int32)
        for r in runs:
            r.seq_len.copy_(torch.from_numpy(lens))
        prompt = np.random.default_rng(47).integers(0, w.vocab, size=(w.batch, n)).astype(np.int32)
        a, b = runs
        dfl.dualflow_prefill_reserve(a.ctx, w.batch * n)
        dfl.dualflow_prefill(a.ctx, a.weights, a.kv, torch.from_numpy(prompt).to(cuda_device), w.batch, n)
        assert a.status() == 0
        dfl.dualflow_set_graphs(b.ctx, 0)
        for t in range(n):
            b.tokens.copy_(torch.from_numpy(prompt[:, t].copy()))
            b.step(aux_on=0)
            b.seq_len.add_(1)
        assert b.status() == 0
        assert torch.equal(a.seq_len, b.seq_len)
        for l in range(w.n_layers):
            for kind in ("K", "V"):
                ta, tb = a.t[f"L{l}.{kind}"], b.t[f"L{l}.{kind}"]
                for s in range(w.batch):
                    err = H.rel_err(H.to_f64(ta[s, :, lens[s]:lens[s] + n, :]), H.to_f64(tb[s, :, lens[s]:lens[s] + n, :]))
                    assert err <= TOL, f"layer {l} {kind} seq {s}: rel err {err:.3e}"
        nxt = torch.from_numpy(np.random.default_rng(48).integers(0, w.vocab, size=w.batch).astype(np.int32))
        for r in runs:
            r.tokens.copy_(nxt)
            r.step(aux_on=1)
            assert r.status() == 0
        for f in range(2):
            err = H.rel_err(H.to_f64(a.logits[f]), H.to_f64(b.logits[f]))
            assert err <= TOL, f"flow {f + 1}: rel err {err:.3e}"
    finally:
        for r in runs:
            r.close()
