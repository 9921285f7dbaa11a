"""The decode loop (dualflow_generate) on the GPU against the oracle's generation loop.

Each step's logits are compared at the path's bar (1e-5 fp32, 2e-2 bf16). A token is an integer
decided by floating point: where the oracle's choice has a margin (top-2 probability gap, or the
sampling uniform's distance from every cumulative boundary) above the near-tie threshold, the GPU
token must equal it; otherwise the GPU token must be one the threshold admits, and the oracle
continues with the GPU's token so that one near tie cannot derail the rest of the comparison.
A paged cache must give bit-identical tokens and logits to the contiguous one, with its new pages
taken from the free list in the documented order."""
import numpy as np
import pytest
import torch

import dual_flow_decode_dualflow_b300 as dfl
import oracle as O
from dfsynth import workloads as W
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

SMALL = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=1, ffn_hidden=512, vocab=1000, batch=3, ctx_len=0,
             ctx_lo=5, ctx_hi=200, gain_sigma=0.1)
# (workload, logits bar, near-tie threshold: relative top-2 probability gap for argmax, absolute
# distance of u from its interval's ends for sampling)
CASES = {
    "tiny_f32_1layer": (W.TINY_F32, 1e-5, (1e-4, 1e-4)),
    "dense_small_g4": (W.DENSE_24L_B32_L4096.replace(**SMALL), 2e-2, (3e-2, 5e-3)),
}


def _uniforms(n, B, seed=5):
    # multiples of 2^-24: exact in fp32 and fp64
    rng = np.random.default_rng(seed)
    return (rng.integers(0, 1 << 24, size=(n, B)) / float(1 << 24)).astype(np.float32)


def _oracle_caches(w):
    out = []
    for l in range(w.n_layers):
        K = H.host_f64(w, f"L{l}.K").reshape(w.cache_shape()).copy()
        V = H.host_f64(w, f"L{l}.V").reshape(w.cache_shape()).copy()
        out.append(O.DenseCache(K=K, V=V))
    return out


def _run_gpu(run, w, n, u=None, aux_on=1):
    dev = run.dev
    tok_out = torch.full((n, w.batch), -7, dtype=torch.int32, device=dev)
    logits_all = torch.full((n, 2, w.batch, w.vocab), float("nan"), device=dev)
    d_u = torch.from_numpy(u).to(dev) if u is not None else None
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dfl.dualflow_generate(run.ctx, run.weights, run.kv, run.tokens, w.batch, n, tok_out, run.logits, u=d_u,
                              logits_all=logits_all, aux_on=aux_on, stream=s)
    s.synchronize()
    return tok_out.cpu().numpy(), logits_all


def _override(gpu_tok, u, tie, counts):
    tie_p, tie_c = tie

    def f(t, b, tok, p):
        g = int(gpu_tok[t, b])
        if u is None:
            srt = np.sort(p)
            if srt[-1] - srt[-2] > tie_p * srt[-1]:
                counts[0] += 1
                assert g == tok, f"step {t} row {b}: GPU token {g}, oracle {tok}"
                return tok
            assert p[g] >= p.max() * (1 - tie_p), f"step {t} row {b}: GPU token {g} is not a near tie"
            return g
        C = np.cumsum(p)
        uu = float(u[t, b])
        lo = C[g - 1] if g > 0 else 0.0
        assert lo <= uu + 6 * tie_c and C[g] >= uu - 6 * tie_c, f"step {t} row {b}: GPU sample {g} off the interval"
        olo = C[tok - 1] if tok > 0 else 0.0  # the oracle's interval [olo, C[tok]) holds u
        if uu - olo > tie_c and C[tok] - uu > tie_c:
            counts[0] += 1
            assert g == tok, f"step {t} row {b}: GPU sample {g}, oracle {tok}"
            return tok
        return g
    return f


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("mode", ["greedy", "sampled", "primary_only"])
def test_generate_parity(cuda_device, name, mode):
    w, tol, tie = CASES[name]
    n = 4
    run = H.DeviceRun(w, cuda_device)
    try:
        u = _uniforms(n, w.batch) if mode == "sampled" else None
        aux_on = 0 if mode == "primary_only" else 1
        gpu_tok, logits_all = _run_gpu(run, w, n, u, aux_on)
        assert run.status() == 0
        assert np.all((gpu_tok >= 0) & (gpu_tok < w.vocab))
        assert np.array_equal(run.seq_len.cpu().numpy(), run.seq_len_np + n)
        counts = [0]
        glob = {"E1": H.LazyRows(w, "E1"), "E2": H.LazyRows(w, "E2"), "W_lm": H.host_f64(w, "W_lm"),
                "g_final": H.host_f64(w, "g_final")}
        ref = O.generate(H.hparams(w), glob, H.LazyLayers(w), _oracle_caches(w), run.tokens_np, run.seq_len_np, n,
                         u=u, aux_on=bool(aux_on), mirror=True, token_override=_override(gpu_tok, u, tie, counts))
        assert np.array_equal(ref["tokens"], gpu_tok)
        # bf16 logits cannot place u inside the narrow intervals of a near-uniform distribution:
        # sampled bf16 tokens are checked for validity only
        if not (mode == "sampled" and w.dtype == "bf16"):
            assert counts[0] > 0, "every choice was a near tie: nothing compared exactly"
        got = H.to_f64(logits_all)
        for t in range(n):
            for f in range(2 if aux_on else 1):
                err = H.rel_err(got[t, f], ref["logits"][t, f])
                assert err <= tol, f"step {t} flow {f + 1}: rel err {err:.3e}"
    finally:
        run.close()


def _paged_copy(run, w, n, extra, seed=31):
    """A paged copy (pages of 16) of a contiguous run's caches: each sequence's held positions
    L_b + 1 mapped to shuffled physical pages, the pages its growth over n steps needs plus `extra`
    in a free list (NaN-filled). Returns (K pages, V pages, table, free list, total pages)."""
    ps = 16
    lens = run.seq_len_np.astype(np.int64)
    held = (lens + 1 + ps - 1) // ps
    grow = (lens + 1 + n + ps - 1) // ps - held
    total = int(held.sum() + grow.sum()) + extra
    perm = np.random.default_rng(seed).permutation(total).astype(np.int32)
    pps = (w.max_ctx + ps - 1) // ps
    table = np.full((w.batch, pps), -1, dtype=np.int32)
    off = 0
    for b in range(w.batch):
        table[b, : held[b]] = perm[off: off + held[b]]
        off += int(held[b])
    free = perm[off:].copy()
    Ks, Vs = [], []
    for l in range(w.n_layers):
        for name, lst in (("K", Ks), ("V", Vs)):
            src = run.t[f"L{l}.{name}"]
            pages = torch.full((total, w.n_kv_heads, ps, w.head_dim), float("nan"), dtype=src.dtype, device=src.device)
            for b in range(w.batch):
                for j in range(held[b]):
                    pages[int(table[b, j])] = src[b, :, j * ps:(j + 1) * ps, :]
            lst.append(pages)
    return Ks, Vs, table, free, total


def test_generate_paged_matches_contiguous(cuda_device):
    """Bit-identical tokens and logits through a shuffled paged cache that grows over the steps,
    its new pages popped from the free list in sequence order."""
    w = CASES["dense_small_g4"][0]
    n = 20  # every sequence crosses at least one page boundary
    run = H.DeviceRun(w, cuda_device)
    ctx_p = None
    try:
        Ks, Vs, table, free, total = _paged_copy(run, w, n, extra=3)
        cfg = H.config_for(w)
        cfg.paged, cfg.page_size, cfg.max_pages = 1, 16, total
        ctx_p = dfl.dualflow_init(cfg)
        seq_p = torch.from_numpy(run.seq_len_np.copy()).to(cuda_device)
        table_d = torch.from_numpy(table.copy()).to(cuda_device)
        kv_p = dfl.make_kv(Ks, Vs, seq_p, table_d)
        free_d = torch.from_numpy(free.copy()).to(cuda_device)
        n_free = torch.tensor([len(free)], dtype=torch.int32, device=cuda_device)
        tok_c, log_c = _run_gpu(run, w, n)
        assert run.status() == 0
        tok_p = torch.full((n, w.batch), -7, dtype=torch.int32, device=cuda_device)
        log_p = torch.full((n, 2, w.batch, w.vocab), float("nan"), device=cuda_device)
        logits = torch.empty((2, w.batch, w.vocab), device=cuda_device)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            dfl.dualflow_generate(ctx_p, run.weights, kv_p, run.tokens, w.batch, n, tok_p, logits, logits_all=log_p,
                                  free_pages=free_d, n_free=n_free, stream=s)
        s.synchronize()
        assert dfl.dualflow_sync_status(ctx_p) == 0
        assert np.array_equal(tok_p.cpu().numpy(), tok_c)
        assert torch.equal(log_p, log_c)
        # the page allocation the loop documents, replayed on the host
        exp_table, exp_free = table.copy(), list(free)
        L = run.seq_len_np.astype(np.int64).copy()
        for _ in range(n):
            for b in range(w.batch):
                L[b] += 1
                if L[b] % 16 == 0 and exp_table[b, L[b] // 16] < 0:
                    exp_table[b, L[b] // 16] = exp_free.pop()
        assert np.array_equal(table_d.cpu().numpy(), exp_table)
        assert int(n_free.item()) == len(exp_free) == 3
        assert np.array_equal(seq_p.cpu().numpy(), L)
    finally:
        if ctx_p:
            dfl.dualflow_free(ctx_p)
        run.close()


def test_generate_stops_at_capacity(cuda_device):
    """A sequence whose next slot would reach max_ctx stops advancing and latches a bounds error."""
    w = CASES["tiny_f32_1layer"][0]
    run = H.DeviceRun(w, cuda_device)
    try:
        room = w.max_ctx - 1 - int(run.seq_len_np.max())
        n = room + 3
        _run_gpu(run, w, n)
        assert run.status() == dfl.DF_ERR_DEVICE_BOUNDS
        assert int(run.seq_len.max().item()) == w.max_ctx - 1
    finally:
        run.close()


def test_generate_host_matches_device(cuda_device):
    """The host-buffer decode call returns the tokens the device call chooses, bit for bit, and
    advances the lengths the same way."""
    w = CASES["dense_small_g4"][0]
    n = 5
    run = H.DeviceRun(w, cuda_device)
    try:
        u = _uniforms(n, w.batch, seed=9)
        ref_tok, _ = _run_gpu(run, w, n, u)
        assert run.status() == 0
        run.seq_len.copy_(torch.from_numpy(run.seq_len_np))
        tok_h = torch.from_numpy(run.tokens_np.copy()).pin_memory()
        out_h = torch.full((n, w.batch), -7, dtype=torch.int32).pin_memory()
        u_h = torch.from_numpy(u).pin_memory()
        s = torch.cuda.Stream()
        dfl.dualflow_generate_host(run.ctx, run.weights, run.kv, tok_h, w.batch, n, out_h, u_host=u_h, stream=s)
        assert run.status() == 0
        assert np.array_equal(out_h.numpy(), ref_tok)
        assert np.array_equal(run.seq_len.cpu().numpy(), run.seq_len_np + n)
        with pytest.raises(dfl.DualFlowError):
            dfl.dualflow_generate_host(run.ctx, run.weights, run.kv, tok_h, w.batch, 257, out_h, stream=s)
    finally:
        run.close()
