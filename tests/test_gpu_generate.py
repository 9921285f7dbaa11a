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


PEAKED_SIGMA = 0.4  # LM-head weights: logits of a few units, so the next-token distribution is peaked


def _peaked_lm(w, dev):
    """A peaked LM head drawn by the seeded generator: (device bf16 [V, d], host fp64 [V, d])."""
    import dfsynth
    t = torch.empty((w.vocab, w.d_model), dtype=torch.bfloat16, device=dev)
    dfsynth.cuda_normal_(t.data_ptr(), w.seed, "W_lm_peaked", t.numel(), PEAKED_SIGMA, w.dtype)
    host = O.widen(dfsynth.host_normal(w.seed, "W_lm_peaked", (w.vocab, w.d_model), PEAKED_SIGMA, w.dtype), w.dtype)
    return t, host.reshape(w.vocab, w.d_model)


def _derived_override(gpu_tok, gpu_logits, u, counts):
    """Token check with a near-tie window derived from the two distributions themselves: the GPU's
    mixture distribution (from its own logits, in fp64) and the oracle's differ in their cumulative
    sums by at most dC, so wherever u is farther than dC from both ends of the oracle's interval (or,
    for argmax, the oracle's top-2 gap exceeds twice the largest probability difference) the GPU's
    token must equal the oracle's. The slack 1e-5 covers the GPU computing its mixture in fp32."""

    def f(t, b, tok, p):
        g = int(gpu_tok[t, b])
        lg = gpu_logits[t, :, b]
        pg = O.choice_distribution(lg[0], lg[1])
        if u is None:
            dp = float(np.max(np.abs(pg - p))) + 1e-5
            srt = np.sort(p)
            if srt[-1] - srt[-2] > 2 * dp:
                counts[0] += 1
                assert g == tok, f"step {t} row {b}: GPU token {g}, oracle {tok}"
                return tok
            assert p[g] >= srt[-1] - 2 * dp, f"step {t} row {b}: GPU token {g} is not a near tie"
            return g
        C, Cg = np.cumsum(p), np.cumsum(pg)
        dC = float(np.max(np.abs(Cg - C))) + 1e-5
        uu = float(u[t, b])
        lo = C[g - 1] if g > 0 else 0.0
        assert lo <= uu + dC and C[g] >= uu - dC, f"step {t} row {b}: GPU sample {g} off the interval"
        olo = C[tok - 1] if tok > 0 else 0.0
        if uu - olo > dC and C[tok] - uu > dC:
            counts[0] += 1
            assert g == tok, f"step {t} row {b}: GPU sample {g}, oracle {tok}"
            return tok
        return g
    return f


@pytest.mark.parametrize("mode", ["greedy", "sampled"])
def test_generate_peaked_bf16(cuda_device, mode):
    """bf16 generation with a peaked next-token distribution: every step's logits against the oracle
    at 2e-2, and the tokens compared exactly outside the derived near-tie window -- at least half of
    the sampled choices are."""
    w = CASES["dense_small_g4"][0].replace(batch=4)
    n = 5
    dev = cuda_device
    W_lm_d, W_lm_h = _peaked_lm(w, dev)
    run = H.DeviceRun(w, dev, overrides={"W_lm": W_lm_d})
    try:
        run.rebuild_structs()
        u = _uniforms(n, w.batch, seed=13) if mode == "sampled" else None
        gpu_tok, logits_all = _run_gpu(run, w, n, u)
        assert run.status() == 0
        got = H.to_f64(logits_all)
        counts = [0]
        glob = {"E1": H.LazyRows(w, "E1"), "E2": H.LazyRows(w, "E2"), "W_lm": W_lm_h,
                "g_final": H.host_f64(w, "g_final")}
        ref = O.generate(H.hparams(w), glob, H.LazyLayers(w), _oracle_caches(w), run.tokens_np, run.seq_len_np, n,
                         u=u, aux_on=True, mirror=True, token_override=_derived_override(gpu_tok, got, u, counts))
        assert np.array_equal(ref["tokens"], gpu_tok)
        total = n * w.batch
        print(f"[generate peaked {mode}] tokens compared exactly: {counts[0]}/{total}")
        assert counts[0] >= total // 2, f"only {counts[0]} of {total} choices compared exactly"
        for t in range(n):
            for f in range(2):
                err = H.rel_err(got[t, f], ref["logits"][t, f])
                assert err <= 2e-2, f"step {t} flow {f + 1}: rel err {err:.3e}"
    finally:
        run.close()


def test_generate_paged_matches_oracle(cuda_device):
    """The decode loop through a shuffled paged cache that grows over the steps, against the
    oracle's decode loop on a paged cache with the same table: logits at 2e-2, tokens exact outside
    the near-tie window, and the pages the loop took from the free list."""
    w = CASES["dense_small_g4"][0]
    tol, tie = CASES["dense_small_g4"][1:]
    n = 20
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
        tok_p = torch.full((n, w.batch), -7, dtype=torch.int32, device=cuda_device)
        log_p = torch.full((n, 2, w.batch, w.vocab), float("nan"), device=cuda_device)
        logits = torch.empty((2, w.batch, w.vocab), device=cuda_device)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            dfl.dualflow_generate(ctx_p, run.weights, kv_p, run.tokens, w.batch, n, tok_p, logits, logits_all=log_p,
                                  free_pages=free_d, n_free=n_free, stream=s)
        s.synchronize()
        assert dfl.dualflow_sync_status(ctx_p) == 0
        gpu_tok = tok_p.cpu().numpy()
        # the table the loop must end with, replayed on the host from the documented order (the
        # page a sequence opens is popped from the top of the free list, sequences in index order)
        exp_table, exp_free = table.copy(), list(free)
        L = run.seq_len_np.astype(np.int64).copy()
        for _ in range(n):
            for b in range(w.batch):
                L[b] += 1
                if L[b] % 16 == 0 and exp_table[b, L[b] // 16] < 0:
                    exp_table[b, L[b] // 16] = exp_free.pop()
        assert np.array_equal(table_d.cpu().numpy(), exp_table)
        # the oracle's paged caches: the cached positions in the pages the table maps, every other
        # slot unwritten (NaN); the oracle's own appends fill the growth pages of exp_table
        caches = []
        for l in range(w.n_layers):
            Kh = H.host_f64(w, f"L{l}.K").reshape(w.cache_shape())
            Vh = H.host_f64(w, f"L{l}.V").reshape(w.cache_shape())
            pk = np.full((total, w.n_kv_heads, 16, w.head_dim), np.nan)
            pv = np.full_like(pk, np.nan)
            for b in range(w.batch):
                for pos in range(int(run.seq_len_np[b])):
                    pid = int(table[b, pos // 16])
                    pk[pid][:, pos % 16] = Kh[b][:, pos]
                    pv[pid][:, pos % 16] = Vh[b][:, pos]
            caches.append(O.PagedCache(pk, pv, exp_table, 16))
        counts = [0]
        glob = {"E1": H.LazyRows(w, "E1"), "E2": H.LazyRows(w, "E2"), "W_lm": H.host_f64(w, "W_lm"),
                "g_final": H.host_f64(w, "g_final")}
        ref = O.generate(H.hparams(w), glob, H.LazyLayers(w), caches, run.tokens_np, run.seq_len_np, n,
                         aux_on=True, mirror=True, token_override=_override(gpu_tok, None, tie, counts))
        assert np.array_equal(ref["tokens"], gpu_tok)
        assert counts[0] > 0
        got = H.to_f64(log_p)
        for t in range(n):
            for f in range(2):
                err = H.rel_err(got[t, f], ref["logits"][t, f])
                assert err <= tol, f"step {t} flow {f + 1}: rel err {err:.3e}"
    finally:
        if ctx_p:
            dfl.dualflow_free(ctx_p)
        run.close()
