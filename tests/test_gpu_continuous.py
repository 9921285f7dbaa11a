"""Continuous batching on the GPU: sequences enter cache slots by a prefill, decode together in
the generation loop, leave (their slot released) and are replaced by new prompts.

The same scenario runs on a contiguous cache and on a paged cache (pages of 16 popped from a
shuffled free list on the device): tokens and logits must be bit-identical, and the paged
bookkeeping (table, free list, lengths) must equal its replay on the host, which follows the
documented order: prefill maps the pages of positions L .. L + n of each prompt's slot in prompt
and page order, every decode step maps the page its next slot opens, a release pushes the slot's
pages back in page order."""
import numpy as np
import pytest
import torch

import dual_flow_decode_dualflow_b300 as dfl
from dfsynth import workloads as W
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

SMALL = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=1, ffn_hidden=512, vocab=1000, batch=3, ctx_len=0,
             ctx_lo=5, ctx_hi=200, gain_sigma=0.1)
PS = 16


class HostPages:
    """Replay of the page bookkeeping the library documents."""

    def __init__(self, B, pps, free, max_ctx):
        self.tab = np.full((B, pps), -1, np.int64)
        self.free = list(free)
        self.L = np.zeros(B, np.int64)
        self.max_ctx = max_ctx

    def prefill(self, slots, n):
        for b in slots:
            for j in range(self.L[b] // PS, min(self.L[b] + n, self.max_ctx - 1) // PS + 1):
                if self.tab[b, j] < 0:
                    self.tab[b, j] = self.free.pop()
            self.L[b] += n

    def generate(self, n):
        for _ in range(n):
            for b in range(len(self.L)):
                self.L[b] += 1
                if self.L[b] % PS == 0 and self.tab[b, self.L[b] // PS] < 0:
                    self.tab[b, self.L[b] // PS] = self.free.pop()

    def release(self, slots):
        for b in slots:
            for j in range(self.tab.shape[1]):
                if self.tab[b, j] >= 0:
                    self.free.append(int(self.tab[b, j]))
                    self.tab[b, j] = -1
            self.L[b] = 0


def _generate(ctx, run, kv, tokens, n, free=None, n_free=None):
    w, dev = run.w, run.dev
    tok_out = torch.full((n, w.batch), -7, dtype=torch.int32, device=dev)
    logits = torch.empty((2, w.batch, w.vocab), device=dev)
    logits_all = torch.full((n, 2, w.batch, w.vocab), float("nan"), device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dfl.dualflow_generate(ctx, run.weights, kv, tokens, w.batch, n, tok_out, logits, logits_all=logits_all,
                              free_pages=free, n_free=n_free, stream=s)
    s.synchronize()
    assert dfl.dualflow_sync_status(ctx) == 0
    return tok_out.cpu().numpy(), logits_all


def test_continuous_batching_paged_matches_contiguous(cuda_device):
    w = W.DENSE_24L_B32_L4096.replace(**SMALL)
    dev = cuda_device
    B, n1, n2, steps = w.batch, 20, 37, 6
    run = H.DeviceRun(w, dev)  # contiguous cache and the weights
    ctx_p = None
    try:
        pps = (w.max_ctx + PS - 1) // PS
        total = B * pps
        cfg = H.config_for(w)
        cfg.paged, cfg.page_size, cfg.max_pages = 1, PS, total
        ctx_p = dfl.dualflow_init(cfg)
        shape = (total, w.n_kv_heads, PS, w.head_dim)
        Ks = [torch.full(shape, float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(w.n_layers)]
        Vs = [torch.full(shape, float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(w.n_layers)]
        table = torch.full((B, pps), -1, dtype=torch.int32, device=dev)
        seq_p = torch.zeros(B, dtype=torch.int32, device=dev)
        perm = np.random.default_rng(7).permutation(total).astype(np.int32)
        free = torch.from_numpy(perm.copy()).to(dev)
        n_free = torch.tensor([total], dtype=torch.int32, device=dev)
        kv_p = dfl.make_kv(Ks, Vs, seq_p, table)
        host = HostPages(B, pps, perm, w.max_ctx)

        # both caches start empty
        all_slots = torch.arange(B, dtype=torch.int32, device=dev)
        dfl.dualflow_release_slots(run.ctx, run.kv, all_slots, B)
        dfl.dualflow_release_slots(ctx_p, kv_p, all_slots, B, free, n_free)
        assert run.status() == 0 and dfl.dualflow_sync_status(ctx_p) == 0
        assert int(n_free.item()) == total and int(run.seq_len.abs().sum().item()) == 0
        for ctx in (run.ctx, ctx_p):
            dfl.dualflow_prefill_reserve(ctx, B * max(n1, n2))

        rng = np.random.default_rng(45)
        P = torch.from_numpy(rng.integers(0, w.vocab, size=(B, n1)).astype(np.int32)).to(dev)
        dfl.dualflow_prefill_slots(run.ctx, run.weights, run.kv, P, None, B, n1)
        dfl.dualflow_prefill_slots(ctx_p, run.weights, kv_p, P, None, B, n1, free, n_free)
        host.prefill(range(B), n1)
        start = torch.from_numpy(rng.integers(0, w.vocab, size=B).astype(np.int32)).to(dev)
        tok_c, log_c = _generate(run.ctx, run, run.kv, start, steps)
        tok_p, log_p = _generate(ctx_p, run, kv_p, start, steps, free, n_free)
        host.generate(steps)
        assert np.array_equal(tok_c, tok_p)
        assert torch.equal(log_c, log_p)

        # the sequence of slot 1 leaves; a longer prompt takes its slot
        one = torch.tensor([1], dtype=torch.int32, device=dev)
        dfl.dualflow_release_slots(run.ctx, run.kv, one, 1)
        dfl.dualflow_release_slots(ctx_p, kv_p, one, 1, free, n_free)
        host.release([1])
        Q = torch.from_numpy(rng.integers(0, w.vocab, size=(1, n2)).astype(np.int32)).to(dev)
        dfl.dualflow_prefill_slots(run.ctx, run.weights, run.kv, Q, one, 1, n2)
        dfl.dualflow_prefill_slots(ctx_p, run.weights, kv_p, Q, one, 1, n2, free, n_free)
        host.prefill([1], n2)
        nxt = torch.from_numpy(tok_c[-1].copy()).to(dev)
        nxt[1] = int(rng.integers(0, w.vocab))
        tok_c2, log_c2 = _generate(run.ctx, run, run.kv, nxt, steps)
        tok_p2, log_p2 = _generate(ctx_p, run, kv_p, nxt, steps, free, n_free)
        host.generate(steps)
        assert np.array_equal(tok_c2, tok_p2)
        assert torch.equal(log_c2, log_p2)

        exp_len = np.array([n1 + 2 * steps, n2 + steps, n1 + 2 * steps])
        assert np.array_equal(run.seq_len.cpu().numpy(), exp_len)
        assert np.array_equal(seq_p.cpu().numpy(), exp_len) and np.array_equal(host.L, exp_len)
        assert np.array_equal(table.cpu().numpy(), host.tab)
        nf = int(n_free.item())
        assert nf == len(host.free)
        assert np.array_equal(free.cpu().numpy()[:nf], np.array(host.free, np.int32))
    finally:
        if ctx_p:
            dfl.dualflow_free(ctx_p)
        run.close()


def test_release_and_prefill_reject_bad_arguments(cuda_device):
    w = W.DENSE_24L_B32_L4096.replace(**SMALL)
    run = H.DeviceRun(w, cuda_device)
    try:
        slots = torch.tensor([0], dtype=torch.int32, device=cuda_device)
        free = torch.zeros(4, dtype=torch.int32, device=cuda_device)
        n_free = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        with pytest.raises(dfl.DualFlowError):  # a contiguous context takes no free list
            dfl.dualflow_release_slots(run.ctx, run.kv, slots, 1, free, n_free)
        with pytest.raises(dfl.DualFlowError):
            dfl.dualflow_release_slots(run.ctx, run.kv, slots, w.batch + 1)
        dfl.dualflow_prefill_reserve(run.ctx, 8)
        tok = torch.zeros((1, 8), dtype=torch.int32, device=cuda_device)
        with pytest.raises(dfl.DualFlowError):
            dfl.dualflow_prefill_slots(run.ctx, run.weights, run.kv, tok, slots, 1, 8, free, n_free)
        with pytest.raises(dfl.DualFlowError):
            dfl.dualflow_prefill_slots(run.ctx, run.weights, run.kv, tok, slots, 1, 9)  # beyond the reserved rows
        # a slot outside the batch is caught on the device and latched; the other lengths stay
        bad = torch.tensor([w.batch + 5], dtype=torch.int32, device=cuda_device)
        dfl.dualflow_release_slots(run.ctx, run.kv, bad, 1)
        assert run.status() == dfl.DF_ERR_DEVICE_BOUNDS
        assert np.array_equal(run.seq_len.cpu().numpy(), run.seq_len_np)
    finally:
        run.close()
