"""Failure paths on the GPU that fault, trap or hang nothing.

An expired bounded wait: with the kernels' pipeline-wait limit lowered to 1 ns (a test-only knob)
the waits on the asynchronous copies give up, the step latches DF_ERR_TIMEOUT, every copy already
issued is still awaited before its CTA exits, and the same context then runs a correct step.

Concurrent launches: two contexts driven from two host threads on their own streams, with different
batch sizes (different dynamic shared memory per launch), give the results of the same calls made
one after the other -- no launch changes a process-wide kernel attribute that another thread's
launch relies on."""
import threading

import pytest
import torch

import dual_flow_decode_dualflow_b300 as dfl
from dfsynth import workloads as W
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

SMALL = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=1, ffn_hidden=512, vocab=1000, batch=3, ctx_len=0,
             ctx_lo=5, ctx_hi=200, gain_sigma=0.1)


def test_expired_wait_reports_timeout_and_context_recovers(cuda_device):
    w = W.DENSE_24L_B32_L4096.replace(**SMALL)
    run = H.DeviceRun(w, cuda_device)
    try:
        dfl.dualflow_set_graphs(run.ctx, 0)
        keep = {k: v.clone() for k, v in run.t.items() if k.endswith((".K", ".V"))}
        run.step(aux_on=1)
        assert run.status() == 0
        good = run.logits.clone()
        dfl.dualflow_set_wait_limit(run.ctx, 1)
        run.step(aux_on=1)
        assert run.status() == dfl.DF_ERR_TIMEOUT
        dfl.dualflow_set_wait_limit(run.ctx, 0)
        for k, v in keep.items():  # the failed step wrote garbage into slot L_b only; start clean
            run.t[k].copy_(v)
        run.logits.fill_(float("nan"))
        run.step(aux_on=1)
        assert run.status() == 0
        assert torch.equal(run.logits, good)
    finally:
        run.close()


def test_expired_wait_in_attention_only_call(cuda_device):
    w = W.ATTN_B8_L2048.replace(d_model=256, n_q_heads=8, n_kv_heads=2, batch=4, ctx_len=0, ctx_lo=100, ctx_hi=900)
    run = H.DeviceRun(w, cuda_device)
    try:
        run.attention(aux_on=1)
        assert run.status() == 0
        good = run.o.clone()
        dfl.dualflow_set_wait_limit(run.ctx, 1)
        run.attention(aux_on=1)
        assert run.status() == dfl.DF_ERR_TIMEOUT
        dfl.dualflow_set_wait_limit(run.ctx, 0)
        run.o.fill_(float("nan"))
        run.attention(aux_on=1)
        assert run.status() == 0
        assert torch.equal(run.o, good)
    finally:
        run.close()


def test_concurrent_contexts_on_two_host_threads(cuda_device):
    base = W.ATTN_B8_L2048.replace(d_model=512, n_q_heads=8, n_kv_heads=2, ctx_len=0, ctx_lo=50, ctx_hi=1500)
    runs = [H.DeviceRun(base.replace(batch=8), cuda_device), H.DeviceRun(base.replace(batch=2, seed=1077), cuda_device)]
    try:
        ref = []
        for r in runs:  # one after the other
            r.attention(aux_on=1)
            assert r.status() == 0
            ref.append(r.o.clone())
            r.o.fill_(float("nan"))
        errors = []

        def worker(r, reps=50):
            try:
                s = torch.cuda.Stream(device=cuda_device)
                for _ in range(reps):
                    r.attention(aux_on=1, stream=s)
                s.synchronize()
            except Exception as exc:  # reported below
                errors.append(exc)

        threads = [threading.Thread(target=worker, args=(r,)) for r in runs]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        assert not errors, errors
        for r, o in zip(runs, ref):
            assert r.status() == 0
            assert torch.equal(r.o, o)
    finally:
        for r in runs:
            r.close()
