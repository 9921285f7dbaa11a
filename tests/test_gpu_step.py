"""The whole dual-flow decode step (dualflow_step) against the oracle, plus the method's invariants
checked on the GPU: primary bit-identical with and without the auxiliary flow, cache untouched
outside slot L_b, auxiliary == primary when the flows are uncoupled and share the embedding.

The parity bar is taken against the oracle's mirror mode, which rounds to bf16 exactly where the
GPU path stores bf16. The error against the plain fp64 definition (no intermediate rounding) is
also reported and bounded: for bf16 storage it is the storage error accumulated over the depth
(measured on B300 at <= 2.8e-3 for the 1-2 layer cases and 1.7e-2 for the 24-layer workload; bounds
1e-2 and 4e-2), for fp32 storage it stays within the fp32 bar of 1e-5."""
TOL_PLAIN_BF16 = 1e-2
TOL_PLAIN_DEEP = 4e-2


def CACHE_DRIFT(l):
    """Bound of the appended K/V entry of layer l (0-based) of the 24-layer workload against the
    mirrored oracle: the bf16 bar up to the eighth layer, then 1e-3 more per layer. The entry is
    computed from the residual stream after l layers, whose deviation from the mirrored oracle grows
    with depth (one-ulp rounding flips of stored operands that the mirror mode cannot follow):
    measured on B300 from 6.8e-4 at the first layer to 1.2e-2 at the eighth and 2.1e-2 at the 23rd,
    a margin of at least 1.6 everywhere."""
    return 2e-2 + 1e-3 * max(0, l - 8)
import numpy as np
import pytest
import torch

from dfsynth import workloads as W
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

SMALL = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=1, ffn_hidden=512, vocab=1000, batch=3, ctx_len=0,
             ctx_lo=5, ctx_hi=200, gain_sigma=0.1)
CASES = {
    "tiny_f32_1layer": (W.TINY_F32, 1e-5),
    "dense_small_g4": (W.DENSE_24L_B32_L4096.replace(**SMALL), 2e-2),
    "dense_small_g2": (W.DENSE_24L_B32_L4096.replace(**dict(SMALL, n_q_heads=4, n_kv_heads=2, batch=5)), 2e-2),
    "dense_small_b32": (W.DENSE_24L_B32_L4096.replace(**dict(SMALL, batch=32, n_layers=1, ctx_lo=60, ctx_hi=70)),
                        2e-2),
    # the full model's widths and batch over two layers: every projection in the tile and split-K
    # configuration of the benchmarked step
    "dense_d2048_2l_b32": (W.DENSE_24L_B32_L4096.replace(n_layers=2, ctx_len=256, gain_sigma=0.1), 2e-2),
}


def _check_logits(run, w, rows, tol, ref, label=""):
    got = H.to_f64(run.logits)[:, rows]
    if label:
        print(f"[step {label}] logits vs mirrored oracle: rel err "
              + " / ".join(f"{H.rel_err(got[f], ref['logits'][f]):.3e}" for f in range(2)))
    for f in range(2):
        err = H.rel_err(got[f], ref["logits"][f])
        assert err <= tol, f"flow {f + 1} logits: rel err {err:.3e}"
        if w.dtype == "f32":
            r = ref["logits"][f]
            assert np.all(np.abs(got[f] - r) <= 1e-5 * np.abs(r) + 1e-6 * np.abs(r).max())


def _check_plain(run, w, rows, tol, label):
    """Logits against the unmirrored oracle: the plain fp64 definition of the step."""
    plain = H.oracle_step(w, rows=rows, mirror=False)
    got = H.to_f64(run.logits)[:, rows]
    for f in range(2):
        err = H.rel_err(got[f], plain["logits"][f])
        print(f"[step {label}] flow {f + 1} logits vs unmirrored oracle: rel err {err:.3e}")
        assert err <= tol, f"flow {f + 1} vs the unmirrored oracle: rel err {err:.3e}"


def _check_cache(run, w, rows, tol, ref, before, label=""):
    """Slot L_b holds the oracle's new entry (tol: a number, or a function of the layer index);
    every other element is bit-identical to before."""
    lens = run.seq_len_np
    bound = tol if callable(tol) else (lambda l: tol)
    worst = []
    for l in range(w.n_layers):
        e = 0.0
        for kind, key in (("K", "k_new"), ("V", "v_new")):
            t = run.t[f"L{l}.{kind}"]
            e = max([e] + [H.rel_err(H.to_f64(t[b, :, lens[b], :]), ref[key][l, i]) for i, b in enumerate(rows)])
            if before is not None:
                exp = before[f"L{l}.{kind}"].clone()
                for b in range(w.batch):
                    exp[b, :, lens[b], :] = t[b, :, lens[b], :]
                assert torch.equal(exp, t), f"layer {l} {kind}: cache changed outside slot L_b"
        worst.append(e)
    if label:
        print(f"[step {label}] appended K/V rel err per layer: " + " ".join(f"{x:.2e}" for x in worst))
    for l, e in enumerate(worst):
        assert e <= bound(l), f"layer {l} appended entry: rel err {e:.3e} > {bound(l):.3e}"


@pytest.mark.parametrize("name", list(CASES))
def test_step_parity(cuda_device, name):
    w, tol = CASES[name]
    run = H.DeviceRun(w, cuda_device)
    try:
        before = {k: v.clone() for k, v in run.t.items() if k.endswith((".K", ".V"))}
        rows = list(range(w.batch))
        run.step(aux_on=1)
        assert run.status() == 0
        ref = H.oracle_step(w, rows=rows)
        _check_logits(run, w, rows, tol, ref)
        _check_cache(run, w, rows, tol, ref, before)
        _check_plain(run, w, rows, tol if w.dtype == "f32" else TOL_PLAIN_BF16, name)
        logits_dual = run.logits.clone()
        caches_dual = {k: run.t[k].clone() for k in before}
        # primary-only step on the same inputs: primary logits and cache bit-identical
        for k in before:
            run.t[k].copy_(before[k])
        run.logits.fill_(float("nan"))
        run.step(aux_on=0)
        assert run.status() == 0
        assert torch.equal(run.logits[0], logits_dual[0])
        assert torch.isnan(run.logits[1]).all()
        for k in before:
            assert torch.equal(run.t[k], caches_dual[k])
    finally:
        run.close()


def test_uncoupled_tied_flows_coincide(cuda_device):
    w = W.DENSE_24L_B32_L4096.replace(**SMALL)
    run = H.DeviceRun(w, cuda_device)
    try:
        run.t["E2"] = run.t["E1"]
        for l in range(w.n_layers):
            for v in "abc":
                run.t[f"L{l}.{v}"] = torch.zeros_like(run.t[f"L{l}.{v}"])
        run.rebuild_structs()
        run.step(aux_on=1)
        assert run.status() == 0
        assert torch.equal(run.logits[0], run.logits[1])
    finally:
        run.close()


def test_graph_replay_matches_direct(cuda_device):
    import dual_flow_decode_dualflow_b300 as dfl
    w = W.DENSE_24L_B32_L4096.replace(**SMALL)
    run = H.DeviceRun(w, cuda_device)
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            run.step(aux_on=1, stream=s)  # captures
            run.step(aux_on=1, stream=s)  # replays
        s.synchronize()
        g = run.logits.clone()
        dfl.dualflow_set_graphs(run.ctx, 0)
        run.step(aux_on=1)
        torch.cuda.synchronize()
        assert torch.equal(g, run.logits)
    finally:
        run.close()


def test_step_host_buffers(cuda_device):
    import dual_flow_decode_dualflow_b300 as dfl
    w = W.DENSE_24L_B32_L4096.replace(**SMALL)
    run = H.DeviceRun(w, cuda_device)
    try:
        run.step(aux_on=1)
        torch.cuda.synchronize()
        ref = run.logits.cpu()
        tok = torch.from_numpy(run.tokens_np).pin_memory()
        out = torch.empty((2, w.batch, w.vocab), dtype=torch.float32).pin_memory()
        dfl.dualflow_step_host(run.ctx, run.weights, run.kv, tok, w.batch, out, 1)
        assert torch.equal(out, ref)
    finally:
        run.close()


def test_bad_token_reported(cuda_device):
    import dual_flow_decode_dualflow_b300 as dfl
    w = W.DENSE_24L_B32_L4096.replace(**SMALL)
    run = H.DeviceRun(w, cuda_device)
    try:
        run.tokens[0] = w.vocab + 5
        run.step(aux_on=1)
        assert run.status() == dfl.DF_ERR_DEVICE_BOUNDS
    finally:
        run.close()


@pytest.mark.slow
def test_step_full_dense_24l_sampled(cuda_device):
    """The full 24-layer, B=32, L=4096 workload, in the launch configuration the benchmark times,
    checked on sampled sequences (sequences are independent, so a subset is exact)."""
    w = W.DENSE_24L_B32_L4096
    rows = [0, 13, 31]
    run = H.DeviceRun(w, cuda_device)
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            run.step(aux_on=1, stream=s)
        s.synchronize()
        assert run.status() == 0
        ref = H.oracle_step(w, rows=rows)
        _check_logits(run, w, rows, 2e-2, ref, "full_24l_b32")
        _check_cache(run, w, rows, CACHE_DRIFT, ref, None, "full_24l_b32")
        _check_plain(run, w, rows, TOL_PLAIN_DEEP, "full_24l_b32")
    finally:
        run.close()


def test_step_parity_paged_ragged(cuda_device):
    """The full step on a paged cache (pages of 16, shuffled physical pages) with ragged lengths: the
    oracle's logits, the appended entry in the page that holds slot L_b, every other element of the
    pages unchanged, and the primary flow bit-identical without the auxiliary flow."""
    w = W.DENSE_24L_B32_L4096.replace(**dict(SMALL, batch=5, paged=True, page_size=16))
    run = H.DeviceRun(w, cuda_device)
    try:
        before = {k: v.clone() for k, v in run.t.items() if k.endswith((".K", ".V"))}
        rows = list(range(w.batch))
        run.step(aux_on=1)
        assert run.status() == 0
        ref = H.oracle_step(w, rows=rows)
        got = H.to_f64(run.logits)
        for f in range(2):
            err = H.rel_err(got[f], ref["logits"][f])
            assert err <= 2e-2, f"flow {f + 1} logits: rel err {err:.3e}"
        lens, table = run.seq_len_np, run.table_np
        for l in range(w.n_layers):
            for kind, key in (("K", "k_new"), ("V", "v_new")):
                t = run.t[f"L{l}.{kind}"]
                exp = before[f"L{l}.{kind}"].clone()
                for i, b in enumerate(rows):
                    pid, slot = int(table[b, lens[b] // 16]), int(lens[b] % 16)
                    assert H.rel_err(H.to_f64(t[pid, :, slot, :]), ref[key][l, i]) <= 2e-2
                    exp[pid, :, slot, :] = t[pid, :, slot, :]
                assert torch.equal(exp, t), f"layer {l} {kind}: pages changed outside slot L_b"
        dual = run.logits.clone()
        for k in before:
            run.t[k].copy_(before[k])
        run.step(aux_on=0)
        assert run.status() == 0
        assert torch.equal(run.logits[0], dual[0])
    finally:
        run.close()
