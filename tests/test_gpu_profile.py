"""Per-kernel timing of the decode step (dualflow_set_profiling / dualflow_profile_read).

Mode 2 (in-graph end stamps, nothing serialised): every family that launched gets a positive
share, the shares add up to no more than the step's own event-timed duration and to most of it,
and the logits are bit-identical to those of an unprofiled step. Mode 1 (event pairs) reports every
family too. The launch counts match the step's structure."""
import pytest
import torch

import dual_flow_decode_dualflow_b300 as dfl
from dfsynth import workloads as W
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


def _timed_step(run, s):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        run.step(aux_on=1, stream=s)
        e1.record(s)
    e1.synchronize()
    return e0.elapsed_time(e1)


@pytest.mark.parametrize("name", ["dense", "moe"])
def test_in_graph_shares(cuda_device, name):
    w = (W.DENSE_24L_B32_L4096 if name == "dense" else W.MOE_16L_B64).replace(n_layers=2, ctx_len=1024)
    run = H.DeviceRun(w, cuda_device)
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            run.step(aux_on=1, stream=s)
        s.synchronize()
        ref = run.logits.clone()
        dfl.dualflow_set_profiling(run.ctx, 2)
        for _ in range(3):
            ms_step = _timed_step(run, s)
        ms, n = dfl.dualflow_profile_read(run.ctx)
        assert run.status() == 0
        assert torch.equal(run.logits, ref)
        per_layer = 5 if w.n_experts == 0 else 8  # MoE: router, routing, gate/up, down, combine
        assert sum(n) == 1 + per_layer * w.n_layers + 1
        for f, name_f in enumerate(dfl.PROF_NAMES):
            if n[f]:
                assert ms[f] > 0.0, f"{name_f}: no time recorded"
        total = sum(ms)
        print(f"[profile {name}] step {ms_step:.4f} ms, sum of in-graph shares {total:.4f} ms: "
              + ", ".join(f"{dfl.PROF_NAMES[f]} {ms[f]:.4f}" for f in range(len(ms)) if n[f]))
        assert total <= ms_step * 1.02 and total >= 0.6 * ms_step
        # the serialising mode reports the same families
        dfl.dualflow_set_profiling(run.ctx, 1)
        _timed_step(run, s)
        ms1, n1 = dfl.dualflow_profile_read(run.ctx)
        assert n1 == n and all((ms1[f] > 0.0) == (n[f] > 0) for f in range(len(n)))
        dfl.dualflow_set_profiling(run.ctx, 0)
    finally:
        run.close()
