"""Attention-only dual-flow decode (dualflow_decode_attention) against the oracle.

bf16 storage, fp32 accumulation: per-tensor max relative error <= 2e-2 against the oracle in
mirror mode (it rounds to bf16 where the GPU stores bf16). Sizes span several 64-key tiles with
ragged tails, empty sequences, equal lengths on both sides of the per-pair cut's limits, paged
caches with shuffled tables, and the two full-size attention workloads (the long ragged one on
sampled sequences, shortest and longest included).
"""
import numpy as np
import pytest
import torch

import dual_flow_decode_dualflow_b300 as dfl
from dfsynth import workloads as W
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
TOL_BF16 = 2e-2

SMALL = dict(d_model=256, n_q_heads=8, n_kv_heads=2, batch=5, ctx_len=0, ctx_lo=1, ctx_hi=300)
CASES = {
    "contig_ragged_g4": W.ATTN_B8_L2048.replace(**SMALL),
    "contig_ragged_g2": W.ATTN_B8_L2048.replace(**dict(SMALL, n_q_heads=4)),
    "contig_ragged_g1": W.ATTN_B8_L2048.replace(**dict(SMALL, n_q_heads=2)),
    "contig_with_empty": W.ATTN_B8_L2048.replace(**dict(SMALL, ctx_lo=0, ctx_hi=3, batch=7)),
    "contig_one_long": W.ATTN_B8_L2048.replace(**dict(SMALL, batch=1, ctx_lo=5000, ctx_hi=5000)),
    "paged16_ragged": W.PAGED_RAGGED_B64.replace(**dict(SMALL, ctx_hi=700, d_model=512)),
    "paged32_ragged": W.PAGED_RAGGED_B64.replace(**dict(SMALL, ctx_hi=700, page_size=32)),
    "paged64_ragged": W.PAGED_RAGGED_B64.replace(**dict(SMALL, ctx_hi=700, page_size=64, n_q_heads=4)),
    "full_b8_l2048": W.ATTN_B8_L2048,
}
# every sequence of the same length: the per-pair cut (CTAs per pair = min(grid / pairs, tiles,
# tiles / 8), the grid capped by the longest cache length), across the boundaries of that rule
for _L in (1, 64, 65, 500, 576, 1024, 1088):
    CASES[f"uniform_l{_L}"] = W.ATTN_B8_L2048.replace(**dict(SMALL, ctx_len=_L))


def _check(run, w, rows):
    ref = H.oracle_attention(w, rows=rows)
    got = H.to_f64(run.o)[:, rows]
    for f in range(2):
        err = H.rel_err(got[f], ref[f])
        assert err <= TOL_BF16, f"flow {f + 1}: rel err {err:.3e}"
    return ref


@pytest.mark.parametrize("name", list(CASES))
def test_attention_parity(cuda_device, name):
    w = CASES[name]
    run = H.DeviceRun(w, cuda_device)
    try:
        run.attention(aux_on=1)
        assert run.status() == 0
        _check(run, w, list(range(w.batch)))
        # primary outputs are bit-identical without the auxiliary flow; auxiliary rows untouched
        o_dual = run.o.clone()
        run.o.fill_(float("nan"))
        run.attention(aux_on=0)
        assert run.status() == 0
        assert torch.equal(run.o[0], o_dual[0])
        assert torch.isnan(run.o[1].float()).all()
        # repeated calls are deterministic, also chained to the preceding call on a stream
        run.attention(aux_on=1)
        assert torch.equal(run.o, o_dual)
        s = torch.cuda.Stream()
        dfl.dualflow_set_call_chaining(run.ctx, 1)
        with torch.cuda.stream(s):
            for _ in range(3):
                run.attention(aux_on=1, stream=s)
        s.synchronize()
        dfl.dualflow_set_call_chaining(run.ctx, 0)
        assert run.status() == 0
        assert torch.equal(run.o, o_dual)
    finally:
        run.close()


@pytest.mark.slow
def test_attention_full_paged_ragged_sampled(cuda_device):
    w = W.PAGED_RAGGED_B64
    lens = w.seq_lens()
    rows = sorted({int(np.argmin(lens)), int(np.argmax(lens)), 5, 37})
    run = H.DeviceRun(w, cuda_device)
    try:
        run.attention(aux_on=1)
        assert run.status() == 0
        _check(run, w, rows)
        o_dual = run.o.clone()
        run.attention(aux_on=0)
        assert torch.equal(run.o[0], o_dual[0])
    finally:
        run.close()


def test_page_permutation_invariance(cuda_device):
    """Permuting the physical pages together with the table gives a bit-identical result."""
    w = CASES["paged16_ragged"]
    run = H.DeviceRun(w, cuda_device)
    try:
        run.attention(aux_on=1)
        o1 = run.o.clone()
        P = run.t["K"].shape[0]
        perm = torch.randperm(P, generator=torch.Generator().manual_seed(3)).to(cuda_device)
        inv = torch.empty_like(perm)
        inv[perm] = torch.arange(P, device=cuda_device)
        K2, V2 = run.t["K"][perm].contiguous(), run.t["V"][perm].contiguous()  # new page i = old page perm[i]
        table2 = torch.where(run.table >= 0, inv[run.table.clamp(min=0)], run.table).to(torch.int32).contiguous()
        import dual_flow_decode_dualflow_b300 as dfl
        run.kv = dfl.make_kv([K2], [V2], run.seq_len, table2)
        run.attention(aux_on=1)
        assert run.status() == 0
        assert torch.equal(run.o, o1)
    finally:
        run.close()


def test_bad_page_id_reported_not_faulted(cuda_device):
    """An out-of-range page id is skipped and latched as DF_ERR_DEVICE_BOUNDS in the status word."""
    import dual_flow_decode_dualflow_b300 as dfl
    w = CASES["paged16_ragged"]
    run = H.DeviceRun(w, cuda_device)
    try:
        bad = run.table.clone()
        bad[0, 0] = 10 ** 6
        run.kv = dfl.make_kv([run.t["K"]], [run.t["V"]], run.seq_len, bad)
        run.attention(aux_on=1)
        assert run.status() == dfl.DF_ERR_DEVICE_BOUNDS
        assert run.status() == 0  # cleared by the read
    finally:
        run.close()
