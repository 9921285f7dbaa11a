"""dualflow_decode_attention_noalloc: the decode attention for callers that may not allocate device
memory (their own pool owns it all, or cudaMalloc's device-wide synchronisation is not allowed on
their path), so cannot create a context. Its scratch lives in a static device array of the library.

Each case calls the allocation-free entry point twice in a row, through the C ABI, on both flows'
queries as the oracle forms them (q2 = Wq.h2 + a (*) q1, both rotated to position seq_len[b] and
rounded to bf16), and compares both outputs with the oracle's attention at the bf16 tolerance of the
other attention tests, and with the context entry point's output on the same workload. One case fills
the array's limit (batch * n_kv_heads = 512 pairs). The file sorts last so that a stop at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import dual_flow_decode_dualflow_b300 as dfl
import oracle as O
from dfsynth import workloads as W
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
TOL_BF16 = 2e-2

SMALL = dict(d_model=256, n_q_heads=8, n_kv_heads=2, batch=6, ctx_len=0, ctx_lo=0, ctx_hi=300)
CASES = {
    "contiguous_ragged": W.ATTN_B8_L2048.replace(**SMALL),
    "paged16_ragged": W.PAGED_RAGGED_B64.replace(**dict(SMALL, ctx_lo=1, ctx_hi=700, d_model=512)),
    # the limit of the static array: 64 sequences x 8 KV heads = 512 (sequence, KV head) pairs
    "paged16_512_pairs": W.PAGED_RAGGED_B64.replace(**dict(ctx_lo=1, ctx_hi=200)),
}


def _rotated_queries(w, dev) -> torch.Tensor:
    """Both flows' queries at their positions, rounded to bf16: [2, B, Hq, D]."""
    q1 = H.host_f64(w, "q1")
    h2, Wq, a = H.host_f64(w, "h2"), H.host_f64(w, "Wq"), H.host_f64(w, "a")
    lens = w.seq_lens()
    q = np.empty((2, w.batch, w.n_q_heads, w.head_dim))
    for b in range(w.batch):
        q2 = Wq @ h2[b] + a * q1[b].reshape(-1)
        q[0, b] = O.rope(q1[b], int(lens[b]), w.rope_base)
        q[1, b] = O.rope(q2.reshape(w.n_q_heads, w.head_dim), int(lens[b]), w.rope_base)
    return torch.from_numpy(O.round_bf16(q).astype(np.float32)).to(torch.bfloat16).to(dev)


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_oracle(cuda_device, name):
    w = CASES[name]
    assert w.batch * w.n_kv_heads <= dfl.DF_NOALLOC_MAX_PAIRS
    run = H.DeviceRun(w, cuda_device)
    try:
        ref = H.oracle_attention(w)  # [2, B, Hq, D], mirrored bf16 storage points
        run.attention(aux_on=1)
        assert run.status() == 0
        ctx_out = H.to_f64(run.o)
        q = _rotated_queries(w, cuda_device)
        cfg = H.config_for(w)
        status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        for call in range(2):
            o = torch.full_like(run.o, float("nan"))
            dfl.dualflow_decode_attention_noalloc(cfg, q, run.kv, 0, w.batch, o, 1, status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
            got = H.to_f64(o)
            for f in range(2):
                err = H.rel_err(got[f], ref[f])
                assert err <= TOL_BF16, f"call {call}, flow {f + 1}: rel err {err:.3e} vs the oracle"
                err = H.rel_err(got[f], ctx_out[f])
                assert err <= TOL_BF16, f"call {call}, flow {f + 1}: rel err {err:.3e} vs the context entry point"
    finally:
        run.close()
