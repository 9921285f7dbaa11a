"""The benchmark's algorithmic byte and FLOP counts (the roofline numerators) against the same
quantities written out by hand from the model shapes, and against the survey's figures for the
pages' configurations (config 2: 42.07 MB per attention-only call; config 3: 9.493 GB per step,
60.8 M parameters per layer)."""
import numpy as np
import pytest

import bench
from dfsynth import workloads as W


def test_dense_step_bytes_by_hand():
    w = W.DENSE_24L_B32_L4096
    d, Hq, Hkv, D, F, V, nL, B, ctx = 2048, 16, 4, 128, 8192, 32000, 24, 32, 4096
    assert (w.d_model, w.n_q_heads, w.n_kv_heads, w.head_dim, w.ffn_hidden, w.vocab, w.n_layers, w.batch) == \
        (d, Hq, Hkv, D, F, V, nL, B)
    per_layer = (Hq + 2 * Hkv) * D * d + d * Hq * D + 2 * F * d + d * F  # Wqkv, Wo, Wgu, Wd
    per_layer += 2 * d + Hq * D + F + d                                 # g_attn, g_mlp, a, b, c
    assert abs(per_layer / 1e6 - 60.8) < 0.05
    weights = 2 * (nL * per_layer + V * d + d)                          # + LM head and final gain
    kv_pos = Hkv * D * 2 * 2                                            # K and V, bf16
    total = weights + B * ctx * kv_pos * nL + B * kv_pos * nL + 2 * B * d * 2 + 2 * B * V * 4
    got = bench.step_bytes(w)
    assert got["weights"] == weights
    assert got["kv_read"] == B * ctx * kv_pos * nL
    assert got["total"] == total
    assert abs(total / 1e9 - 9.493) / 9.493 < 2e-3
    # one attention launch: positions 0..4096 of every (sequence, KV head), q in, o out
    assert got["attention_per_launch"] == B * (ctx + 1) * kv_pos + 2 * (2 * B * Hq * D * 2)


def test_moe_step_bytes_count_only_touched_experts():
    w = W.MOE_16L_B64
    full = bench.step_bytes(w)["weights"]
    half = bench.step_bytes(w, experts_touched=[w.n_experts // 2] * w.n_layers)["weights"]
    expert = (2 * w.ffn_hidden * w.d_model + w.d_model * w.ffn_hidden) * 2  # one expert's gate/up + down, bf16
    assert full - half == w.n_layers * (w.n_experts // 2) * expert


def test_attention_call_bytes_config2():
    w = W.ATTN_B8_L2048
    got = bench.call_bytes(w)
    B, L, Hkv, D, Hq, d = 8, 2048, 4, 128, 16, 2048
    assert got["kv_read"] == B * L * Hkv * D * 2 * 2
    assert got["weights"] == Hq * D * d * 2
    assert abs(got["total"] / 1e6 - 42.07) < 0.01


@pytest.mark.parametrize("name", ["prefill", "prefill_moe"])
def test_prefill_flops_by_hand(name):
    w = bench.workload(name)
    n = 512
    rows = w.batch * n
    d, Hq, Hkv, D = w.d_model, w.n_q_heads, w.n_kv_heads, w.head_dim
    macs = (Hq + 2 * Hkv) * D * d + d * Hq * D
    if w.n_experts:
        macs += w.n_experts * d + w.topk_primary * 3 * w.ffn_hidden * d  # router + the chosen experts
    else:
        macs += 3 * w.ffn_hidden * d
    # causal: position t attends t + 1 keys; QK^T and PV are 2 D MACs per head per pair
    pairs = w.batch * sum(t + 1 for t in range(n))
    flops = w.n_layers * (2 * macs * rows + 2 * 2 * D * Hq * pairs)
    assert bench.prefill_flops(w, n) == pytest.approx(flops, rel=1e-12)
    if name == "prefill":
        assert abs(flops / 1e12 - 48.66) < 0.01


def test_replicas_single_process():
    reps = bench.Replicas()
    assert reps.max(3.0, 1.5) == [3.0, 1.5]
    assert reps.rate(32, 0.002) == pytest.approx(16000.0)
    reps.barrier()  # a no-op without a process group


def test_step_percentiles_nearest_rank():
    t = list(range(1, 51))  # 1 .. 50 ms, shuffled below
    import random
    random.Random(3).shuffle(t)
    got = bench.step_percentiles(t)
    assert got == {"n": 50, "p10_ms": 5.0, "p50_ms": 25.0, "p90_ms": 45.0}
    assert bench.step_percentiles([7.0]) == {"n": 1, "p10_ms": 7.0, "p50_ms": 7.0, "p90_ms": 7.0}


def test_dense_family_bytes_by_hand():
    """Each kernel family's roofline numerator: its weights once, its activations in and out once,
    and for attention the KV of every layer; the weights of the families add up to the step's."""
    w = W.DENSE_24L_B32_L4096
    d, Hq, Hkv, D, F, V, nL, B = 2048, 16, 4, 128, 8192, 32000, 24, 32
    M, es = 2 * B, 2
    fb = bench.family_bytes(w)
    assert fb["qkv"] == nL * ((Hq + 2 * Hkv) * D * d * es + M * d * es + M * Hq * D * es + B * 2 * Hkv * D * es)
    assert fb["o_proj"] == nL * (d * Hq * D * es + M * Hq * D * es + 2 * M * d * 4 + M * d * es)
    assert fb["gate_up"] == nL * (2 * F * d * es + M * d * es + M * F * es)
    assert fb["down"] == nL * (d * F * es + M * F * es + 2 * M * d * 4 + M * d * es)
    assert fb["lm_head"] == V * d * es + M * d * es + M * V * 4
    assert fb["attention"] == nL * bench.step_bytes(w)["attention_per_launch"]
    weights = nL * ((Hq + 2 * Hkv) * D * d + d * Hq * D + 2 * F * d + d * F) * es + V * d * es
    activations = (nL * (M * d * es + M * Hq * D * es + B * 2 * Hkv * D * es)
                   + nL * (M * Hq * D * es + 2 * M * d * 4 + M * d * es) + nL * (M * d * es + M * F * es)
                   + nL * (M * F * es + 2 * M * d * 4 + M * d * es) + M * d * es + M * V * 4)
    assert sum(fb[k] for k in ("qkv", "o_proj", "gate_up", "down", "lm_head")) == weights + activations
    # weights read per step by the families = the step's weight bytes except gains and coupling vectors
    small = nL * (2 * d + Hq * D + F + d) * es + d * es
    assert bench.step_bytes(w)["weights"] == weights + small


def test_moe_family_bytes_count_touched_experts():
    w = W.MOE_16L_B64
    full = bench.family_bytes(w)
    half = bench.family_bytes(w, experts_touched=[w.n_experts // 2] * w.n_layers)
    F, d = w.ffn_hidden, w.d_model
    assert full["gate_up"] - half["gate_up"] == w.n_layers * (w.n_experts // 2) * 2 * F * d * 2
    assert full["down"] - half["down"] == w.n_layers * (w.n_experts // 2) * d * F * 2


def test_host_cpu_reports_cores():
    cpu = bench.host_cpu()
    assert cpu["cores"] >= 1 and isinstance(cpu["model"], str)
    with bench.OracleThreads() as th:
        assert 1 <= th.threads <= max(cpu["cores"], 1)
