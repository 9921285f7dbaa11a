"""The seeded input generator: determinism, slicing, distribution and format conversions."""
import numpy as np

import dfsynth
from dfsynth import workloads as W


def test_slices_reproduce_whole():
    full = dfsynth.host_normal(7, "t", (1000,), 0.5, "bf16")
    part = dfsynth.host_normal(7, "t", (300,), 0.5, "bf16", offset=400)
    assert np.array_equal(full[400:700], part)
    assert not np.array_equal(full, dfsynth.host_normal(8, "t", (1000,), 0.5, "bf16"))
    assert not np.array_equal(full, dfsynth.host_normal(7, "u", (1000,), 0.5, "bf16"))


def test_normal_moments_and_range():
    x = dfsynth.host_normal(1, "m", (2_000_000,), 1.0, "f32").astype(np.float64)
    assert abs(x.mean()) < 3e-3 and abs(x.std() - 1.0) < 3e-3
    assert np.abs(x).max() <= 6.0  # Irwin-Hall of 12 uniforms is bounded by 6
    # n is an integer: every f32 value times 65536 is integral
    assert np.all(np.mod(x * 65536.0, 1.0) == 0.0)


def test_bf16_is_rounded_f32():
    f = dfsynth.host_normal(3, "r", (10000,), 0.02, "f32")
    b = dfsynth.host_normal(3, "r", (10000,), 0.02, "bf16")
    assert np.array_equal(dfsynth.f32_to_bf16_bits(f), b)
    assert np.max(np.abs(dfsynth.bf16_bits_to_f32(b) - f) / np.abs(f).max()) < 2 ** -8


def test_uniform_int_and_permutation():
    t = dfsynth.host_uniform_int(5, "tok", 100000, 0, 31999)
    assert t.min() >= 0 and t.max() <= 31999 and len(np.unique(t)) > 30000
    p = dfsynth.host_permutation(5, "perm", 5000)
    assert np.array_equal(np.sort(p), np.arange(5000)) and not np.array_equal(p, np.arange(5000))


def test_workload_page_table():
    w = W.PAGED_RAGGED_B64.replace(batch=6, ctx_lo=3, ctx_hi=70, page_size=16)
    lens = w.seq_lens()
    table, total = w.page_table()
    used = table[table >= 0]
    assert np.array_equal(np.sort(used), np.arange(total))
    for b in range(w.batch):
        n = (lens[b] + 15) // 16
        assert np.all(table[b, :n] >= 0) and np.all(table[b, n:] == -1)


def test_workload_sizes():
    w = W.DENSE_24L_B32_L4096
    per_layer = sum(s.numel for s in W.layer_specs(w, 0) if s.name[-1] not in "KV")
    assert per_layer == 2048 * (3072 + 2048 + 16384 + 8192) + 2048 * 3 + 2048 + 8192  # 60.8 M
    assert w.max_ctx == 4160 and w.cache_shape() == (32, 4, 4160, 128)
