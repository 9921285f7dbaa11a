"""The oracle against its pins, and deliberately broken oracles against the same pins.

Every pin must pass on the real oracle. Each mutant plants one plausible mistake in a copy
of the oracle's source (on the CPU, never in the GPU path) and must fail at least one pin.
"""
import os
import sys
import types

import pytest

import oracle.dualflow_oracle as O
from tests import oracle_pins

SRC = open(os.path.join(os.path.dirname(O.__file__), "dualflow_oracle.py")).read()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(O)


MUTANTS = {
    "rope_sign": ("lo * cos - hi * sin", "lo * cos + hi * sin"),
    "rope_freq": ("theta = base ** (-2.0 * np.arange(half, dtype=F64) / D)",
                  "theta = base ** (-2.0 * np.arange(half, dtype=F64) / half)"),
    "key_not_rotated": ("k_new = _store(rope(k1, pos, hp.rope_base), hp, mirror)", "k_new = _store(k1, hp, mirror)"),
    "no_attention_scale": ("s = (q @ K.T) / np.sqrt(F64(D))", "s = (q @ K.T)"),
    "gqa_modulo": ("attention(q[f][h][None, :], Kc[g], Vc[g])",
                   "attention(q[f][h][None, :], Kc[h % hp.n_kv_heads], Vc[h % hp.n_kv_heads])"),
    "new_entry_not_attended": ("    if append:", "    if False:"),
    "q_coupling_wrong_source": ('q2 = Wq @ x[1] + P["a"] * q1', 'q2 = Wq @ x[1] + P["a"] * (Wq @ x[1])'),
    "q_coupling_after_rope": ('q2 = Wq @ x[1] + P["a"] * q1  # query coupling, before RoPE (R1)\n'
                              '        q.append(rope(q2.reshape(Hq, D), pos, hp.rope_base))',
                              'q2 = Wq @ x[1]\n        q.append(rope(q2.reshape(Hq, D), pos, hp.rope_base) + '
                              'P["a"].reshape(Hq, D) * q[0])'),
    "b_dropped": ('u.append(silu(Wg @ x[1]) * (Wu @ x[1]) + P["b"] * u[0])', 'u.append(silu(Wg @ x[1]) * (Wu @ x[1]))'),
    "c_wrong_source": ('y[1] = y[1] + P["c"] * y[0]', 'y[1] = y[1] + P["c"] * y[1]'),
    "silu_is_sigmoid": ("return z / (1.0 + np.exp(-z))", "return 1.0 / (1.0 + np.exp(-z))"),
    "rmsnorm_wrong_axis": ("np.mean(h * h, axis=-1, keepdims=True)", "np.mean(h * h, axis=0, keepdims=True)"),
    "rmsnorm_no_sqrt": ("return 1.0 / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)",
                        "return 1.0 / (np.mean(h * h, axis=-1, keepdims=True) + eps)"),
    "mirror_norm_unscaled": ("return round_bf16(h * g) * rms_scale(h, hp.rms_eps)", "return round_bf16(h * g)"),
    "mirror_norm_no_gain": ("return round_bf16(h * g) * rms_scale(h, hp.rms_eps)",
                            "return round_bf16(h) * rms_scale(h, hp.rms_eps)"),
    "primary_uses_E2": ('h[0, i] = glob["E1"][tokens[b]]', 'h[0, i] = glob["E2"][tokens[b]]'),
    "no_router_replay": ("S2 = topk_lower_index(r1, hp.topk_aux)", "S2 = topk_lower_index(r2, hp.topk_aux)"),
    "aux_weights_from_primary": ("    w2 = softmax(r2[S2])\n    return", "    w2 = softmax(r1[S2])\n    return"),
    "moe_b_dropped": ('u2 = u2 + P["b"] * u1[int(e)]', "u2 = u2"),
    "topk_ties_high": ("key=lambda i: (-r[i], i)", "key=lambda i: (-r[i], -i)"),
    "round_truncates": ("np.round(np.ldexp(m, 8))", "np.trunc(np.ldexp(m, 8))"),
    "alpha_from_aux": ("alpha = 0.5 + 0.5 * float(np.sum(p1 * p1))", "alpha = 0.5 + 0.5 * float(np.sum(p2 * p2))"),
    "o_proj_dropped": ('h[f, i] = h[f, i] + P["Wo"] @ o[f]', "h[f, i] = h[f, i]"),
    "paged_wrong_page": ("ks = [np.asarray(self.K[int(self.table[b, j])], dtype=F64) for j in range(n)]",
                         "ks = [np.asarray(self.K[int(self.table[b, n - 1 - j])], dtype=F64) for j in range(n)]"),
    "final_norm_dropped": ('xf = _normed(h[f, i], glob["g_final"], hp, mirror)', "xf = h[f, i]"),
    "sample_at_or_above": ("np.cumsum(p) > u", "np.cumsum(p) >= u"),
    "sample_fallback_first": ("return int(np.nonzero(p > 0)[0][-1])", "return int(np.nonzero(p > 0)[0][0])"),
    "mix_weights_swapped": ("pm = alpha * p1 + (1.0 - alpha) * p2", "pm = alpha * p2 + (1.0 - alpha) * p1"),
    "generate_no_append": ('append_entry(caches[layer], b, int(L[b]), r["k_new"][layer, b], r["v_new"][layer, b])',
                           "pass"),
    "generate_no_increment": ("        L = L + 1\n        tokens = out_tok[t].copy()", "        tokens = out_tok[t].copy()"),
    "prefill_no_append": ('                append_entry(caches[layer], b, int(L[b]), r["k_new"][layer, b], r["v_new"][layer, b])\n        L = L + 1\n    return dict(logits=logits',
                          '                pass\n        L = L + 1\n    return dict(logits=logits'),
    "generate_primary_choice": ("    if logits2 is None:\n        p = softmax", "    if True:\n        p = softmax"),
    "paged_append_wrong_slot": ("cache.K[pid][:, L % cache.page_size, :] = k",
                                "cache.K[pid][:, (L + 1) % cache.page_size, :] = k"),
    "paged_append_first_page": ("pid = int(cache.table[b, L // cache.page_size])", "pid = int(cache.table[b, 0])"),
}


def _mutant(name, old, new):
    assert SRC.count(old) >= 1, f"mutant {name}: pattern not found in the oracle source"
    src = SRC.replace(old, new, 1)
    modname = f"_oracle_mutant_{name}"
    mod = types.ModuleType(modname)
    mod.__file__ = f"<{modname}>"
    sys.modules[modname] = mod
    exec(compile(src, modname, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    mod = _mutant(name, *MUTANTS[name])
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passes every pin"
