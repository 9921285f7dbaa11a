"""The C-ABI library without a GPU: it loads, exports every declared symbol, and rejects bad
configurations on the host before touching the device."""
import ctypes
import os
import re

import pytest

import dual_flow_decode_dualflow_b300 as dfl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dualflow.h")


def declared_functions():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"DF_API\s+(?:const\s+)?\w+\*?\s+(dualflow_\w+)\s*\(", txt)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("dualflow_init", "dualflow_decode_attention", "dualflow_stacked_linear", "dualflow_coupled_mlp",
              "dualflow_step", "dualflow_free"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = dfl.load_library()
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(dfl.C_FUNCTIONS) >= set(declared_functions())


def test_status_strings():
    for code in range(9):
        s = dfl.dualflow_status_string(code)
        assert s and s != "unknown status"
    assert dfl.dualflow_status_string(99) == "unknown status"


def _good(**kw):
    base = dict(n_layers=2, d_model=256, n_q_heads=4, n_kv_heads=1, head_dim=128, ffn_hidden=512, vocab=1000,
                dtype=dfl.DF_DTYPE_BF16, max_batch=4, max_ctx=256)
    base.update(kw)
    return dfl.make_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), dfl.DF_ERR_DTYPE),
    (dict(d_model=0), dfl.DF_ERR_ARG),
    (dict(max_batch=-1), dfl.DF_ERR_ARG),
    (dict(n_q_heads=6, n_kv_heads=4), dfl.DF_ERR_SHAPE),
    (dict(head_dim=64), dfl.DF_ERR_UNSUPPORTED),
    (dict(n_q_heads=16, n_kv_heads=1), dfl.DF_ERR_UNSUPPORTED),
    (dict(d_model=200), dfl.DF_ERR_UNSUPPORTED),
    (dict(max_batch=200), dfl.DF_ERR_UNSUPPORTED),
    (dict(paged=1, page_size=16, max_pages=0), dfl.DF_ERR_ARG),
    (dict(paged=1, page_size=8, max_pages=10), dfl.DF_ERR_UNSUPPORTED),
    (dict(n_experts=4, topk_primary=5, topk_aux=1), dfl.DF_ERR_SHAPE),
    (dict(rms_eps=-1.0), dfl.DF_ERR_ARG),
])
def test_init_rejects_bad_config_on_host(kw, code):
    rc, h = dfl.dualflow_init_status(_good(**kw))
    assert rc == code and h is None


def test_null_arguments_rejected():
    lib = dfl.load_library()
    assert lib.dualflow_init(None, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_free(None) == dfl.DF_OK
    assert lib.dualflow_step(None, None, None, None, 1, None, 1, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_decode_attention(None, None, None, None, None, None, 0, 1, None, 1, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_stacked_linear(None, None, 1, 0, None, 1, 64, None, 0, None, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_coupled_mlp(None, None, None, 0, 1, 1, None, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_set_graphs(None, 1) == dfl.DF_ERR_ARG
    assert lib.dualflow_sync_status(None, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_mixture_head(None, None, 1, None, None, None, None, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_generate(None, None, None, None, 1, 1, None, None, None, None, None, None, 1,
                                 None) == dfl.DF_ERR_ARG
    assert lib.dualflow_prefill_reserve(None, 16) == dfl.DF_ERR_ARG
    assert lib.dualflow_prefill(None, None, None, None, 1, 1, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_prefill_slots(None, None, None, None, None, 1, 1, None, None, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_release_slots(None, None, None, 1, None, None, None) == dfl.DF_ERR_ARG
    assert lib.dualflow_set_nvtx(None, 1) == dfl.DF_ERR_ARG
    assert lib.dualflow_set_call_chaining(None, 1) == dfl.DF_ERR_ARG
    assert lib.dualflow_set_wait_limit(None, 0) == dfl.DF_ERR_ARG
    assert lib.dualflow_router_logits(None, None, 1, None) == dfl.DF_ERR_ARG


def test_noalloc_limit_constant_matches_header():
    m = re.search(r"#define\s+DF_NOALLOC_MAX_PAIRS\s+(\d+)", open(HEADER).read())
    assert m and int(m.group(1)) == dfl.DF_NOALLOC_MAX_PAIRS


@pytest.mark.parametrize("batch,kv_heads,code", [
    (65, 8, dfl.DF_ERR_SHAPE),    # 520 pairs: above the static array's limit of 512
    (513, 1, dfl.DF_ERR_SHAPE),   # 513 pairs
    (5, 4, dfl.DF_ERR_SHAPE),     # batch above cfg.max_batch
    (0, 4, dfl.DF_ERR_SHAPE),
])
def test_noalloc_rejects_sizes_on_host(batch, kv_heads, code):
    """The allocation-free attention rejects a batch beyond its static scratch (or the config)
    before touching the device: the pointers below are never dereferenced."""
    lib = dfl.load_library()
    cfg = _good(n_q_heads=2 * kv_heads, n_kv_heads=kv_heads, max_batch=max(batch, 1) if batch != 5 else 4)
    fake = ctypes.c_void_p(0x1000)  # 16-byte aligned, never read
    kv = dfl.dualflow_kv()
    arr = (ctypes.c_void_p * 1)(0x2000)
    kv.k = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    kv.v = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    kv.seq_len = 0x3000
    kv.n_layers = 1
    rc = lib.dualflow_decode_attention_noalloc(ctypes.byref(cfg), fake, ctypes.byref(kv), 0, batch, fake, 1, None, None)
    assert rc == code
