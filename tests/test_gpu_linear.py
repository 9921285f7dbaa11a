"""dualflow_stacked_linear (tcgen05 path) against numpy float64 products of the same stored values."""
import numpy as np
import pytest
import torch

import dfsynth
import dual_flow_decode_dualflow_b300 as dfl
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu


def _bf16(seed, name, shape, sigma, dev):
    host = dfsynth.host_normal(seed, name, shape, sigma, "bf16")
    t = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).to(dev)
    return t, dfsynth.bf16_bits_to_f32(host).astype(np.float64)


def _ctx(max_batch):
    cfg = dfl.make_config(n_layers=1, d_model=2048, n_q_heads=16, n_kv_heads=4, head_dim=128, ffn_hidden=8192,
                          vocab=32000, dtype=dfl.DF_DTYPE_BF16, max_batch=max_batch, max_ctx=64)
    return dfl.dualflow_init(cfg)


@pytest.fixture(scope="module")
def ctx(cuda_device):
    """Capacity 2 x 64 rows: the split-K (cluster) path is taken where the output has few tiles."""
    h = _ctx(64)
    yield h
    dfl.dualflow_free(h)


@pytest.fixture(scope="module")
def ctx_wide(cuda_device):
    """Capacity 2 x 128 rows: too many rows for a split CTA to hold, every launch is unsplit."""
    h = _ctx(128)
    yield h
    dfl.dualflow_free(h)


# (rows, n, k) chosen so that the reduction is split 8 ways (few tiles, long k), 4, 2 and not at all,
# with ragged row counts and ragged output tiles
SHAPES = [(1, 0, 128, 64), (3, 3, 200, 128), (8, 0, 2048, 2048), (32, 32, 2048, 2048), (32, 32, 3072, 2048),
          (32, 32, 2048, 8192), (64, 64, 1000, 512), (5, 5, 32000, 2048), (17, 0, 130, 192), (32, 32, 16384, 2048),
          (24, 24, 4096, 1024), (7, 7, 1000, 4096)]


def _store_f32(cuda_device, ctx, mp, ma, n, k):
    x, xr = _bf16(11, "x", (mp + ma, k), 1.0, cuda_device)
    W, Wr = _bf16(12, "W", (n, k), 0.02, cuda_device)
    y = torch.full((mp + ma, n), float("nan"), device=cuda_device)
    dfl.dualflow_stacked_linear(ctx, x, mp, ma, W, n, k, y, dfl.DF_EPI_STORE_F32)
    assert dfl.dualflow_sync_status(ctx) == 0
    ref = xr @ Wr.T
    assert H.rel_err(H.to_f64(y), ref) < 1e-5


@pytest.mark.parametrize("mp,ma,n,k", SHAPES)
def test_store_f32(cuda_device, ctx, mp, ma, n, k):
    _store_f32(cuda_device, ctx, mp, ma, n, k)


@pytest.mark.parametrize("mp,ma,n,k", [(128, 128, 384, 256), (100, 100, 2048, 2048)])
def test_store_f32_wide(cuda_device, ctx_wide, mp, ma, n, k):
    _store_f32(cuda_device, ctx_wide, mp, ma, n, k)


def test_rows_beyond_capacity_rejected(cuda_device, ctx):
    x, _ = _bf16(13, "x", (130, 128), 1.0, cuda_device)
    W, _ = _bf16(14, "W", (128, 128), 0.02, cuda_device)
    y = torch.zeros((130, 128), device=cuda_device)
    with pytest.raises(dfl.DualFlowError) as e:
        dfl.dualflow_stacked_linear(ctx, x, 65, 65, W, 128, 128, y, dfl.DF_EPI_STORE_F32)
    assert e.value.code == dfl.DF_ERR_SHAPE


@pytest.mark.parametrize("epi", [dfl.DF_EPI_STORE_BF16, dfl.DF_EPI_ADD_F32, dfl.DF_EPI_COUPLE_ADD])
def test_epilogues(cuda_device, ctx, epi):
    mp = ma = 24
    n, k = 2048, 1024
    x, xr = _bf16(21, "x", (mp + ma, k), 1.0, cuda_device)
    W, Wr = _bf16(22, "W", (n, k), 0.02, cuda_device)
    c, cr = _bf16(23, "c", (n,), 0.1, cuda_device)
    z = xr @ Wr.T
    if epi == dfl.DF_EPI_STORE_BF16:
        y = torch.zeros((mp + ma, n), dtype=torch.bfloat16, device=cuda_device)
        dfl.dualflow_stacked_linear(ctx, x, mp, ma, W, n, k, y, epi)
        assert H.rel_err(H.to_f64(y), z) < 2 ** -8
        return
    y0 = torch.from_numpy(dfsynth.host_normal(24, "y", (mp + ma, n), 1.0, "f32")).to(cuda_device)
    y = y0.clone()
    dfl.dualflow_stacked_linear(ctx, x, mp, ma, W, n, k, y, epi, c if epi == dfl.DF_EPI_COUPLE_ADD else None)
    assert dfl.dualflow_sync_status(ctx) == 0
    if epi == dfl.DF_EPI_COUPLE_ADD:
        z[mp:] = z[mp:] + cr * z[:mp]
    ref = H.to_f64(y0) + z
    assert H.rel_err(H.to_f64(y) - H.to_f64(y0), ref - H.to_f64(y0)) < 1e-5


def test_rows_are_independent(cuda_device, ctx):
    """The primary rows' results do not depend on whether auxiliary rows are present."""
    n, k = 2048, 2048
    x, _ = _bf16(31, "x", (64, k), 1.0, cuda_device)
    W, _ = _bf16(32, "W", (n, k), 0.02, cuda_device)
    y1 = torch.zeros((64, n), device=cuda_device)
    y2 = torch.zeros((32, n), device=cuda_device)
    dfl.dualflow_stacked_linear(ctx, x, 32, 32, W, n, k, y1, dfl.DF_EPI_STORE_F32)
    dfl.dualflow_stacked_linear(ctx, x[:32].contiguous(), 32, 0, W, n, k, y2, dfl.DF_EPI_STORE_F32)
    torch.cuda.synchronize()
    assert torch.equal(y1[:32], y2)


def test_shape_errors_on_host(cuda_device, ctx):
    x, _ = _bf16(41, "x", (4, 100), 1.0, cuda_device)
    W, _ = _bf16(42, "W", (64, 100), 0.02, cuda_device)
    y = torch.zeros((4, 64), device=cuda_device)
    with pytest.raises(dfl.DualFlowError) as e:
        dfl.dualflow_stacked_linear(ctx, x, 4, 0, W, 64, 100, y, dfl.DF_EPI_STORE_F32)  # k % 64 != 0
    assert e.value.code == dfl.DF_ERR_SHAPE
