"""dualflow_coupled_mlp (the MLP block of one layer, in place on the fp32 residual) against the
oracle's dense MLP with the shared pre-MLP RMSNorm and the couplings b (intermediate) and c
(output), bf16 storage: per-tensor relative error of the residual update <= 2e-2; the primary rows
are bit-identical with and without the auxiliary flow."""
import numpy as np
import pytest
import torch

import dfsynth
import dual_flow_decode_dualflow_b300 as dfl
import oracle as O
from dfsynth import workloads as W
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu

CASES = {
    "small_b3": W.DENSE_24L_B32_L4096.replace(n_layers=1, d_model=256, n_q_heads=4, n_kv_heads=1, ffn_hidden=512,
                                              vocab=64, batch=3, ctx_len=8, gain_sigma=0.1),
    "d2048_f8192_b32": W.DENSE_24L_B32_L4096.replace(n_layers=1, vocab=64, ctx_len=8, gain_sigma=0.1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_coupled_mlp_parity(cuda_device, name):
    w = CASES[name]
    run = H.DeviceRun(w, cuda_device)
    try:
        B, d = w.batch, w.d_model
        h0 = dfsynth.host_normal(77, "mlp_h", (2, B, d), 1.0, "f32")
        h = torch.from_numpy(h0.copy()).to(cuda_device)
        dfl.dualflow_coupled_mlp(run.ctx, h, run.weights, 0, B, 1)
        assert run.status() == 0
        got = H.to_f64(h) - h0.astype(np.float64)
        hp = H.hparams(w)
        P = H.LazyLayers(w)[0]
        for b in range(B):
            x = [O.dualflow_oracle._normed(h0[f, b].astype(np.float64), P["g_mlp"], hp, True) for f in range(2)]
            y = O.dualflow_oracle._dense_mlp(hp, P, x, True, True)
            for f in range(2):
                err = H.rel_err(got[f, b], y[f])
                assert err <= 2e-2, f"row {b}, flow {f + 1}: rel err {err:.3e}"
        dual = h.clone()
        h1 = torch.from_numpy(h0.copy()).to(cuda_device)
        dfl.dualflow_coupled_mlp(run.ctx, h1, run.weights, 0, B, 0)
        assert run.status() == 0
        assert torch.equal(h1[0], dual[0]), "primary rows depend on the auxiliary flow"
        assert torch.equal(h1[1], torch.from_numpy(h0[1]).to(cuda_device)), "auxiliary rows written with aux_on=0"
    finally:
        run.close()
