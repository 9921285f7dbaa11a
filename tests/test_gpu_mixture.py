"""dualflow_mixture_head (mixture of both flows' next-token distributions and the token choice)
against the oracle's fp64 mixture head and inverse-transform sampling.

The GPU computes in fp32: alpha and p_mix are compared at the fp32 bar (1e-5 of the largest
value). Tokens are integers decided by floating point: where the oracle's decision has a margin
above that bar (a top-2 gap for the argmax, a distance from every cumulative boundary for a
sample) the GPU token must equal the oracle's; otherwise it must be one of the tokens the bar
admits (a value within the bar of the maximum; a token whose cumulative interval reaches u within
the bar)."""
import numpy as np
import pytest
import torch

import dfsynth
import dual_flow_decode_dualflow_b300 as dfl
import oracle as O

pytestmark = pytest.mark.gpu
TOL = 1e-5


def _ctx(vocab, max_batch):
    cfg = dfl.make_config(n_layers=1, d_model=256, n_q_heads=4, n_kv_heads=4, head_dim=64, ffn_hidden=1024,
                          vocab=vocab, dtype=dfl.DF_DTYPE_F32, max_batch=max_batch, max_ctx=16)
    return dfl.dualflow_init(cfg)


def _logits(seed, B, V, sigma):
    return dfsynth.host_normal(seed, "mix_logits", (2, B, V), sigma, "f32")


def _uniforms(seed, B):
    # multiples of 2^-24: exact in fp32 and fp64
    return (dfsynth.host_uniform_int(seed, "mix_u", B, 0, 1 << 24) / float(1 << 24)).astype(np.float32)


def _run(dev, V, lg, u=None):
    B = lg.shape[1]
    ctx = _ctx(V, max(B, 1))
    try:
        d_lg = torch.from_numpy(lg.copy()).to(dev)
        alpha = torch.full((B,), float("nan"), device=dev)
        pm = torch.full((B, V), float("nan"), device=dev)
        tok = torch.full((B,), -7, dtype=torch.int32, device=dev)
        d_u = torch.from_numpy(u).to(dev) if u is not None else None
        dfl.dualflow_mixture_head(ctx, d_lg, B, d_u, alpha, pm, tok)
        torch.cuda.synchronize()
        return alpha.cpu().numpy().astype(np.float64), pm.cpu().numpy().astype(np.float64), tok.cpu().numpy()
    finally:
        dfl.dualflow_free(ctx)


def _check_greedy(pm_ref, tok):
    mx = pm_ref.max()
    srt = np.sort(pm_ref)
    if srt[-1] - srt[-2] > TOL * mx:
        assert tok == int(np.argmax(pm_ref)), (tok, int(np.argmax(pm_ref)))
        return 1
    assert pm_ref[tok] >= mx - TOL * mx
    return 0


def _check_sample(pm_ref, u, tok):
    """tok's cumulative interval [C_{tok-1}, C_tok) holds u within the bar; exact where u is far
    from every boundary."""
    C = np.cumsum(pm_ref)
    lo = C[tok - 1] if tok > 0 else 0.0
    assert lo <= u + TOL and C[tok] >= u - TOL, (tok, lo, C[tok], u)
    assert pm_ref[tok] > 0
    if np.min(np.abs(C - u)) > TOL and u < C[-1] - TOL:
        assert tok == O.sample_inverse_cdf(pm_ref, float(u))
        return 1
    return 0


@pytest.mark.parametrize("V,B,sigma", [(1000, 5, 3.0), (12345, 7, 2.0), (32000, 32, 3.0), (32000, 3, 12.0),
                                       (4097, 1, 1.0)])
def test_mixture_head_parity(cuda_device, V, B, sigma):
    lg = _logits(61 + V % 7, B, V, sigma)
    u = _uniforms(62, B)
    alpha, pm, tok = _run(cuda_device, V, lg)
    _, pm_s, tok_s = _run(cuda_device, V, lg, u)
    exact = 0
    for b in range(B):
        a_ref, pm_ref, _ = O.mixture_head(lg[0, b].astype(np.float64), lg[1, b].astype(np.float64))
        assert abs(alpha[b] - a_ref) <= TOL * a_ref, (b, alpha[b], a_ref)
        assert np.max(np.abs(pm[b] - pm_ref)) <= TOL * np.max(pm_ref), b
        assert np.array_equal(pm[b], pm_s[b])
        exact += _check_greedy(pm_ref, int(tok[b]))
        exact += _check_sample(pm_ref, float(u[b]), int(tok_s[b]))
    assert exact > 0


def test_mixture_head_special_cases(cuda_device):
    V, B = 5000, 4
    lg = np.zeros((2, B, V), np.float32)
    lg[1] = _logits(63, B, V, 1.0)[1]
    lg[0, 1, 4321] = 200.0          # confident primary: alpha = 1, p_mix = one-hot
    lg[0, 2] = lg[1, 2]             # identical flows: p_mix = p1
    lg[:, 3] = 0.0                  # both uniform: alpha = 1/2 + 1/(2V), p_mix uniform
    alpha, pm, tok = _run(cuda_device, V, lg)
    assert abs(alpha[0] - (0.5 + 0.5 / V)) <= 1e-6
    assert abs(alpha[1] - 1.0) <= 1e-6 and tok[1] == 4321 and abs(pm[1, 4321] - 1.0) <= 1e-6
    _, p1, _ = O.mixture_head(lg[0, 2].astype(np.float64), lg[0, 2].astype(np.float64))
    assert np.max(np.abs(pm[2] - p1)) <= TOL * p1.max()
    assert np.max(np.abs(pm[3] - 1.0 / V)) <= TOL / V and tok[3] == 0  # all equal: the lowest index
    # sampling: u = 0 takes the first token with mass; u just below 1 the last
    u = np.array([0.0, 0.5, 0.0, 1.0 - 2.0 ** -24], np.float32)
    _, _, ts = _run(cuda_device, V, lg, u)
    assert ts[0] == 0 and ts[1] == 4321 and ts[2] == 0 and ts[3] >= V - 2


def test_mixture_head_deterministic_and_capturable(cuda_device):
    V, B = 32000, 8
    lg = torch.from_numpy(_logits(64, B, V, 3.0).copy()).to(cuda_device)
    u = torch.from_numpy(_uniforms(65, B)).to(cuda_device)
    ctx = _ctx(V, B)
    try:
        outs = []
        for _ in range(2):
            a = torch.empty(B, device=cuda_device)
            p = torch.empty(B, V, device=cuda_device)
            t = torch.empty(B, dtype=torch.int32, device=cuda_device)
            dfl.dualflow_mixture_head(ctx, lg, B, u, a, p, t)
            outs.append((a, p, t))
        torch.cuda.synchronize()
        for x, y in zip(*outs):
            assert torch.equal(x, y)
        # captured into a CUDA graph and replayed: the same outputs
        s = torch.cuda.Stream()
        a = torch.empty(B, device=cuda_device)
        p = torch.empty(B, V, device=cuda_device)
        t = torch.empty(B, dtype=torch.int32, device=cuda_device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                dfl.dualflow_mixture_head(ctx, lg, B, u, a, p, t, s)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(a, outs[0][0]) and torch.equal(p, outs[0][1]) and torch.equal(t, outs[0][2])
        # outputs are optional
        dfl.dualflow_mixture_head(ctx, lg, B)
        torch.cuda.synchronize()
    finally:
        dfl.dualflow_free(ctx)


def test_mixture_head_rejects_bad_arguments(cuda_device):
    ctx = _ctx(1000, 4)
    try:
        lg = torch.zeros(2, 4, 1000, device=cuda_device)
        with pytest.raises(dfl.DualFlowError):
            dfl.dualflow_mixture_head(ctx, lg, 5)
        with pytest.raises(dfl.DualFlowError):
            dfl.dualflow_mixture_head(ctx, None, 4)
    finally:
        dfl.dualflow_free(ctx)
