"""The generator's device fill writes exactly the bits of its host fill."""
import numpy as np
import pytest
import torch

import dfsynth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,n,offset,sigma", [("bf16", 100_003, 0, 0.02), ("bf16", 5000, 123_456, 1.0),
                                                  ("f32", 70_001, 7, 0.1)])
def test_device_fill_matches_host(cuda_device, dtype, n, offset, sigma):
    t = torch.empty(n, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device=cuda_device)
    dfsynth.cuda_normal_(t.data_ptr(), 77, "fill", n, sigma, dtype, offset=offset)
    host = dfsynth.host_normal(77, "fill", (n,), sigma, dtype, offset=offset)
    got = t.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else got.numpy()
    assert np.array_equal(got, host)
