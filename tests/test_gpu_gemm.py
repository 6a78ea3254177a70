"""GPU parity of the tensor-core projection GEMM (dec_gemm_bf16) against a
float64 matrix product of the same bf16 operands: tile edges, K tails, both
tile widths, with and without the low-order activation plane."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

SHAPES = [(128, 128, 64), (200, 384, 200), (512, 960, 576), (300, 2048, 256), (64, 1536, 128),
          (1000, 256, 1024), (129, 3072, 576)]


@pytest.fixture(scope="module")
def dec_mod():
    from decoder_only_forward_gb300 import build
    build.build()
    from decoder_only_forward_gb300 import dec
    return dec


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_gemm_matches_f64(dec_mod, shape, split):
    m, n, k = shape
    g = torch.Generator().manual_seed(m * 7 + n * 3 + k)
    a = torch.randn(m, k, generator=g)
    b = (0.02 * torch.randn(n, k, generator=g)).to(torch.bfloat16)
    a_hi = a.to(torch.bfloat16)
    a_lo = (a - a_hi.float()).to(torch.bfloat16) if split else None
    c = torch.full((m, n), float("nan"), device="cuda")
    dec_mod.gemm_bf16(a_hi.cuda(), None if a_lo is None else a_lo.cuda(), b.cuda(), c)
    torch.cuda.synchronize()
    av = a_hi.double() + (a_lo.double() if split else 0)
    ref = (av @ b.double().T).numpy()
    np.testing.assert_allclose(c.cpu().numpy(), ref, atol=2e-5, rtol=1e-4)
    if split:   # the pair carries the f32 activation to ~2^-16 relative
        full = (a.double() @ b.double().T).numpy()
        assert np.abs(c.cpu().numpy() - full).max() < 1e-3 * np.abs(full).max()
