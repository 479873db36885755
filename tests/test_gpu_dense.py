"""The dense tcgen05 GEMM (dflash_linear_dense) against the plain definition
y = x w^T computed in fp64 on the CPU from the same bf16 values, at the
shapes of the drafter's context-window ingest (fc over the window's tap
rows: K = 5 x 2560; context K/V: N = 2 x 1024) and at ragged M and N
(partial 128-row and 256-column tiles), with and without a low plane of x.

Bound: fp32 accumulation of K products, |y - y_ref| <= K * 2^-23 * sum_i
|x_i w_i| (plus the hi/lo sum), per element."""

import numpy as np
import pytest
import torch

from tests import gpu_common as G

pytestmark = pytest.mark.gpu

CASES = [
    (1, 4, 64, False),          # one row, one column group
    (100, 200, 64, False),      # ragged M and N inside one tile
    (128, 256, 128, False),     # exactly one tile
    (300, 1000, 2560, True),    # ragged over several tiles, hi + lo planes
    (1024, 2560, 12800, False),  # fc over a 1024-row window (5 taps x 2560)
    (1024, 2048, 2560, True),   # context K/V of one draft layer (hi + lo input)
]


@pytest.mark.parametrize("m,n,k,split", CASES)
def test_dense_matches_fp64_definition(m, n, k, split):
    G.build_lib()
    from block_diffusion_speculative_gather_gb300 import capi
    g = torch.Generator(device="cuda").manual_seed(m * 7 + n * 3 + k)
    w = (torch.randn(n, k, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    xf = torch.randn(m, k, device="cuda", generator=g)
    x = xf.to(torch.bfloat16)
    x_lo = (xf - x.float()).to(torch.bfloat16) if split else None
    y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    capi.dflash_linear_dense(w, x, y, err, x_lo=x_lo)
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0]
    wd = w.double().cpu().numpy()
    xd = x.double().cpu().numpy()
    ref = xd @ wd.T
    mag = np.abs(xd) @ np.abs(wd).T
    if split:
        xl = x_lo.double().cpu().numpy()
        ref += xl @ wd.T
        mag += np.abs(xl) @ np.abs(wd).T
    got = y.double().cpu().numpy()
    assert np.isfinite(got).all()
    bound = k * 2.0 ** -23 * mag * (2 if split else 1) + 1e-30
    assert (np.abs(got - ref) <= bound).all(), float(np.max(np.abs(got - ref) / bound))


def test_dense_rejects_bad_shapes():
    G.build_lib()
    from block_diffusion_speculative_gather_gb300 import capi
    w = torch.zeros(8, 96, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(4, 96, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(4, 8, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.DFlashError):
        capi.dflash_linear_dense(w, x, y, err)          # k = 96 is not a multiple of 64
