"""The standalone weight-streaming GEMM (dflash_linear) against a plain
PyTorch fp32 reference of the same op on the same bf16 inputs, at the
shapes of the round (q/k/v, o, fused gate/up, down, LM head) and at a
single tile; plus the row independence the round's batch invariance rests
on."""

import pytest
import torch

from tests import gpu_common as G

pytestmark = pytest.mark.gpu

SHAPES = [(128, 64), (384, 320), (6144, 2560), (2560, 4096), (19456, 2560), (2560, 9728),
          (151936, 2560)]


def _run(capi, w, x):
    n, k = w.shape
    ws = torch.zeros(capi.dflash_linear_workspace_bytes(n, k), dtype=torch.uint8, device="cuda")
    y = torch.empty((16, n), dtype=torch.float32, device="cuda")
    capi.dflash_linear(w, x, y, ws)
    torch.cuda.synchronize()
    # the tickets (after the 4 MiB of partial tiles) are back at zero
    tickets = ws[4 << 20:(4 << 20) + (n // 128) * 4]
    assert int(tickets.count_nonzero()) == 0
    return y, ws


@pytest.mark.parametrize("n,k", SHAPES)
def test_linear_matches_torch_fp32(n, k):
    G.build_lib()
    from block_diffusion_speculative_gather_gb300 import capi
    g = torch.Generator(device="cuda").manual_seed(n + k)
    w = (torch.randn(n, k, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(16, k, device="cuda", generator=g).to(torch.bfloat16)
    x[11:] = 0
    y, _ = _run(capi, w, x)
    ref = x.float() @ w.float().T
    err = (y - ref).abs().max() / ref.abs().max()
    assert err < 1e-5, float(err)
    assert torch.all(y[11:] == 0)


def test_linear_rows_are_independent():
    G.build_lib()
    from block_diffusion_speculative_gather_gb300 import capi
    g = torch.Generator(device="cuda").manual_seed(7)
    w = (torch.randn(2560, 9728, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(16, 9728, device="cuda", generator=g).to(torch.bfloat16)
    y1, ws = _run(capi, w, x)
    x2 = x.clone()
    x2[1:] = torch.randn(15, 9728, device="cuda", generator=g).to(torch.bfloat16)
    y2 = torch.empty_like(y1)
    capi.dflash_linear(w, x2, y2, ws)
    torch.cuda.synchronize()
    assert torch.equal(y1[0], y2[0])
    x3 = torch.zeros_like(x)
    x3[0] = x[0]
    y3 = torch.empty_like(y1)
    capi.dflash_linear(w, x3, y3, ws)
    torch.cuda.synchronize()
    assert torch.equal(y1[0], y3[0])
