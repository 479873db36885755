"""The standalone weight-streaming GEMM (dflash_linear) against a plain
PyTorch fp32 reference of the same op on the same bf16 inputs, at the
shapes of the round (q/k/v, o, fused gate/up, down, LM head) and at a
single tile; plus the row independence the round's batch invariance rests
on, and the error words a call reports when one of its bounded waits runs
out."""

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
    err = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    capi.dflash_linear(w, x, y, ws, err)
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0]
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
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    capi.dflash_linear(w, x2, y2, ws, err)
    torch.cuda.synchronize()
    assert torch.equal(y1[0], y2[0])
    x3 = torch.zeros_like(x)
    x3[0] = x[0]
    y3 = torch.empty_like(y1)
    capi.dflash_linear(w, x3, y3, ws, err)
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0]
    assert torch.equal(y1[0], y3[0])


def test_linear_reports_a_wait_that_ran_out():
    """A split tile's owner waits (bounded, 2 s) for the other CTAs' parts to
    be counted on the tile's ticket.  A workspace whose ticket starts far
    below zero (the caller skipped the zero-fill) never reaches the count:
    the wait runs out, the kernel skips that tile's epilogue and returns, and
    the call's err words read {1, 105} (timeout, the split-K owner's wait) --
    no fault, the context stays usable, and the next call on a zero-filled
    workspace is correct with err {0, 0}."""
    G.build_lib()
    from block_diffusion_speculative_gather_gb300 import capi
    g = torch.Generator(device="cuda").manual_seed(11)
    n, k = 128, 9728                # one tile, 152 k-blocks: split over every SM
    w = (torch.randn(n, k, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(16, k, device="cuda", generator=g).to(torch.bfloat16)
    ws = torch.zeros(capi.dflash_linear_workspace_bytes(n, k), dtype=torch.uint8, device="cuda")
    ws[4 << 20:(4 << 20) + 4].view(torch.int32).fill_(-(1 << 30))
    y = torch.zeros((16, n), dtype=torch.float32, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    capi.dflash_linear(w, x, y, ws, err)
    torch.cuda.synchronize()
    assert err.tolist() == [1, 105]
    y2, _ = _run(capi, w, x)
    ref = x.float() @ w.float().T
    assert float((y2 - ref).abs().max() / ref.abs().max()) < 1e-5
