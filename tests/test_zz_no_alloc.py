"""dflash_linear_noalloc, the workspace-free form of dflash_linear for
callers that cannot allocate device memory (a host framework that owns the
device allocator, or a latency-critical loop where cudaMalloc would
synchronise the device).  Its split-K scratch is a fixed array inside the
library, shared by every call on the device.

Checked through the C ABI against dflash_linear on two calls in a row (the
second on other operands and another shape, so it runs on the scratch the
first one left behind), within the GEMM tests' tolerance, each call's error
words {0, 0}; plus the size limit.  (The error words come from the same
launch helper as dflash_linear's, whose timeout report test_gpu_linear.py
makes run out.)  This file is collected last so that a failure here comes
after every other test has run.
"""

import pytest
import torch

from tests import gpu_common as G

pytestmark = pytest.mark.gpu

TOL = 1e-5   # the dflash_linear tests' bound (rel. to max |y|)


def _operands(n, k, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    w = (torch.randn(n, k, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    x = torch.randn(16, k, device="cuda", generator=g).to(torch.bfloat16)
    x[13:] = 0
    return w, x


def _with_workspace(capi, w, x):
    n, k = w.shape
    ws = torch.zeros(capi.dflash_linear_workspace_bytes(n, k), dtype=torch.uint8, device="cuda")
    y = torch.empty((16, n), dtype=torch.float32, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    capi.dflash_linear(w, x, y, ws, err)
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0]
    return y


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    G.build_lib()
    from block_diffusion_speculative_gather_gb300 import capi
    for n, k, seed in [(19456, 2560, 1), (2560, 9728, 2)]:
        w, x = _operands(n, k, seed)
        ref = _with_workspace(capi, w, x)
        y = torch.full((16, n), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.full((2,), -1, dtype=torch.int32, device="cuda")
        capi.dflash_linear_noalloc(w, x, y, err)
        torch.cuda.synchronize()
        assert err.tolist() == [0, 0]
        rel = float((y - ref).abs().max() / ref.abs().max())
        assert rel <= TOL, (n, k, rel)
        assert torch.all(y[13:] == 0)
        # same kernel, grid and reduction order: in practice bit-identical
        assert torch.equal(y, ref), (n, k)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    G.build_lib()
    from block_diffusion_speculative_gather_gb300 import capi
    n, k = 262144 + 128, 64
    w = torch.zeros((n, k), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((16, k), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((16, n), dtype=torch.float32, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.DFlashError) as e:
        capi.dflash_linear_noalloc(w, x, y, err)
    assert e.value.code == -3          # DFLASH_ERR_ARG
    assert "262144" in str(e.value)
