"""GPU parity of the INT4 group-64 drafter (the long-context drafter
workload's format) on one Qwen3-4B-shaped layer: the library quantises the
fp32 draws with its own kernel, the oracle with its own code (the two are
bit-identical, see test_quantizer_bit_exact_with_oracle), and the drafter
fed 300 external tap rows with a 64-row sliding window must give logits
within rel 2e-2 of the oracle's dequantised fp64 drafter."""

import numpy as np
import pytest
import torch

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.configs import DRAFT_INT4
from oracle import dflash_oracle as O
from tests import gpu_common as G
from tests.oracle_inputs import ModelTensors, oracle_config, oracle_draft

pytestmark = pytest.mark.gpu
TOL = 2e-2
W = DRAFT_INT4.with_(name="int4_1layer", drf_layers=1, n_ctx=300, window=64, max_seq=400)


@pytest.mark.parametrize("window,n_ext", [(64, 300), (0, 40)])
def test_int4_drafter_matches_oracle(window, n_ext):
    G.build_lib()
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    w = W.with_(window=window)
    m = ModelTensors(w)
    dec = DFlash(w, m)
    taps = synth.tap_rows(n_ext, w.n_taps * w.hidden)
    ext = taps.view(n_ext, w.n_taps, w.hidden).permute(1, 0, 2).contiguous()
    dl = G.logits_buf(w.vocab)
    dec.set_logits_out(None, dl)
    dec.prefill_taps(ext, hc=1, first_token=777, max_new=64)
    ids = dec.draft().cpu().numpy()
    dec.check()
    ref, _ = O.draft_forward(oracle_draft(m), m.embed.float().numpy(), oracle_config(w),
                             taps.float().numpy(), 777, n_ext, w.block)
    err = G.rel_err_rows(dl[1:w.block].cpu().numpy(), ref[1:])
    assert err.max() < TOL, err
    G.check_ids(ids[:w.block - 1], ref[1:], TOL)
    dec.close()
