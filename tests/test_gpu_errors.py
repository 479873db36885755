"""Failure handling on the GPU without faulting it: calls out of order,
capacity overflow, a bad token id (the kernel records the device error word
and skips it), and the kernels' bounded wait running out (a barrier that
nothing arrives on), each reported as a status while the context stays
usable."""

import pytest
import torch

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.configs import TINY
from tests import gpu_common as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dec():
    G.build_lib()
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    d = DFlash(TINY, synth.ModelTensors(TINY, std=0.1))
    yield d
    d.close()


def _code(exc):
    return exc.value.code


def test_calls_before_prefill_are_state_errors():
    from block_diffusion_speculative_gather_gb300 import capi
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    d = DFlash(TINY, synth.ModelTensors(TINY, std=0.1))
    with pytest.raises(capi.DFlashError) as e:
        d.draft()
    assert _code(e) == -7
    with pytest.raises(capi.DFlashError) as e:
        d.verify(None)
    assert _code(e) == -7
    d.close()


def test_prompt_beyond_capacity(dec):
    from block_diffusion_speculative_gather_gb300 import capi
    long = torch.zeros(TINY.max_seq, dtype=torch.int32)
    with pytest.raises(capi.DFlashError) as e:
        dec.prefill(long, 8)
    assert _code(e) == -2


def test_bad_draft_token_sets_device_error_and_recovers(dec):
    from block_diffusion_speculative_gather_gb300 import capi
    prompt = torch.from_numpy(synth.uniform_ids(TINY.prompt_len, TINY.vocab))
    dec.prefill(prompt, 16)
    bad = torch.full((TINY.block - 1,), TINY.vocab + 5, dtype=torch.int32, device="cuda")
    dec.verify(bad)
    with pytest.raises(capi.DFlashError) as e:
        dec.check()
    assert _code(e) == -5
    dec.check()                       # the flag was cleared by the report
    g = dec.greedy(prompt, 8)         # and the context still works
    assert len(g) == 8


def test_bounded_wait_times_out_and_context_survives(dec):
    from block_diffusion_speculative_gather_gb300 import capi
    capi.dflash_selftest_timeout(dec.ctx, 20_000_000, dec.stream)   # 20 ms
    with pytest.raises(capi.DFlashError) as e:
        dec.check()
    assert _code(e) == -6
    dec.check()
    prompt = torch.from_numpy(synth.uniform_ids(TINY.prompt_len, TINY.vocab))
    assert dec.generate(prompt, 12) == dec.greedy(prompt, 12)
