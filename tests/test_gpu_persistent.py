"""The persistent round schedule (one cooperative launch per forward, phases
separated by grid barriers; selected with DFLASH_PERSISTENT=1 at init)
against the default per-launch schedule, on the Qwen3-4B-shaped bf16
2-layer workload of test_gpu_bf16.py.

Both schedules run the same device functions; the split of a small GEMM
across CTAs may differ, so logits are compared at rel 1e-4 and ids on rows
whose top-2 margin exceeds that.  On the persistent schedule: speculative
== greedy bit-exactly and a 16-row verify reproduces 1-row verifies
bit-for-bit (batch invariance).
"""

import os

import numpy as np
import pytest
import torch

from block_diffusion_speculative_gather_gb300 import synth
from tests import gpu_common as G
from tests.oracle_inputs import ModelTensors
from tests.test_gpu_bf16 import W

pytestmark = pytest.mark.gpu
TOL = 1e-4


def _make(m, persistent):
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    old = os.environ.get("DFLASH_PERSISTENT")
    os.environ["DFLASH_PERSISTENT"] = "1" if persistent else "0"
    try:
        return DFlash(W, m)
    finally:
        if old is None:
            del os.environ["DFLASH_PERSISTENT"]
        else:
            os.environ["DFLASH_PERSISTENT"] = old


@pytest.fixture(scope="module")
def pair():
    G.build_lib()
    m = ModelTensors(W, std=0.02, norm_std=0.1)
    prompt = torch.from_numpy(synth.uniform_ids(W.prompt_len, W.vocab))
    return dict(m=m, prompt=prompt, ref=_make(m, False), per=_make(m, True))


def _draft(dec, prompt):
    dec.prefill(prompt, W.n_new)
    dl = G.logits_buf(W.vocab)
    dec.set_logits_out(None, dl)
    ids = dec.draft().cpu().numpy()
    dec.check()
    dec.set_logits_out(None, None)
    return ids, dl.cpu().numpy()


def test_persistent_draft_matches_per_launch(pair):
    ids_r, lg_r = _draft(pair["ref"], pair["prompt"])
    ids_p, lg_p = _draft(pair["per"], pair["prompt"])
    rows = slice(1, W.block)
    err = G.rel_err_rows(lg_p[rows], lg_r[rows])
    assert err.max() < TOL, err
    G.check_ids(ids_p[:W.block - 1], lg_r[rows].astype(np.float64), TOL)


def test_persistent_verify_matches_per_launch(pair):
    d = synth.uniform_ids(W.block - 1, W.vocab, seed=11).tolist()
    out = []
    for key in ("ref", "per"):
        dec = pair[key]
        dec.prefill(pair["prompt"], W.n_new)
        vl = G.logits_buf(W.vocab)
        dec.set_logits_out(vl, None)
        toks, n = dec.verify(torch.tensor(d, dtype=torch.int32, device="cuda"))
        dec.check()
        dec.set_logits_out(None, None)
        st = dec.stats()
        out.append((vl.cpu().numpy(), toks.cpu().tolist(), int(n.item()), st.n, st.last_accept))
    (lr, tr, nr, pr, ar), (lp, tp, np_, pp, ap) = out
    err = G.rel_err_rows(lp, lr)
    assert err.max() < TOL, err
    if all(G.decidable(r.astype(np.float64), TOL) for r in lr[: ar + 1]):
        assert (tp[:np_], np_, pp, ap) == (tr[:nr], nr, pr, ar)


def test_persistent_spec_equals_greedy(pair):
    dec = pair["per"]
    gg = dec.greedy(pair["prompt"], W.n_new)
    sp = dec.generate(pair["prompt"], W.n_new)
    dec.check()
    assert sp == gg


def test_persistent_batch_invariance(pair):
    dec, P, B = pair["per"], W.prompt_len, W.block
    gg = dec.greedy(pair["prompt"], W.n_new)
    dec.prefill(pair["prompt"], W.n_new)
    vl = G.logits_buf(W.vocab)
    dec.set_logits_out(vl, None)
    dec.verify(torch.tensor(gg[1:B], dtype=torch.int32, device="cuda"))
    batch = vl[:B].clone()
    dec.rollback(P, gg[0])
    for i in range(B):
        dec.verify(None)
        assert torch.equal(vl[0], batch[i]), f"row {i}"
    dec.set_logits_out(None, None)
    dec.check()
