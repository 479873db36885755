"""Parity at the workloads' full sizes, in the launch configuration the bench
times, on outputs the oracle can compute one by one:

* drafter alone, bf16 (5 layers, 1024 tap rows, block 16): the block's 15
  draft rows;
* INT4 drafter (16384 tap rows, window 2048, block 8): the block's 7 rows;
* 36-layer target verify of 16 rows over a 1024-position synthetic KV cache
  (adopted through dflash_adopt_kv): logits, acceptance, rollback;
* the same verify over a 16384-position cache at 1 and 16 rows: row 0 of the
  16-row verify is bit-identical to the 1-row verify (batch invariance at
  full size) and both follow the oracle.

The 36-layer verify also runs the GPU's own greedy continuation as drafts
(all 15 accepted by construction) against the oracle's forward of the same
rows: the GPU's tokens are compared with the oracle's argmaxes up to the
first row not decidable at the GPU's measured error, acceptance exactly
where that prefix covers the oracle's accepted rows.

Norm weights are drawn N(1, 0.1).  Tolerance rel 2e-2 (bf16/INT4 weights
against the fp64 oracle); ids bit-exact on every row decidable at the GPU
row's measured error, with a floor taken at DEC_TOL.
"""

import numpy as np
import pytest
import torch

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.configs import DRAFT_BF16, DRAFT_INT4, E2E_BF16
from oracle import dflash_oracle as O
from tests import gpu_common as G
from tests.oracle_inputs import ModelTensors, oracle_config, oracle_draft, oracle_target

pytestmark = pytest.mark.gpu
TOL = 2e-2
DEC_TOL = 4e-3     # the accuracy the floors are taken at (36 fp16-cache layers)
NORM_STD = 0.1


def _ext(taps, w):
    n = taps.shape[0]
    return taps.view(n, w.n_taps, w.hidden).permute(1, 0, 2).contiguous()


@pytest.mark.parametrize("w", [DRAFT_BF16, DRAFT_INT4], ids=["bf16", "int4"])
def test_drafter_full_size(w):
    G.build_lib()
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    m = ModelTensors(w, norm_std=NORM_STD)
    dec = DFlash(w, m)
    taps = synth.tap_rows(w.n_ctx, w.n_taps * w.hidden)
    dl = G.logits_buf(w.vocab)
    dec.set_logits_out(None, dl)
    dec.prefill_taps(_ext(taps, w), hc=1, first_token=4242, max_new=64)
    ids = dec.draft().cpu().numpy()
    dec.check()
    st = dec.stats()
    assert st.n == w.n_ctx and st.block_len == w.block
    gpu = dl[1:w.block].cpu().numpy()
    dec.close()
    del dec
    lo = max(0, w.n_ctx - w.window) if w.window else 0
    taps_np = np.zeros((w.n_ctx, w.n_taps * w.hidden), np.float32)
    taps_np[lo:] = taps[lo:].float().numpy()          # rows before the window are never read
    ref, _ = O.draft_forward(oracle_draft(m), m.embed.float().numpy(), oracle_config(w),
                             taps_np, 4242, w.n_ctx, w.block)
    G.check_rows(f"fullsize_drafter_{w.name}", gpu, ids[:w.block - 1], ref[1:], TOL, DEC_TOL)


@pytest.fixture(scope="module")
def target():
    G.build_lib()
    w = E2E_BF16.with_(drf_layers=0, max_seq=16384 + 64)
    m = ModelTensors(w, norm_std=NORM_STD)
    return w, m, oracle_target(m)


def _synthetic_kv(dec, w, n):
    """N(0,1) K/V at positions [0, n) of every layer, in the library's cache
    layout [L][2][n_kv][cap][hd] (fp16), and the same values for the oracle."""
    # [L, 2, n_kv, n, hd], held as fp16 (the cache type of bf16 models);
    # the oracle reads the same fp16 values
    kv = synth.kv_rows(w.tgt_layers, w.n_kv, n, w.head_dim).to(torch.float16)
    cap = (w.max_seq + 63) // 64 * 64
    dev = dec.kv_target.view(torch.float16).view(w.tgt_layers, 2, w.n_kv, cap, w.head_dim)
    dev[:, :, :, :n, :] = kv.to("cuda")
    cache = O.KVCache(w.tgt_layers, w.n_kv, w.head_dim)
    kvf = kv.float().numpy()
    for l in range(w.tgt_layers):
        cache.write(l, range(n), np.moveaxis(kvf[l, 0], 0, 1), np.moveaxis(kvf[l, 1], 0, 1))
    return cache


@pytest.mark.parametrize("n,max_seq,form", [(1024, 1600, 2), (1024, 1600, 1), (16384, 16448, 1)],
                         ids=["1k-tcgen05", "1k-mma", "16k-mma"])
def test_verify_full_size_over_synthetic_cache(target, n, max_seq, form, monkeypatch):
    """36-layer verify over an n-token cache, with the tcgen05 attention
    (opt-in; a 1600-position cache, the end-to-end workload's, gives splits
    of two chunks) and with the default mma.sync form (one chunk per split
    at 1600 positions, several at 16448)."""
    from block_diffusion_speculative_gather_gb300 import capi
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    w, m, tw = target
    w = w.with_(max_seq=max_seq)
    if form == 2:
        monkeypatch.setenv("DFLASH_ATTN_TC", "1")
    dec = DFlash(w, m)
    monkeypatch.delenv("DFLASH_ATTN_TC", raising=False)
    assert capi.dflash_attention_form(dec.ctx, 0) == form
    cache = _synthetic_kv(dec, w, n)
    t_n = 31337
    d = synth.uniform_ids(15, w.vocab, seed=5).tolist()
    vl = G.logits_buf(w.vocab)
    dec.set_logits_out(vl, None)
    dec.adopt_kv(n, t_n, 64)
    toks, ne = dec.verify(torch.tensor(d, dtype=torch.int32, device="cuda"))
    dec.check()
    batch = vl.clone()
    toks, ne = toks.cpu().tolist(), int(ne.item())
    st = dec.stats()
    dec.adopt_kv(n, t_n, 64)
    dec.verify(None)                    # one row: the plain greedy step
    dec.check()
    assert torch.equal(vl[0], batch[0]), "row 0 differs between a 16-row and a 1-row verify"
    # the GPU's greedy continuation of 16 steps, then those tokens verified
    # as drafts in one 16-row forward (all accepted: speculative == greedy)
    dec.adopt_kv(n, t_n, 64)
    gtoks = []
    for _ in range(16):
        t1, n1 = dec.verify(None)
        gtoks.extend(t1[: int(n1.item())].tolist())
    dg = gtoks[:15]
    dec.adopt_kv(n, t_n, 64)
    ctoks, cne = dec.verify(torch.tensor(dg, dtype=torch.int32, device="cuda"))
    dec.check()
    cont = vl.clone()
    ctoks, cne = ctoks.cpu().tolist(), int(cne.item())
    cst = dec.stats()
    assert cne == 16 and ctoks == gtoks[:16]
    dec.close()
    del dec
    ref, _ = O.target_forward(tw, oracle_config(w), [t_n] + d, n, cache)
    tag = f"fullsize_verify_{n}_{form}"
    G.check_rows(tag, batch[:16].cpu().numpy(), None, ref, TOL, DEC_TOL)
    G.accept_prefix_check(tag + "_random_drafts", toks, ne, st, ref, d, batch[:16].cpu().numpy(),
                          TOL, DEC_TOL, n)
    cache.truncate(n)
    ref_c, _ = O.target_forward(tw, oracle_config(w), [t_n] + dg, n, cache)
    G.check_rows(tag + "_continuation", cont[:16].cpu().numpy(), ctoks, ref_c, TOL, DEC_TOL)
    a, k = G.accept_prefix_check(tag + "_continuation_accept", ctoks, cne, cst, ref_c, dg,
                                 cont[:16].cpu().numpy(), TOL, DEC_TOL, n)
