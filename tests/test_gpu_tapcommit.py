"""GPU check of the tap commit's context K/V over several draft layers.

The tap commit projects the committed rows' context (fc, context norm) to
every draft layer's K and V.  By default (bf16 models whose drafter has more
than one layer) that is one GEMM over a copy of the layers' [W_k; W_v] made
at init, whose epilogue takes the layer from the tile index; environment
DFLASH_CTXKV_GROUP=0 at init runs one GEMM per layer instead.  The two
differ only in fp32 summation order, so after the same prefill and the same
verify (the GPU's own greedy continuation as drafts: every draft accepted,
16 rows committed) the draft cache rows of the committed positions agree to
fp16 rounding, the prefill's rows are bit-identical, and the next draft's
logits agree within a quarter of the parity tolerance; the grouped form's
next draft also matches the oracle's drafter over the same context (the
oracle target's taps of all P + 16 positions), so a tap commit that writes
wrong context rows fails here even though speculative decoding, which
verifies every draft, would stay lossless.

Shapes: a Qwen3-4B-shaped layer (head_dim 128: one head per 128-row tile,
16 tiles per layer), a head_dim-64 model (two heads per tile) and an INT4
drafter (codes copied by rows, their bf16 scales by columns), a 32-key
drafter window that the commit slides; the many-sequence round (which
reuses the first context's copy) at S = 2.
"""

import pytest
import torch

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.configs import E2E_BF16, Workload
from oracle import dflash_oracle as O
from tests import gpu_common as G
from tests.oracle_inputs import ModelTensors, oracle_config, oracle_draft, oracle_target

pytestmark = pytest.mark.gpu
TOL = 2e-2
DEC_TOL = {"hd128": 1e-3, "hd64": 1e-3, "int4-drafter": 2e-3, "hd128-window": 1e-3}   # as in the bf16 / INT4 parity modules

QWEN = E2E_BF16.with_(name="tc_qwen", tgt_layers=2, drf_layers=3, tap_layers=(0, 1), prompt_len=40,
                      n_new=48, max_seq=256)
CASES = {
    "hd128": QWEN,
    "hd64": Workload(name="tc_hd64", hidden=512, n_q=8, n_kv=4, head_dim=64, ffn=1536, vocab=4096,
                     tgt_layers=2, drf_layers=3, tap_layers=(0, 1), block=16, window=0, dtype="bf16",
                     prompt_len=200, n_new=40, max_seq=512),
    "int4-drafter": QWEN.with_(name="tc_int4", drf_int4=True),
    # a 32-key drafter window: the next draft sees prefill rows 24..39 and
    # the committed rows 40..55
    "hd128-window": QWEN.with_(name="tc_window", window=32),
}


def _model(W):
    return ModelTensors(W, std=0.02 if W.hidden > 1024 else 0.05, norm_std=0.1)


def _close_rows(a, b):
    """Largest difference of two cache blocks relative to each row's largest magnitude."""
    scale = b.abs().amax(dim=-1, keepdim=True).clamp_min(1e-6)
    return ((a - b).abs() / scale).max().item()


@pytest.mark.parametrize("case", list(CASES))
def test_grouped_tap_commit_matches_per_layer(case, monkeypatch):
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    G.build_lib()
    W = CASES[case]
    m = _model(W)
    P, B = W.prompt_len, W.block
    prompt = torch.from_numpy(synth.uniform_ids(P, W.vocab, seed=5))
    cap = (W.max_seq + 63) // 64 * 64
    out = []
    for env in (None, "0"):
        if env is not None:
            monkeypatch.setenv("DFLASH_CTXKV_GROUP", env)
        dec = DFlash(W, m)
        monkeypatch.delenv("DFLASH_CTXKV_GROUP", raising=False)
        gg = dec.greedy(prompt, B + 1)               # the GPU's own greedy continuation
        dec.prefill(prompt, W.n_new)
        toks, n = dec.verify(torch.tensor(gg[1:B], dtype=torch.int32, device="cuda"))
        dec.check()
        assert int(n.item()) == B, "every draft of the greedy continuation is accepted"
        assert toks.cpu().tolist() == gg[1:B + 1]
        kd = dec.kv_draft.view(torch.float16).view(W.drf_layers, 2, W.n_kv, cap, W.head_dim)
        dl = G.logits_buf(W.vocab)
        dec.set_logits_out(None, dl)
        ids = dec.draft().cpu().numpy()
        dec.check()
        out.append((kd[:, :, :, :P + B].float().clone(), dl[1:B].clone(), ids[:B - 1].copy()))
        dec.close()
    (kd_g, dl_g, ids_g), (kd_p, dl_p, _) = out
    assert torch.equal(kd_g[:, :, :, :P], kd_p[:, :, :, :P]), "the prefill's context rows take one path"
    committed = kd_p[:, :, :, P:P + B]
    assert committed.abs().amax(dim=-1).min().item() > 0, "every committed row of every layer is written"
    assert _close_rows(kd_g[:, :, :, P:P + B], committed) < 2.0 ** -8
    err = G.rel_err_rows(dl_g.cpu().numpy(), dl_p.cpu().numpy())
    assert err.max() < TOL / 4, err
    # the oracle's drafter over the context the commit built: the target's
    # taps of the prompt and the 16 verified rows, the pending token gg[B]
    tw, dw, cfg = oracle_target(m), oracle_draft(m), oracle_config(W)
    _, taps = O.target_forward(tw, cfg, prompt.tolist() + gg[:B], 0,
                               O.KVCache(W.tgt_layers, W.n_kv, W.head_dim))
    ref, _ = O.draft_forward(dw, tw.embed, cfg, taps, gg[B], P + B, B)
    G.check_rows(f"tap_commit_{case}", dl_g.cpu().numpy(), ids_g, ref[1:], TOL, DEC_TOL[case])


def test_grouped_tap_commit_many_sequences(monkeypatch):
    """The many-sequence round's tap commit (one dense GEMM over the first
    context's copy and one cache-row launch for every layer) against its
    per-layer form, two sequences of different prompt lengths, and each
    sequence's next draft against the oracle's drafter over its context."""
    from block_diffusion_speculative_gather_gb300.runtime import DFlashBatch
    G.build_lib()
    W = QWEN
    m = _model(W)
    B = W.block
    lens = (40, 29)
    prompts = [torch.from_numpy(synth.uniform_ids(L, W.vocab, seed=31 + i)) for i, L in enumerate(lens)]
    cap = (W.max_seq + 63) // 64 * 64
    out = []
    for env in (None, "0"):
        if env is not None:
            monkeypatch.setenv("DFLASH_CTXKV_GROUP", env)
        dec = DFlashBatch(W, m, S=2)
        monkeypatch.delenv("DFLASH_CTXKV_GROUP", raising=False)
        gg = dec.greedy(prompts, B + 1)
        dec.prefill(prompts, W.n_new)
        drafts = torch.tensor([g[1:B] for g in gg], dtype=torch.int32, device="cuda")
        toks, n = dec.verify(drafts)
        dec.check()
        assert n.cpu().tolist() == [B, B]
        kd = dec.kv_draft.view(torch.float16).view(2, W.drf_layers, 2, W.n_kv, cap, W.head_dim)
        dl = torch.zeros((2 * 16, W.vocab), dtype=torch.float32, device="cuda")
        dec.set_logits_out(None, dl)
        ids = dec.draft().cpu().numpy()
        dec.check()
        out.append(([kd[s, :, :, :, :lens[s] + B].float().clone() for s in range(2)], dl.clone(), ids.copy(),
                    gg))
        dec.close()
    (kd_g, dl_g, ids_g, gg), (kd_p, dl_p, _, _) = out
    tw, dw, cfg = oracle_target(m), oracle_draft(m), oracle_config(W)
    for s, L in enumerate(lens):
        assert torch.equal(kd_g[s][..., :L, :], kd_p[s][..., :L, :])
        committed = kd_p[s][..., L:L + B, :]
        assert committed.abs().amax(dim=-1).min().item() > 0
        assert _close_rows(kd_g[s][..., L:L + B, :], committed) < 2.0 ** -8
        rows = slice(16 * s + 1, 16 * s + B)
        err = G.rel_err_rows(dl_g[rows].cpu().numpy(), dl_p[rows].cpu().numpy())
        assert err.max() < TOL / 4, (s, err)
        _, taps = O.target_forward(tw, cfg, prompts[s].tolist() + gg[s][:B], 0,
                                   O.KVCache(W.tgt_layers, W.n_kv, W.head_dim))
        ref, _ = O.draft_forward(dw, tw.embed, cfg, taps, gg[s][B], L + B, B)
        G.check_rows(f"tap_commit_batch_{s}", dl_g[rows].cpu().numpy(), ids_g[s][:B - 1], ref[1:], TOL,
                     DEC_TOL["hd128"])
