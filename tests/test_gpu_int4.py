"""GPU parity of the INT4 group-64 drafter (the long-context drafter
workload's format) on one Qwen3-4B-shaped layer: the library quantises the
fp32 draws with its own kernel, the oracle with its own code (the two are
bit-identical, see test_quantizer_bit_exact_with_oracle), and the drafter
fed 300 external tap rows with a 64-row sliding window must give logits
within rel 2e-2 of the oracle's dequantised fp64 drafter.  Norm weights are
drawn N(1, 0.1); ids are checked on every row decidable at the GPU row's
measured error, with a floor taken at DEC_TOL (see tests/gpu_common.py):
2e-3 here, because GEMMs with INT4 weights take their activations as one
f16 plane (11 mantissa bits; bf16 weights take hi/lo bf16 planes, ~16)."""

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
DEC_TOL = 2e-3
NORM_STD = 0.1
W = DRAFT_INT4.with_(name="int4_1layer", drf_layers=1, n_ctx=300, window=64, max_seq=400)


@pytest.mark.parametrize("window,n_ext", [(64, 300), (0, 40)])
def test_int4_drafter_matches_oracle(window, n_ext):
    G.build_lib()
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    w = W.with_(window=window)
    m = ModelTensors(w, norm_std=NORM_STD)
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
    G.check_rows(f"int4_drafter_w{window}", dl[1:w.block].cpu().numpy(), ids[:w.block - 1],
                 ref[1:], TOL, DEC_TOL)
    dec.close()


# ---------------------------------------------------------------- 4-bit target

def _w4():
    from block_diffusion_speculative_gather_gb300.configs import E2E_BF16
    return E2E_BF16.with_(name="int4_target_2layer", tgt_layers=2, drf_layers=1, tap_layers=(0, 1),
                          prompt_len=40, n_new=40, max_seq=256, tgt_int4=True, lm_int4=True,
                          drf_int4=True)


@pytest.fixture(scope="module")
def int4_target():
    G.build_lib()
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    from tests.oracle_inputs import oracle_target
    w = _w4()
    m = ModelTensors(w, norm_std=NORM_STD)
    tw, cfg = oracle_target(m), oracle_config(w)
    prompt = synth.uniform_ids(w.prompt_len, w.vocab)
    g = O.greedy(tw, cfg, prompt.tolist(), w.n_new)
    tf, _ = O.target_forward(tw, cfg, prompt.tolist() + g[:-1], 0,
                             O.KVCache(w.tgt_layers, w.n_kv, w.head_dim))
    return dict(w=w, m=m, tw=tw, dw=oracle_draft(m), cfg=cfg, prompt=torch.from_numpy(prompt),
                greedy=g, greedy_logits=tf[len(prompt) - 1:], dec=DFlash(w, m))


@pytest.mark.parametrize("cut", [0, 7, None], ids=["cut0", "cut7", "all"])
def test_int4_target_and_lm_head_verify_match_oracle(int4_target, cut):
    """Target layers and the LM head in INT4 group-64 (both models 4-bit):
    a 16-row verify of the oracle's greedy continuation cut at draft 0, 7 or
    not at all -- logits within rel 2e-2 of the oracle's dequantised fp64
    target, acceptance, emitted tokens and rollback exact (asserted)."""
    T = int4_target
    w, dec, tw, cfg = T["w"], T["dec"], T["tw"], T["cfg"]
    P, B = w.prompt_len, w.block
    dec.prefill(T["prompt"], w.n_new)
    t_n = dec.stats().t_n
    assert t_n == T["greedy"][0]
    d = list(T["greedy"][1:B])
    if cut is not None:
        d[cut] = (d[cut] + 1) % w.vocab
    vl = G.logits_buf(w.vocab)
    dec.set_logits_out(vl, None)
    toks, n = dec.verify(torch.tensor(d, dtype=torch.int32, device="cuda"))
    dec.check()
    dec.set_logits_out(None, None)
    cache = O.KVCache(2, w.n_kv, w.head_dim)
    O.target_forward(tw, cfg, T["prompt"].tolist(), 0, cache)
    ref, _ = O.target_forward(tw, cfg, [t_n] + d, P, cache)
    gpu = vl[:B].cpu().numpy()
    G.check_rows(f"int4_verify_{cut}", gpu, None, ref, TOL, DEC_TOL)
    a = G.accept_check(f"int4_accept_{cut}", toks.cpu().tolist(), int(n.item()), dec.stats(),
                       ref, d, gpu, TOL, P)
    assert a == (B - 1 if cut is None else cut)


def test_int4_greedy_stream_matches_oracle(int4_target):
    """Plain greedy decoding of the INT4 target + INT4 LM head against the
    oracle's greedy stream (dequantised fp64 weights), compared while
    decidable at each step's measured error."""
    T = int4_target
    w, dec = T["w"], T["dec"]
    P = w.prompt_len
    vl = G.logits_buf(w.vocab)
    dec.set_logits_out(vl, None)
    dec.prefill(T["prompt"], w.n_new)
    rows = [vl[(P - 1) % 16].clone()]
    st = dec.stats()
    toks = [st.t_n]
    while not st.finished and len(toks) < w.n_new:
        t, n = dec.verify(None)
        toks.extend(t[: int(n.item())].tolist())
        rows.append(vl[0].clone())
        st = dec.stats()
    dec.check()
    dec.set_logits_out(None, None)
    gl = T["greedy_logits"]
    floor = next((i for i, r in enumerate(gl) if not G.decidable(r, DEC_TOL)), len(gl))
    n = G.stream_prefix("int4_greedy_stream", toks, [r.cpu().numpy() for r in rows],
                        T["greedy"], gl, TOL)
    assert n >= floor and n > 0, (n, floor)


def test_int4_target_draft_uses_int4_lm_head(int4_target):
    """The drafter's logits come from the same INT4 LM head."""
    T = int4_target
    w, dec = T["w"], T["dec"]
    dec.prefill(T["prompt"], w.n_new)
    dl = G.logits_buf(w.vocab)
    dec.set_logits_out(None, dl)
    ids = dec.draft().cpu().numpy()
    dec.check()
    dec.set_logits_out(None, None)
    t_n = dec.stats().t_n
    cache = O.KVCache(2, w.n_kv, w.head_dim)
    _, p_taps = O.target_forward(T["tw"], T["cfg"], T["prompt"].tolist(), 0, cache)
    ref, _ = O.draft_forward(T["dw"], T["tw"].embed, T["cfg"], p_taps, t_n, w.prompt_len, w.block,
                             lm_head=T["tw"].lm_head)
    G.check_rows("int4_target_draft", dl[1:w.block].cpu().numpy(), ids[:w.block - 1], ref[1:],
                 TOL, DEC_TOL)


def test_int4_target_spec_equals_greedy_and_batch_invariant(int4_target):
    T = int4_target
    w, dec = T["w"], T["dec"]
    gg = dec.greedy(T["prompt"], w.n_new)
    sp = dec.generate(T["prompt"], w.n_new)
    dec.check()
    assert sp == gg
    P, B = w.prompt_len, w.block
    dec.prefill(T["prompt"], w.n_new)
    vl = G.logits_buf(w.vocab)
    dec.set_logits_out(vl, None)
    dec.verify(torch.tensor(gg[1:B], dtype=torch.int32, device="cuda"))
    batch = vl[:B].clone()
    dec.rollback(P, gg[0])
    for i in range(B):
        dec.verify(None)
        assert torch.equal(vl[0], batch[i]), f"row {i}"
    dec.set_logits_out(None, None)
    dec.close()


def test_int4_target_dense_prefill_matches_chunked_and_oracle(int4_target, monkeypatch):
    """The dense prefill of an INT4 target (f16 rows times each layer's
    matrices dequantised exactly to f16) against the 16-row forwards
    (DFLASH_DENSE_PREFILL=0) on a 300-token prompt: target and draft cache
    rows to fp16 rounding, the last chunk's logits within the tolerance of
    each other and of the oracle's dequantised fp64 target."""
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    T = int4_target
    w = T["w"].with_(max_seq=512)
    P = 300
    prompt = torch.from_numpy(synth.uniform_ids(P, w.vocab, seed=23))
    cap = (w.max_seq + 63) // 64 * 64
    out = []
    for env in (None, "0"):
        if env is not None:
            monkeypatch.setenv("DFLASH_DENSE_PREFILL", env)
        dec = DFlash(w, T["m"])
        monkeypatch.delenv("DFLASH_DENSE_PREFILL", raising=False)
        vl = G.logits_buf(w.vocab)
        dec.set_logits_out(vl, None)
        dec.prefill(prompt, 8)
        dec.check()
        kt = dec.kv_target.view(torch.float16).view(w.tgt_layers, 2, w.n_kv, cap, w.head_dim)
        kd = dec.kv_draft.view(torch.float16).view(w.drf_layers, 2, w.n_kv, cap, w.head_dim)
        out.append((kt[:, :, :, :P].float().clone(), kd[:, :, :, :P].float().clone(), vl[:P % 16 or 16].clone()))
        dec.close()
    (kt_d, kd_d, lg_d), (kt_c, kd_c, lg_c) = out
    for a, b in ((kt_d, kt_c), (kd_d, kd_c)):
        scale = b.abs().amax(dim=-1, keepdim=True).clamp_min(1e-6)
        assert ((a - b).abs() / scale).max().item() < 2.0 ** -8
    err = G.rel_err_rows(lg_d.cpu().numpy(), lg_c.cpu().numpy())
    assert err.max() < TOL / 4, err
    ref, _ = O.target_forward(T["tw"], T["cfg"], prompt.tolist(), 0, O.KVCache(2, w.n_kv, w.head_dim))
    last = (P - 1) // 16 * 16
    G.check_rows("int4_dense_prefill", lg_d.cpu().numpy(), None, ref[last:P], TOL, DEC_TOL)
