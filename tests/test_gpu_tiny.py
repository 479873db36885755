"""GPU parity on the tiny fp32 workload (2-layer target, 1-layer drafter,
block 8, window 64, 32-token prompt, 64 tokens), through the C ABI.

Tolerance: logits within rel 1e-4 of the fp64 oracle (per row, max abs
difference over max |oracle|); token ids bit-exact wherever the oracle's
top-2 margin exceeds twice that; GPU speculative output bit-identical to GPU
plain greedy; acceptance lengths and rollback positions exact.  Norm
weights are drawn N(1, 0.1); ids are checked on every row decidable at the
GPU row's measured error, with a floor taken at DEC_TOL (tests/gpu_common.py).
"""

import numpy as np
import pytest
import torch

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.configs import TINY
from oracle import dflash_oracle as O
from tests import gpu_common as G
from tests.oracle_inputs import ModelTensors, oracle_config, oracle_draft, oracle_target

pytestmark = pytest.mark.gpu
TOL = 1e-4
DEC_TOL = 1e-5


@pytest.fixture(scope="module", params=[0.02, 0.1], ids=["std0.02", "std0.1"])
def tiny(request):
    G.build_lib()
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    m = ModelTensors(TINY, std=request.param, norm_std=0.1)
    tw, dw, cfg = oracle_target(m), oracle_draft(m), oracle_config(TINY)
    prompt = synth.uniform_ids(TINY.prompt_len, TINY.vocab)
    cache = O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim)
    p_logits, p_taps = O.target_forward(tw, cfg, prompt.tolist(), 0, cache)
    g = O.greedy(tw, cfg, prompt.tolist(), TINY.n_new)
    # teacher-forced logits of every greedy step (row k predicts token k)
    tf, _ = O.target_forward(tw, cfg, prompt.tolist() + g[:-1], 0,
                             O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim))
    dec = DFlash(TINY, m)
    return dict(m=m, tw=tw, dw=dw, cfg=cfg, prompt=torch.from_numpy(prompt), p_logits=p_logits,
                p_taps=p_taps, greedy=g, greedy_logits=tf[len(prompt) - 1:], dec=dec)


def test_prefill_logits_and_first_token(tiny):
    dec = tiny["dec"]
    vl = G.logits_buf(TINY.vocab)
    dec.set_logits_out(vl, None)
    dec.prefill(tiny["prompt"], TINY.n_new)
    dec.check()
    dec.set_logits_out(None, None)
    st = dec.stats()
    P = TINY.prompt_len
    last_chunk = (P - 1) // 16 * 16
    rows = P - last_chunk
    dec_rows = G.check_rows("tiny_prefill", vl[:rows].cpu().numpy(), None,
                            tiny["p_logits"][last_chunk:P], TOL, DEC_TOL)
    assert st.n == P and st.generated == 1 and st.ctx_len == P
    assert st.block_len == TINY.block
    assert dec_rows[-1], "the last prompt row is not decidable"
    assert st.t_n == int(np.argmax(tiny["p_logits"][P - 1]))


def test_draft_matches_uncached_oracle(tiny):
    """GPU drafter (persistent draft KV cache) vs the oracle drafter that
    re-projects the context window from the raw taps."""
    dec, P = tiny["dec"], TINY.prompt_len
    dec.prefill(tiny["prompt"], TINY.n_new)
    dl = G.logits_buf(TINY.vocab)
    dec.set_logits_out(None, dl)
    ids = dec.draft().cpu().numpy()
    dec.check()
    dec.set_logits_out(None, None)
    t_n = dec.stats().t_n
    ref_logits, ref_ids = O.draft_forward(tiny["dw"], tiny["tw"].embed, tiny["cfg"],
                                          tiny["p_taps"], t_n, P, TINY.block)
    G.check_rows("tiny_draft", dl[1:TINY.block].cpu().numpy(), ids[:TINY.block - 1],
                 ref_logits[1:], TOL, DEC_TOL)


@pytest.mark.parametrize("cut", [0, 3, 7])
def test_verify_accept_rollback_match_oracle(tiny, cut):
    """Drafts = the oracle's greedy continuation corrupted at position `cut`
    (7 = not corrupted): acceptance length, emitted tokens, logits and the
    rolled-back positions follow the oracle."""
    dec, P, B = tiny["dec"], TINY.prompt_len, TINY.block
    g = tiny["greedy"]
    dec.prefill(tiny["prompt"], TINY.n_new)
    st = dec.stats()
    d = list(g[1:B])
    if cut < B - 1:
        d[cut] = (d[cut] + 1) % TINY.vocab
    vl = G.logits_buf(TINY.vocab)
    dec.set_logits_out(vl, None)
    toks, n = dec.verify(torch.tensor(d, dtype=torch.int32, device="cuda"))
    dec.check()
    dec.set_logits_out(None, None)
    cache = O.KVCache(len(tiny["tw"].layers), TINY.n_kv, TINY.head_dim)
    O.target_forward(tiny["tw"], tiny["cfg"], tiny["prompt"].tolist(), 0, cache)
    ref_logits, _ = O.target_forward(tiny["tw"], tiny["cfg"], [st.t_n] + d, P, cache)
    gpu = vl[:B].cpu().numpy()
    G.check_rows(f"tiny_verify_{cut}", gpu, None, ref_logits, TOL, DEC_TOL)
    st2 = dec.stats()
    a = G.accept_check(f"tiny_accept_{cut}", toks.tolist(), int(n.item()), st2, ref_logits, d,
                       gpu, TOL, P)
    assert a == cut
    assert all(t == -1 for t in toks[int(n.item()):].tolist())
    assert st2.ctx_len == st2.n and st2.generated == 1 + int(n.item())


def test_spec_equals_greedy_and_oracle(tiny):
    dec = tiny["dec"]
    gg = dec.greedy(tiny["prompt"], TINY.n_new)
    sp = dec.generate(tiny["prompt"], TINY.n_new)
    dec.check()
    assert sp == gg, "GPU speculative output differs from GPU greedy"
    st = dec.stats()
    assert st.generated == TINY.n_new and st.n == TINY.prompt_len + TINY.n_new - 1
    n = G.compared_prefix(gg, tiny["greedy"], tiny["greedy_logits"], TOL)
    assert n >= 8, f"only {n} decidable tokens compared"


@pytest.mark.parametrize("k", [1, 4])
def test_graphed_loop_equals_greedy(tiny, k):
    """Rounds replayed from a CUDA graph of k rounds (tokens and progress read
    back once per replay) emit exactly the greedy stream, and stop at the
    budget even when the last replay runs past the finish."""
    dec = tiny["dec"]
    gg = dec.greedy(tiny["prompt"], TINY.n_new)
    gr = dec.generate_graphed(tiny["prompt"], TINY.n_new, rounds_per_replay=k)
    dec.check()
    assert gr == gg
    st = dec.stats()
    assert st.finished and st.generated == TINY.n_new
    dec._round_graph = None


def test_adaptive_block_follows_oracle_policy(tiny):
    """The adaptive block cap on the device: every round's block length is
    the oracle's policy (adaptive_block_cap / adaptive_ema_update) applied to
    the acceptances the device saw, under drafts that are the GPU greedy
    continuation wrong at their first position for the first ten positions
    (so the cap falls to 4 rows and climbs back); the output is the greedy
    stream."""
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    w = TINY.with_(adaptive_block=True)
    dec = DFlash(w, tiny["m"])
    P = w.prompt_len
    gg = dec.greedy(tiny["prompt"], w.n_new)
    full = tiny["prompt"].tolist() + gg
    rounds = []

    def draft_fn(d):
        st = d.stats()
        if rounds:
            rounds[-1]["a"] = st.last_accept
        ids = full[st.n + 1:st.n + st.block_len]
        if ids and st.n < P + 10:
            ids[0] = (ids[0] + 1) % w.vocab
        rounds.append(dict(n=st.n, gen=st.generated, bl=st.block_len))
        ids = (ids + [0] * w.block)[:w.block - 1]
        return torch.tensor(ids, dtype=torch.int32, device="cuda")

    out = dec.generate(tiny["prompt"], w.n_new, draft_fn=draft_fn)
    dec.check()
    rounds[-1]["a"] = dec.stats().last_accept
    assert out == gg
    ema = float(w.block - 1)
    for r in rounds:
        want = min(O.adaptive_block_cap(ema, w.block), w.n_new - r["gen"], w.max_seq - r["n"])
        assert r["bl"] == want, (r, ema)
        ema = O.adaptive_ema_update(ema, r["a"])
    bls = [r["bl"] for r in rounds]
    assert 4 in bls and max(bls[bls.index(4):]) == w.block
    dec.close()


def test_spec_with_adversarial_drafts_equals_greedy(tiny):
    dec, B = tiny["dec"], TINY.block
    gg = dec.greedy(tiny["prompt"], TINY.n_new)
    rng = np.random.default_rng(3)

    def oracle_like(d):        # the GPU greedy continuation: full acceptance
        st = d.stats()
        k = st.generated
        ids = gg[k:k + B - 1] + [0] * (B - 1)
        return torch.tensor(ids[:B - 1], dtype=torch.int32, device="cuda")

    def random_ids(d):
        return torch.from_numpy(rng.integers(0, TINY.vocab, B - 1).astype(np.int32)).cuda()

    for fn in (oracle_like, random_ids):
        out = dec.generate(tiny["prompt"], TINY.n_new, draft_fn=fn)
        assert out == gg, fn.__name__
        st = dec.stats()
        assert 1 <= st.emitted / max(1, st.rounds) <= B
        if fn is oracle_like:
            assert st.accept_hist[B - 2] >= st.rounds - 2   # every draft position accepted


def test_batch_invariance_rows_equal_single_row(tiny):
    """Row i of a 8-row verify has the bit-identical logits of the i-th
    one-row (greedy) step: the kernels never change with the row count."""
    dec, P, B = tiny["dec"], TINY.prompt_len, TINY.block
    gg = dec.greedy(tiny["prompt"], TINY.n_new)
    dec.prefill(tiny["prompt"], TINY.n_new)
    vl = G.logits_buf(TINY.vocab)
    dec.set_logits_out(vl, None)
    d = torch.tensor(gg[1:B], dtype=torch.int32, device="cuda")
    dec.verify(d)
    batch = vl[:B].clone()
    dec.rollback(P, gg[0])
    for i in range(B):
        dec.verify(None)
        assert torch.equal(vl[0], batch[i]), f"row {i} differs"
    dec.set_logits_out(None, None)
    dec.check()


def test_eos_truncates_like_greedy(tiny):
    from block_diffusion_speculative_gather_gb300.runtime import DFlash
    dec = tiny["dec"]
    gg = dec.greedy(tiny["prompt"], TINY.n_new)
    eos = gg[20]
    de = DFlash(TINY.with_(eos_id=eos), tiny["m"])
    ge = de.greedy(tiny["prompt"], TINY.n_new)
    se = de.generate(tiny["prompt"], TINY.n_new)
    assert ge == gg[: gg.index(eos) + 1]
    assert se == ge
    de.close()


def test_budget_shrinks_last_round(tiny):
    dec = tiny["dec"]
    for n_new in (2, 9, 10, 17):
        gg = dec.greedy(tiny["prompt"], n_new)
        sp = dec.generate(tiny["prompt"], n_new)
        assert len(gg) == n_new and sp == gg


def test_tap_reduce_matches_oracle():
    G.build_lib()
    from block_diffusion_speculative_gather_gb300 import capi
    for hc, H, rows in [(4, 64, 5), (4, 4096, 33), (1, 256, 16), (3, 128, 7)]:
        streams = synth.hc_streams(4, rows, hc, H)
        out = torch.empty((rows, 4 * H), dtype=torch.float32, device="cuda")
        dev = [streams[i].cuda().contiguous() for i in range(4)]
        capi.dflash_tap_reduce(dev, rows, hc, H, out)
        torch.cuda.synchronize()
        ref = O.tap_concat([streams[i].float().numpy() for i in range(4)], hc)
        np.testing.assert_allclose(out.cpu().numpy(), ref, rtol=2e-7, atol=1e-7)


def test_quantizer_bit_exact_with_oracle():
    G.build_lib()
    from block_diffusion_speculative_gather_gb300 import capi
    w = synth.normal((384, 512), 0.02, 0, "quant-test")
    w[5, :64] = 0.0
    wt = torch.from_numpy(w).cuda()
    packed = torch.empty((384, 256), dtype=torch.uint8, device="cuda")
    scales = torch.empty((8, 384), dtype=torch.int16, device="cuda")
    capi.dflash_quantize_int4g64(wt, packed, scales)
    torch.cuda.synchronize()
    ref_p, ref_s = O.quantize_int4_g64(w)
    # the library's words interleave 8 consecutive inputs: k0+2j in nibble j,
    # k0+2j+1 in nibble j+4; decode them back to the oracle's natural order
    words = packed.cpu().numpy().view(np.uint32)                 # [384, 64]
    nib = (words[..., None] >> (4 * np.arange(8, dtype=np.uint32))) & 0xF
    codes = np.empty((384, 64, 8), np.uint8)
    codes[..., 0::2] = nib[..., 0:4]
    codes[..., 1::2] = nib[..., 4:8]
    codes = codes.reshape(384, 512)
    ref_codes = np.empty((384, 512), np.uint8)
    ref_codes[:, 0::2] = ref_p & 0xF
    ref_codes[:, 1::2] = ref_p >> 4
    np.testing.assert_array_equal(codes, ref_codes)
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint16).T, ref_s)
