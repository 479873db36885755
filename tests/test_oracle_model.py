"""Pins of the oracle's target, drafter and speculative loop.

* target_forward / draft_forward against a float64 composition of torch
  library routines (F.linear, F.rms_norm, scaled_dot_product_attention with
  GQA and a boolean mask, F.silu, RoPE as a complex rotation via torch.polar);
* invariants the definitions imply: causality, incremental == full-sequence
  decoding, RoPE shift invariance of the drafter, window locality;
* the speculative loop: output identical to plain greedy decoding for the
  real drafter and for adversarial drafts, first-mismatch acceptance
  lengths, rollback positions and the budget.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.configs import TINY
from oracle import dflash_oracle as O
from tests.oracle_inputs import ModelTensors, oracle_config, oracle_draft, oracle_target

T64 = torch.float64


@pytest.fixture(scope="module", params=[0.02, 0.1], ids=["std0.02", "std0.1"])
def tiny(request):
    m = ModelTensors(TINY, std=request.param)
    return dict(tw=oracle_target(m), dw=oracle_draft(m), cfg=oracle_config(TINY),
                prompt=synth.uniform_ids(TINY.prompt_len, TINY.vocab).tolist())


# ------------------------------------------------------- torch composition

def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def _rope_polar(x, positions, theta):
    d = x.shape[-1]
    half = d // 2
    freq = 1.0 / theta ** (torch.arange(half, dtype=T64) * 2 / d)
    ang = torch.tensor(positions, dtype=T64)[:, None] * freq[None, :]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, :]
    z = torch.complex(x[..., :half], x[..., half:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def _torch_layer(x, lw, cfg, q_pos, k_rows, mask):
    """One decoder layer; k_rows(h, k_norm) -> (k, v) of all keys."""
    H, d = cfg.hidden, cfg.head_dim
    h = F.rms_norm(x, (H,), _t(lw["ln_attn"]), eps=cfg.rms_eps)
    q = F.linear(h, _t(lw["wq"])).view(len(q_pos), cfg.n_q, d)
    q = _rope_polar(F.rms_norm(q, (d,), _t(lw["q_norm"]), eps=cfg.rms_eps), q_pos,
                    cfg.rope_theta)
    k, v = k_rows(h)
    a = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None],
                                       v.permute(1, 0, 2)[None], attn_mask=mask,
                                       scale=1 / math.sqrt(d), enable_gqa=True)
    x = x + F.linear(a[0].permute(1, 0, 2).reshape(len(q_pos), -1), _t(lw["wo"]))
    h2 = F.rms_norm(x, (H,), _t(lw["ln_mlp"]), eps=cfg.rms_eps)
    return x + F.linear(F.silu(F.linear(h2, _t(lw["w_gate"]))) * F.linear(h2, _t(lw["w_up"])),
                        _t(lw["w_down"]))


def _torch_kv(h, lw, cfg, pos):
    d = cfg.head_dim
    k = F.linear(h, _t(lw["wk"])).view(len(pos), cfg.n_kv, d)
    k = _rope_polar(F.rms_norm(k, (d,), _t(lw["k_norm"]), eps=cfg.rms_eps), pos, cfg.rope_theta)
    v = F.linear(h, _t(lw["wv"])).view(len(pos), cfg.n_kv, d)
    return k, v


def _torch_target_logits(tw, cfg, tokens):
    T = len(tokens)
    pos = list(range(T))
    x = _t(tw.embed)[torch.tensor(tokens)]
    mask = torch.ones(T, T, dtype=torch.bool).tril()
    for lw in tw.layers:
        x = _torch_layer(x, lw, cfg, pos, lambda h, lw=lw: _torch_kv(h, lw, cfg, pos), mask)
    return F.linear(F.rms_norm(x, (cfg.hidden,), _t(tw.final_norm), eps=cfg.rms_eps),
                    _t(tw.embed)).numpy()


def _torch_draft_logits(dw, embed, cfg, taps, t_n, n, bl):
    lo = 0 if cfg.window == 0 else max(0, n - cfg.window)
    ctx_pos = list(range(lo, n))
    H, d = cfg.hidden, cfg.head_dim
    c = F.linear(_t(taps[lo:n]), _t(dw.fc))
    c = F.rms_norm(c, (H,), _t(dw.ctx_norm), eps=cfg.rms_eps)
    blk = list(range(n, n + bl))
    x = _t(embed)[torch.tensor([t_n] + [cfg.vocab - 1] * (bl - 1))]
    mask = torch.ones(bl, len(ctx_pos) + bl, dtype=torch.bool)

    def kv(h, lw):
        kc, vc = _torch_kv(c, lw, cfg, ctx_pos)
        kb, vb = _torch_kv(h, lw, cfg, blk)
        return torch.cat([kc, kb]), torch.cat([vc, vb])

    for lw in dw.layers:
        x = _torch_layer(x, lw, cfg, blk, lambda h, lw=lw: kv(h, lw), mask)
    return F.linear(F.rms_norm(x, (H,), _t(dw.final_norm), eps=cfg.rms_eps), _t(embed)).numpy()


def test_target_forward_matches_torch_composition(tiny):
    tw, cfg, prompt = tiny["tw"], tiny["cfg"], tiny["prompt"]
    cache = O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim)
    logits, taps = O.target_forward(tw, cfg, prompt, 0, cache)
    ref = _torch_target_logits(tw, cfg, prompt)
    np.testing.assert_allclose(logits, ref, rtol=1e-10, atol=1e-10)
    assert taps.shape == (len(prompt), cfg.n_taps * cfg.hidden)


def test_draft_forward_matches_torch_composition(tiny):
    tw, dw, cfg = tiny["tw"], tiny["dw"], tiny["cfg"]
    taps = synth.tap_rows(100, cfg.n_taps * cfg.hidden, torch.float32).numpy()
    for n, window in [(0, 64), (10, 64), (100, 64), (100, 0)]:
        cfg.window = window
        logits, ids = O.draft_forward(dw, tw.embed, cfg, taps, 17, n, 8)
        ref = _torch_draft_logits(dw, tw.embed, cfg, taps, 17, n, 8)
        np.testing.assert_allclose(logits, ref, rtol=1e-10, atol=1e-10)
        assert ids == [int(np.argmax(ref[j])) for j in range(1, 8)]
    cfg.window = TINY.window


def test_untied_lm_head_reads_only_the_logits(tiny):
    """An untied LM head L replaces the embedding in the logits only: with
    L = 2 E every logit doubles exactly (the embedding gather, hence every
    hidden state, is unchanged), for the target and for the drafter."""
    import dataclasses
    tw, dw, cfg, prompt = tiny["tw"], tiny["dw"], tiny["cfg"], tiny["prompt"]
    tw2 = dataclasses.replace(tw, lm_head=2.0 * tw.embed.astype(np.float64))
    l1, t1 = O.target_forward(tw, cfg, prompt, 0, O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim))
    l2, t2 = O.target_forward(tw2, cfg, prompt, 0, O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim))
    np.testing.assert_array_equal(l2, 2.0 * l1)
    np.testing.assert_array_equal(t2, t1)
    taps = synth.tap_rows(40, cfg.n_taps * cfg.hidden, torch.float32).numpy()
    d1, _ = O.draft_forward(dw, tw.embed, cfg, taps, 17, 40, 8)
    d2, _ = O.draft_forward(dw, tw.embed, cfg, taps, 17, 40, 8, lm_head=tw2.lm_head)
    np.testing.assert_array_equal(d2, 2.0 * d1)


# ------------------------------------------------------- invariants

def test_incremental_decoding_equals_full_forward(tiny):
    tw, cfg, prompt = tiny["tw"], tiny["cfg"], tiny["prompt"][:12]
    full, full_taps = O.target_forward(tw, cfg, prompt, 0,
                                       O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim))
    cache = O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim)
    rows, trows = [], []
    for p, t in enumerate(prompt):
        lg, tp = O.target_forward(tw, cfg, [t], p, cache)
        rows.append(lg[0])
        trows.append(tp[0])
    np.testing.assert_allclose(np.stack(rows), full, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(np.stack(trows), full_taps, rtol=1e-11, atol=1e-11)


def test_target_is_causal(tiny):
    tw, cfg, prompt = tiny["tw"], tiny["cfg"], tiny["prompt"]
    mk = lambda: O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim)
    a, _ = O.target_forward(tw, cfg, prompt[:10], 0, mk())
    b, _ = O.target_forward(tw, cfg, prompt[:10] + [1, 2, 3], 0, mk())
    np.testing.assert_allclose(a, b[:10], rtol=1e-11, atol=1e-11)


def test_draft_shift_invariance(tiny):
    """Shifting the block and every context position by the same amount
    leaves the drafter's logits unchanged (RoPE is relative)."""
    tw, dw, cfg = tiny["tw"], tiny["dw"], tiny["cfg"]
    taps = synth.tap_rows(300, cfg.n_taps * cfg.hidden, torch.float32).numpy()
    a, _ = O.draft_forward(dw, tw.embed, cfg, taps[:100], 5, 100, 8)
    shifted = np.concatenate([np.zeros((200, taps.shape[1])), taps[:100]])
    b, _ = O.draft_forward(dw, tw.embed, cfg, shifted, 5, 300, 8)
    np.testing.assert_allclose(a, b, rtol=1e-8, atol=1e-8)


def test_draft_window_locality(tiny):
    """Tap rows before the window do not matter; rows inside it do."""
    tw, dw, cfg = tiny["tw"], tiny["dw"], tiny["cfg"]
    taps = synth.tap_rows(100, cfg.n_taps * cfg.hidden, torch.float32).numpy()
    base, _ = O.draft_forward(dw, tw.embed, cfg, taps, 5, 100, 8)
    outside = taps.copy()
    outside[:100 - cfg.window] = 7.0
    same, _ = O.draft_forward(dw, tw.embed, cfg, outside, 5, 100, 8)
    np.testing.assert_array_equal(base, same)
    inside = taps.copy()
    inside[100 - cfg.window] += 1.0
    diff, _ = O.draft_forward(dw, tw.embed, cfg, inside, 5, 100, 8)
    assert np.max(np.abs(diff - base)) > 1e-6


def test_draft_block_is_bidirectional(tiny):
    """Block row 0 depends on the later block rows (non-causal block)."""
    tw, dw, cfg = tiny["tw"], tiny["dw"], tiny["cfg"]
    taps = synth.tap_rows(20, cfg.n_taps * cfg.hidden, torch.float32).numpy()
    a, _ = O.draft_forward(dw, tw.embed, cfg, taps, 5, 20, 2)
    b, _ = O.draft_forward(dw, tw.embed, cfg, taps, 5, 20, 8)
    assert np.max(np.abs(a[0] - b[0])) > 1e-9


# ------------------------------------------------------- speculative loop

def _check_trace(tr, cfg, prompt, n_new):
    assert len(tr.tokens) == n_new
    total = 1                                   # the prefill's first token
    for r in tr.per_round:
        total += r["emitted"]
        assert 1 <= r["emitted"] <= r["bl"]
        assert r["emitted"] == r["a"] + 1
        assert r["kv_len"] == len(prompt) + total - 1
        assert r["ctx_len"] == r["kv_len"]


def test_spec_equals_greedy_with_real_drafter(tiny):
    tw, dw, cfg, prompt = tiny["tw"], tiny["dw"], tiny["cfg"], tiny["prompt"]
    g = O.greedy(tw, cfg, prompt, TINY.n_new)
    tr = O.spec_decode(tw, dw, cfg, prompt, TINY.n_new)
    assert tr.tokens == g
    _check_trace(tr, cfg, prompt, TINY.n_new)


def test_spec_equals_greedy_with_adversarial_drafts(tiny):
    tw, cfg, prompt = tiny["tw"], tiny["cfg"], tiny["prompt"]
    n_new = 40
    g = O.greedy(tw, cfg, prompt, n_new)
    rng = np.random.default_rng(11)

    def random_drafts(t_n, n, bl, hist):
        return rng.integers(0, cfg.vocab, size=bl - 1).tolist()

    def oracle_drafts(t_n, n, bl, hist):
        k = len(hist) - len(prompt)
        return g[k:k + bl - 1]

    cut = {}

    def corrupted(t_n, n, bl, hist):
        d = oracle_drafts(t_n, n, bl, hist)
        j = int(rng.integers(0, bl - 1))
        d[j] = (d[j] + 1) % cfg.vocab
        cut[n] = j
        return d

    for fn in (random_drafts, oracle_drafts, corrupted):
        tr = O.spec_decode(tw, None, cfg, prompt, n_new, draft_override=fn)
        assert tr.tokens == g, fn.__name__
        _check_trace(tr, cfg, prompt, n_new)
        if fn is oracle_drafts:
            assert all(r["a"] == r["bl"] - 1 for r in tr.per_round)
        if fn is corrupted:
            for r in tr.per_round:
                if r["bl"] > 1:
                    assert r["a"] == cut[r["n"]]


def test_adaptive_block_spec_equals_greedy_and_follows_the_policy(tiny):
    """With the adaptive cap the loop stays lossless, and each round's block
    is min(cap(ema), budget) with ema the halving average of the accepted
    drafts so far (drafts copied from greedy, wrong at their first position
    for the first ten positions and right afterwards, so the cap falls to 4
    rows and climbs back)."""
    import dataclasses
    tw, dw, prompt = tiny["tw"], tiny["dw"], tiny["prompt"]
    cfg = dataclasses.replace(tiny["cfg"], adaptive_block=True)
    g = O.greedy(tw, cfg, prompt, TINY.n_new)
    full = list(prompt) + g

    def drafts(t_n, n, bl, hist):
        d = full[n + 1:n + bl]
        if d and n < len(prompt) + 10:
            d[0] = (d[0] + 1) % cfg.vocab
        return d

    tr = O.spec_decode(tw, dw, cfg, prompt, TINY.n_new, draft_override=drafts)
    assert tr.tokens == g
    ema, B = 7.0, cfg.block
    for r in tr.per_round:
        gen = r["n"] - len(prompt) + 1
        want = min(O.adaptive_block_cap(ema, B), TINY.n_new - gen, cfg.max_seq - r["n"])
        assert r["bl"] == want
        ema = O.adaptive_ema_update(ema, r["a"])
    bls = [r["bl"] for r in tr.per_round]
    assert 4 in bls and bls.index(4) < len(bls) - 1 and max(bls[bls.index(4):]) == cfg.block
    tr2 = O.spec_decode(tw, dw, cfg, prompt, TINY.n_new)
    assert tr2.tokens == g


def test_spec_eos_and_budget(tiny):
    tw, cfg, prompt = tiny["tw"], tiny["cfg"], tiny["prompt"]
    g = O.greedy(tw, cfg, prompt, 30)
    eos = g[17]
    cfg_e = oracle_config(TINY, eos_id=eos)
    ge = O.greedy(tw, cfg_e, prompt, 30)
    assert ge == g[:g.index(eos) + 1]

    def oracle_drafts(t_n, n, bl, hist):
        k = len(hist) - len(prompt)
        return g[k:k + bl - 1]

    tr = O.spec_decode(tw, None, cfg_e, prompt, 30, draft_override=oracle_drafts)
    assert tr.tokens == ge
    # odd budget: the last round shrinks, a 1-token remainder skips the draft
    for n_new in (9, 10, 17):
        tr = O.spec_decode(tw, None, cfg, prompt, n_new, draft_override=oracle_drafts)
        assert tr.tokens == g[:n_new]
        assert tr.per_round[-1]["bl"] == min(cfg.block, n_new - 1 - sum(
            r["emitted"] for r in tr.per_round[:-1]))


def test_tap_commit_holds_the_full_forward_taps(tiny):
    """After the loop, the draft context's tap row at every position p is the
    target's tap row of a single forward over the whole confirmed sequence
    at p: rounds commit exactly the taps of the accepted verify rows (the
    pending token's row is not committed)."""
    tw, dw, cfg, prompt = tiny["tw"], tiny["dw"], tiny["cfg"], tiny["prompt"]
    g = O.greedy(tw, cfg, prompt, 40)

    def drafts(t_n, n, bl, hist):   # right for most rows, wrong at every third round
        k = len(hist) - len(prompt)
        d = g[k:k + bl - 1]
        if d and (n % 3) == 0:
            d[len(d) // 2] = (d[len(d) // 2] + 1) % cfg.vocab
        return d

    for fn in (drafts, None):
        tr = O.spec_decode(tw, dw, cfg, prompt, 40, draft_override=fn)
        assert tr.tokens == g
        seq = list(prompt) + tr.tokens[:-1]
        _, full = O.target_forward(tw, cfg, seq, 0, O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim))
        assert len(tr.ctx_taps) == len(seq)
        np.testing.assert_allclose(np.stack(tr.ctx_taps), full, rtol=1e-10, atol=1e-10)


def test_batch_of_sequences_equals_each_sequence_alone(tiny):
    """Lockstep multi-sequence rounds: every sequence's tokens are its own
    greedy decoding and its rounds those of its single-sequence run; the
    batched round count is the longest sequence's, each batched round's
    verify rows are the block lengths of the sequences still running, and
    reordering the batch reorders the results."""
    tw, dw, cfg = tiny["tw"], tiny["dw"], tiny["cfg"]
    prompts = [tiny["prompt"], synth.uniform_ids(20, TINY.vocab, seed=5).tolist(),
               synth.uniform_ids(27, TINY.vocab, seed=6).tolist()]
    budgets = [24, 9, 16]
    greedy = [O.greedy(tw, cfg, p, b) for p, b in zip(prompts, budgets)]

    def copy_of(i):   # drafts copied from greedy, wrong at every third round
        def fn(t_n, n, bl, hist):
            k = len(hist) - len(prompts[i])
            d = greedy[i][k:k + bl - 1]
            if d and (n // 2) % 3 == 0:
                d[-1] = (d[-1] + 1) % cfg.vocab
            return d
        return fn

    for overrides in (None, [copy_of(0), None, copy_of(2)]):
        bt = O.spec_decode_batch(tw, dw, cfg, prompts, budgets, overrides)
        for i, tr in enumerate(bt.traces):
            assert tr.tokens == greedy[i]
            f = overrides[i] if overrides else None
            assert tr.per_round == O.spec_decode(tw, dw, cfg, prompts[i], budgets[i], f).per_round
        assert bt.rounds == max(tr.rounds for tr in bt.traces)
        assert len({tr.rounds for tr in bt.traces}) > 1          # sequences leave at different rounds
        for r in range(bt.rounds):
            assert bt.rows_per_round[r] == sum(tr.per_round[r]["bl"] for tr in bt.traces
                                               if r < tr.rounds)
        rev = O.spec_decode_batch(tw, dw, cfg, prompts[::-1], budgets[::-1],
                                  overrides[::-1] if overrides else None)
        assert [t.tokens for t in rev.traces] == [t.tokens for t in bt.traces][::-1]
        assert rev.rows_per_round == bt.rows_per_round


def test_tap_is_residual_after_layer(tiny):
    """A tap at the last layer is the stream the final norm reads: the logits
    follow from it through final RMSNorm and the tied LM head."""
    tw, cfg, prompt = tiny["tw"], tiny["cfg"], tiny["prompt"][:6]
    cfg_last = oracle_config(TINY, tap_layers=[len(tw.layers) - 1])
    logits, taps = O.target_forward(tw, cfg_last, prompt, 0,
                                    O.KVCache(len(tw.layers), cfg.n_kv, cfg.head_dim))
    again = F.linear(F.rms_norm(_t(taps), (cfg.hidden,), _t(tw.final_norm), eps=cfg.rms_eps),
                     _t(tw.embed)).numpy()
    np.testing.assert_allclose(logits, again, rtol=1e-12, atol=1e-12)
