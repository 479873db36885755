"""GPU parity of the many-sequence round (dflash_batch_*): three independent
sequences of different prompt lengths and budgets on the Qwen3-4B-shaped
2-layer bf16 model (hidden 2560, 32 q / 8 kv heads, head_dim 128, SwiGLU
9728, vocab 151936, one drafter layer, block 16; norm weights N(1, 0.1)),
their rows run together through the dense tcgen05 GEMM.

Checked against the oracle: every sequence's draft rows (the uncached
drafter), its verify rows and acceptance for greedy-continuation drafts cut
at 0, 7 or not at all (one cut per sequence, in the same batched verify),
its greedy stream, and lockstep multi-round decoding against
spec_decode_batch with the same injected drafts on both sides (per round
acceptance and emitted tokens).  Against the GPU itself: speculative ==
greedy per sequence (lossless), and a sequence's logits are bit-identical
whether it runs alone (S = 1) or beside others (S = 3).

Tolerance and decidability as in test_gpu_bf16.py: logits within rel 2e-2,
ids exact on rows decidable at the GPU row's measured error, floors at
DEC_TOL.
"""

import numpy as np
import pytest
import torch

from block_diffusion_speculative_gather_gb300 import synth
from block_diffusion_speculative_gather_gb300.configs import E2E_BF16
from oracle import dflash_oracle as O
from tests import gpu_common as G
from tests.oracle_inputs import ModelTensors, oracle_config, oracle_draft, oracle_target

pytestmark = pytest.mark.gpu
TOL = 2e-2
DEC_TOL = 1e-3
W = E2E_BF16.with_(name="bf16_2layer_batch", tgt_layers=2, drf_layers=1, tap_layers=(0, 1),
                   max_seq=256)
LENS = (40, 33, 57)
BUDGETS = (16, 11, 20)
CUTS = (0, 7, None)


@pytest.fixture(scope="module")
def batch():
    G.build_lib()
    from block_diffusion_speculative_gather_gb300.runtime import DFlashBatch
    m = ModelTensors(W, std=0.02, norm_std=0.1)
    tw, dw, cfg = oracle_target(m), oracle_draft(m), oracle_config(W)
    prompts, taps, greedy, glogits = [], [], [], []
    for i, P in enumerate(LENS):
        p = synth.uniform_ids(P, W.vocab, seed=40 + i)
        lg, tp = O.target_forward(tw, cfg, p.tolist(), 0, O.KVCache(2, W.n_kv, W.head_dim))
        g = O.greedy(tw, cfg, p.tolist(), BUDGETS[i])
        tf, _ = O.target_forward(tw, cfg, p.tolist() + g[:-1], 0, O.KVCache(2, W.n_kv, W.head_dim))
        prompts.append(torch.from_numpy(p))
        taps.append(tp)
        greedy.append(g)
        glogits.append(tf[P - 1:])
    dec = DFlashBatch(W, m, S=len(LENS))
    return dict(m=m, tw=tw, dw=dw, cfg=cfg, prompts=prompts, taps=taps, greedy=greedy,
                glogits=glogits, dec=dec)


def _budgets():
    return list(BUDGETS)


def test_batch_draft_matches_oracle(batch):
    dec = batch["dec"]
    dec.prefill(batch["prompts"], _budgets())
    dl = torch.zeros((16 * dec.S, W.vocab), dtype=torch.float32, device="cuda")
    dec.set_logits_out(None, dl)
    ids = dec.draft().cpu().numpy()
    dec.check()
    dec.set_logits_out(None, None)
    for s, P in enumerate(LENS):
        st = dec.stats(s)
        assert st.t_n == batch["greedy"][s][0] and st.n == P
        bl = st.block_len                 # min(16, budget - 1): the block this sequence drafted
        ref, _ = O.draft_forward(batch["dw"], batch["tw"].embed, batch["cfg"], batch["taps"][s], st.t_n,
                                 P, bl)
        G.check_rows(f"batch_draft_{s}", dl[16 * s + 1:16 * s + bl].cpu().numpy(), ids[s][:bl - 1],
                     ref[1:], TOL, DEC_TOL)
        assert all(int(x) == -1 for x in ids[s][bl - 1:])


def test_batch_verify_and_accept_match_oracle(batch):
    """One batched verify: sequence s verifies its oracle greedy continuation
    cut at CUTS[s] (0, 7, none); each sequence's 16 rows against the oracle,
    its acceptance, emitted tokens (bonus included) and rolled-back length."""
    dec, B = batch["dec"], W.block
    dec.prefill(batch["prompts"], _budgets())
    drafts = torch.zeros((dec.S, B - 1), dtype=torch.int32)
    ds = []
    for s in range(dec.S):
        g = batch["greedy"][s]
        d = (list(g[1:B]) + [0] * B)[:B - 1]
        bl = dec.stats(s).block_len
        d = d[:bl - 1] + [0] * (B - bl)
        if CUTS[s] is not None:
            d[CUTS[s]] = (d[CUTS[s]] + 1) % W.vocab
        drafts[s] = torch.tensor(d, dtype=torch.int32)
        ds.append(d[:bl - 1])
    vl = torch.zeros((16 * dec.S, W.vocab), dtype=torch.float32, device="cuda")
    dec.set_logits_out(vl, None)
    toks, n = dec.verify(drafts.cuda())
    dec.check()
    dec.set_logits_out(None, None)
    toks, n = toks.cpu().tolist(), n.cpu().tolist()
    for s, P in enumerate(LENS):
        cache = O.KVCache(2, W.n_kv, W.head_dim)
        O.target_forward(batch["tw"], batch["cfg"], batch["prompts"][s].tolist(), 0, cache)
        ref, _ = O.target_forward(batch["tw"], batch["cfg"], [batch["greedy"][s][0]] + ds[s], P, cache)
        T = len(ds[s]) + 1
        gpu = vl[16 * s:16 * s + T].cpu().numpy()
        G.check_rows(f"batch_verify_{s}", gpu, None, ref, TOL, DEC_TOL)
        # exact acceptance where the accepted rows are decidable, else
        # agreement up to the first undecidable row (this seed's prompt 2
        # has rows with top-2 margins of 0.08 % of the largest logit)
        a, k = G.accept_prefix_check(f"batch_accept_{s}", toks[s], n[s], dec.stats(s), ref, ds[s], gpu,
                                     TOL, DEC_TOL, P)
        assert a == (T - 1 if CUTS[s] is None else CUTS[s])
        if CUTS[s] is not None:
            assert k > a, (s, k, a)       # the cut rows are decidable: the exact check ran


def test_batch_greedy_streams_match_oracle(batch):
    dec = batch["dec"]
    vl = torch.zeros((16 * dec.S, W.vocab), dtype=torch.float32, device="cuda")
    dec.set_logits_out(vl, None)
    dec.prefill(batch["prompts"], _budgets())
    # the prefill's last rows come from each context's own 16-row forward;
    # the stream starts from the batched steps (token 1 on)
    outs = [[dec.stats(s).t_n] for s in range(dec.S)]
    rows = [[] for _ in range(dec.S)]
    while not all(dec.stats(s).finished for s in range(dec.S)):
        toks, n = dec.verify(None)
        toks, n = toks.cpu().tolist(), n.cpu().tolist()
        for s in range(dec.S):
            if n[s]:
                outs[s].extend(toks[s][:n[s]])
                rows[s].append(vl[16 * s].clone())
    dec.check()
    dec.set_logits_out(None, None)
    for s in range(dec.S):
        assert len(outs[s]) == BUDGETS[s]
        assert outs[s][0] == batch["greedy"][s][0]
        gl = batch["glogits"][s][1:]
        floor = next((i for i, r in enumerate(gl) if not G.decidable(r, DEC_TOL)), len(gl))
        k = G.stream_prefix(f"batch_greedy_stream_{s}", outs[s][1:], [r.cpu().numpy() for r in rows[s]],
                            batch["greedy"][s][1:], gl, TOL)
        assert k >= floor and k > 0, (s, k, floor)
        batch.setdefault("prefix", {})[s] = 1 + k      # tokens that must agree with the oracle


def _injected(g, s, n, bl, k):
    """Drafts of a round (both sides): the oracle greedy continuation from
    token k, its first mismatch at a position drawn from (sequence, n)."""
    d = [int(g[min(k + j, len(g) - 1)]) for j in range(bl - 1)]
    cut = (7 * n + 3 * s) % (bl + 2)
    if cut < bl - 1:
        d[cut] = (d[cut] + 1) % W.vocab
    return d


def test_batch_rounds_match_spec_decode_batch(batch):
    """Lockstep speculative rounds of the three sequences with injected drafts
    (the same on both sides): every round's emitted tokens and the final
    streams equal the oracle's spec_decode_batch, and equal greedy."""
    dec, B = batch["dec"], W.block
    gs = batch["greedy"]
    plens = list(LENS)

    def override(s):
        return lambda t_n, n, bl, hist: _injected(gs[s], s, n, bl, len(hist) - plens[s])

    bt = O.spec_decode_batch(batch["tw"], batch["dw"], batch["cfg"],
                             [p.tolist() for p in batch["prompts"]], _budgets(),
                             draft_overrides=[override(s) for s in range(dec.S)])
    per_round = [[r["emitted"] for r in tr.per_round] for tr in bt.traces]

    def draft_fn(d):
        out = torch.zeros((d.S, B - 1), dtype=torch.int32)
        for s in range(d.S):
            st = d.stats(s)
            if st.block_len > 1:
                ids = _injected(gs[s], s, st.n, st.block_len, st.generated)
                out[s, :len(ids)] = torch.tensor(ids, dtype=torch.int32)
        return out.cuda()

    dec.prefill(batch["prompts"], _budgets())
    outs = [[dec.stats(s).t_n] for s in range(dec.S)]
    gpu_rounds = [[] for _ in range(dec.S)]
    while not all(dec.stats(s).finished for s in range(dec.S)):
        d = draft_fn(dec)
        dec.draft()                                   # runs; its ids are replaced
        toks, n = dec.verify(d)
        toks, n = toks.cpu().tolist(), n.cpu().tolist()
        for s in range(dec.S):
            if n[s]:
                outs[s].extend(toks[s][:n[s]])
                gpu_rounds[s].append(n[s])
    dec.check()
    for s in range(dec.S):
        assert bt.traces[s].tokens == gs[s]           # the oracle's own invariant
        # tokens up to the greedy stream's decidable prefix, and every round
        # that lies inside it, exactly as the oracle's
        K = batch.get("prefix", {}).get(s, 1)
        assert outs[s][:K] == gs[s][:K], s
        done = 1
        for i, (g_n, o_n) in enumerate(zip(gpu_rounds[s], per_round[s])):
            if done + o_n > K:
                break
            assert g_n == o_n, (s, i, gpu_rounds[s], per_round[s])
            done += o_n
        assert max(per_round[s]) > 1                  # some drafts were accepted
        if K == len(gs[s]):
            assert outs[s] == gs[s] and gpu_rounds[s] == per_round[s]


def test_batch_spec_equals_batch_greedy(batch):
    """Losslessness of the batched round: with the drafter's own ids, every
    sequence's speculative output equals its batched greedy decoding."""
    dec = batch["dec"]
    gg = dec.greedy(batch["prompts"], _budgets())
    sp = dec.generate(batch["prompts"], _budgets())
    dec.check()
    assert sp == gg


def test_batch_sequence_independent_of_batch_size(batch):
    """Sequence 0 alone (S = 1) and beside two others (S = 3): its draft and
    verify logits are bit-identical (split counts and tile widths depend on
    N and K only; attention and norms work per row)."""
    from block_diffusion_speculative_gather_gb300.runtime import DFlashBatch
    dec3 = batch["dec"]
    dec1 = DFlashBatch(W, batch["m"], S=1)
    out = []
    for dec, S in ((dec3, 3), (dec1, 1)):
        dec.prefill(batch["prompts"][:S], _budgets()[:S])
        vl = torch.zeros((16 * S, W.vocab), dtype=torch.float32, device="cuda")
        dl = torch.zeros((16 * S, W.vocab), dtype=torch.float32, device="cuda")
        dec.set_logits_out(vl, dl)
        d = dec.draft()
        dec.verify(d)
        dec.check()
        dec.set_logits_out(None, None)
        out.append((dl[:16].clone(), vl[:16].clone(), d[0].clone()))
    dec1.close()
    assert torch.equal(out[0][2], out[1][2])
    assert torch.equal(out[0][0], out[1][0])
    assert torch.equal(out[0][1], out[1][1])


def test_batch_sequence_independent_of_tile_width(batch):
    """Nine sequences take two row tiles, so the projections run 256-column
    tiles (one wave of CTAs) where one to eight sequences run 128-column
    tiles, at the same k-split counts: sequence 0's draft and verify logits
    must still be bit-identical to its S = 1 run."""
    from block_diffusion_speculative_gather_gb300.runtime import DFlashBatch
    prompts = list(batch["prompts"]) + [torch.from_numpy(synth.uniform_ids(24 + 5 * i, W.vocab, seed=70 + i))
                                        for i in range(6)]
    budgets = _budgets() + [12] * 6
    out = []
    for S in (9, 1):
        dec = DFlashBatch(W, batch["m"], S=S)
        dec.prefill(prompts[:S], budgets[:S])
        vl = torch.zeros((16 * S, W.vocab), dtype=torch.float32, device="cuda")
        dl = torch.zeros((16 * S, W.vocab), dtype=torch.float32, device="cuda")
        dec.set_logits_out(vl, dl)
        d = dec.draft()
        dec.verify(d)
        dec.check()
        dec.set_logits_out(None, None)
        out.append((dl[:16].clone(), vl[:16].clone(), d[0].clone()))
        dec.close()
    assert torch.equal(out[0][2], out[1][2])
    assert torch.equal(out[0][0], out[1][0])
    assert torch.equal(out[0][1], out[1][1])


def test_batch_maximum_sequences(batch):
    """The largest batch the library takes (32 sequences: four row tiles,
    the attention over several waves of CTAs, the largest workspace): the
    first and the last sequence's draft and verify logits are bit-identical
    to their own S = 1 runs."""
    from block_diffusion_speculative_gather_gb300 import capi
    from block_diffusion_speculative_gather_gb300.runtime import DFlashBatch
    S = 32
    prompts = [torch.from_numpy(synth.uniform_ids(20 + (7 * i) % 40, W.vocab, seed=200 + i)) for i in range(S)]
    budgets = [8 + i % 5 for i in range(S)]

    def run(ps, bs):
        dec = DFlashBatch(W, batch["m"], S=len(ps))
        dec.prefill(ps, bs)
        n = len(ps)
        vl = torch.zeros((16 * n, W.vocab), dtype=torch.float32, device="cuda")
        dl = torch.zeros((16 * n, W.vocab), dtype=torch.float32, device="cuda")
        dec.set_logits_out(vl, dl)
        d = dec.draft()
        dec.verify(d)
        dec.check()
        dec.set_logits_out(None, None)
        dec.close()
        return dl, vl, d

    dl, vl, d = run(prompts, budgets)
    for s in (0, S - 1):
        dl1, vl1, d1 = run([prompts[s]], [budgets[s]])
        assert torch.equal(d[s], d1[0]), s
        assert torch.equal(dl[16 * s:16 * s + 16], dl1[:16]), s
        assert torch.equal(vl[16 * s:16 * s + 16], vl1[:16]), s
    with pytest.raises(capi.DFlashError):
        DFlashBatch(W, batch["m"], S=S + 1)
