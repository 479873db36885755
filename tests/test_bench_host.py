"""Host logic of the bench (no GPU).

* The clock record taken during the timed region: the parser that decides
  whether a run is kept (a throttle reason reported as Active, the median SM
  clock against the maximum) on fabricated `nvidia-smi` lines.
* The injected-acceptance schedule: every round's block length and its
  emitted count follow from the oracle's own rules — block_len (and, with
  the adaptive cap, adaptive_block_cap / adaptive_ema_update) and
  first-mismatch acceptance of the draft row against the greedy
  continuation ("[RFC] DFlash", "Key Implementation Details" Phase 3;
  "Requested changes" 1) — so the bench's injected rounds are rounds the
  method would run, whatever profile the generator draws.
"""

import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from oracle import dflash_oracle as O  # noqa: E402


def _summary(lines):
    cs = bench.ClockSampler(0)          # no sampler process is started
    cs.f.write("".join(line + "\n" for line in lines))
    return cs.summary()


def test_clock_summary_median_max_and_reasons():
    na = "Not Active"
    lines = [
        f"0, 2070, 2070, 1010.5, 0x0000000000000000, {na}, {na}, {na}, {na}",
        f"0, 1995, 2070, 1390.0, 0x0000000000000004, {na}, {na}, {na}, Active",
        f"0, 2070, 2070, 1200.0, 0x0000000000000000, {na}, {na}, {na}, {na}",
        "garbled line",
        f"0, [N/A], 2070, 1.0, 0x0, {na}, {na}, {na}, {na}",
    ]
    s = _summary(lines)
    assert s["sm_mhz"] == 2070.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]      # kept and noted, not a rejection


def test_clock_summary_reports_every_slowdown_reason():
    na = "Not Active"
    s = _summary([f"0, 1200, 2070, 700.0, 0x0000000000000068, Active, Active, Active, {na}"])
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1200.0 and s["sm_max_mhz"] == 2070.0


def test_clock_summary_without_samples():
    assert _summary([]) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}


def _replay_with_oracle(g, rows, emitted, n_new, B, prompt_len, max_seq, adaptive):
    """Re-derives each round's block length and acceptance with the oracle."""
    gen, n, ema = 1, prompt_len, float(np.float32(B - 1))
    for row, e in zip(rows, emitted):
        cap = O.adaptive_block_cap(ema, B) if adaptive else B
        bl = O.block_len(cap, n_new, gen, max_seq, n)
        assert bl >= 1
        targets = [int(t) for t in g[gen:gen + bl]]          # the greedy target's rows
        a, out, finished = O.accept(row[:bl - 1], targets, eos_id=-1)
        assert not finished
        assert a + 1 == e, (gen, bl, a, e)
        assert out == targets[:e]
        if adaptive:
            ema = O.adaptive_ema_update(ema, a)
        gen += e
        n += e
    return gen, n


@pytest.mark.parametrize("adaptive", [False, True])
@pytest.mark.parametrize("n_new,max_seq", [(512, 4096), (100, 1024 + 57)])
def test_injected_schedule_follows_the_oracle_rules(adaptive, n_new, max_seq):
    B, prompt_len, vocab = 16, 1024, 151936
    g = np.random.default_rng(3).integers(0, vocab, size=n_new + B + 1)
    rows, emitted = bench.injected_schedule(g, n_new, B, prompt_len, max_seq, vocab, seed=11,
                                            adaptive=adaptive)
    assert len(rows) == len(emitted) > 0
    assert all(len(r) == B - 1 for r in rows)
    gen, n = _replay_with_oracle(g, rows, emitted, n_new, B, prompt_len, max_seq, adaptive)
    # the run ends exactly at the token budget or at the sequence capacity
    assert gen == n_new or n == max_seq
    assert n <= max_seq
    # a profile that both accepts whole blocks and stops early
    assert max(emitted) > 1 and min(emitted) < B


def test_injected_schedule_cuts_at_the_budget():
    # a budget a few tokens past a block: the last round's block is short
    B, vocab = 16, 1000
    g = np.arange(40) % vocab
    rows, emitted = bench.injected_schedule(g, 20, B, 8, 4096, vocab, seed=0)
    assert sum(emitted) == 20 - 1
    _replay_with_oracle(g, rows, emitted, 20, B, 8, 4096, False)
