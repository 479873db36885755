"""Pins of the oracle's masks, taps, acceptance, block length and INT4 format.

Hand-worked fixtures live in tests/golden/ with the passage they follow.
"""

import json
import os

import numpy as np
import pytest
import torch

from oracle import dflash_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- hc-mean tap

def test_hc_mean_hand_example():
    g = _golden("hc_mean_hand.json")
    row = np.array([g["row"]], dtype=np.float64)
    np.testing.assert_array_equal(O.hc_mean(row, g["hc"]), [g["mean"]])
    assert not np.array_equal(O.hc_mean(row, g["hc"]), [g["wrong_layout_mean"]])


def test_hc_mean_is_torch_unflatten_mean():
    x = np.random.default_rng(0).standard_normal((7, 4 * 32))
    ref = torch.from_numpy(x).unflatten(-1, (4, 32)).mean(-2).numpy()
    np.testing.assert_allclose(O.hc_mean(x, 4), ref, rtol=1e-14, atol=1e-15)


def test_hc_one_is_identity_and_concat_order():
    a = np.arange(6.0).reshape(2, 3)
    b = -np.arange(6.0).reshape(2, 3)
    np.testing.assert_array_equal(O.hc_mean(a, 1), a)
    np.testing.assert_array_equal(O.tap_concat([a, b], 1), np.concatenate([a, b], 1))


# ---------------------------------------------------------------- block mask

def _brute_force_visible(n, bl, window):
    """Enumerate (query, key) pairs from the set definition.

    keys: context positions 0..n-1 then block rows; a block row sees every
    block row, and a context position p when no window is set or p lies in
    the W positions just before the block start n.
    """
    ctx = list(range(n))
    vis = np.zeros((bl, n + bl), dtype=bool)
    for i in range(bl):
        for j, p in enumerate(ctx):
            if window == 0 or n - window <= p:
                vis[i, j] = True
        for j in range(bl):
            vis[i, n + j] = True
    return vis


@pytest.mark.parametrize("n", [0, 1, 5, 70])
@pytest.mark.parametrize("bl", [1, 2, 8])
@pytest.mark.parametrize("window", [0, 4, 64])
def test_block_mask_brute_force(n, bl, window):
    got = O.block_visible(list(range(n)), n, bl, window)
    np.testing.assert_array_equal(got, _brute_force_visible(n, bl, window))


def test_block_mask_window_covering_context_equals_no_window():
    for n in [0, 3, 64]:
        np.testing.assert_array_equal(O.block_visible(list(range(n)), n, 8, 64),
                                      O.block_visible(list(range(n)), n, 8, 0))


def test_causal_mask_brute_force():
    q = [5, 6, 7]
    k = list(range(8))
    got = O.causal_visible(q, k)
    for i, qp in enumerate(q):
        for j, kp in enumerate(k):
            assert got[i, j] == (kp <= qp)


# ---------------------------------------------------------------- acceptance

def test_accept_hand_cases():
    for c in _golden("accept_cases.json")["accept"]:
        a, emitted, finished = O.accept(c["draft"], c["target"], c["eos"])
        assert (a, emitted, finished) == (c["a"], c["emitted"], c["finished"]), c["name"]
        # accepted length (a + 1) bounds the emitted count
        assert 1 <= len(emitted) <= a + 1


def test_block_len_hand_cases():
    for c in _golden("accept_cases.json")["block_len"]:
        assert O.block_len(c["block"], c["max_new"], c["generated"], c["max_seq"],
                           c["pos"]) == c["bl"], c["name"]


def test_first_mismatch_brute_force():
    rng = np.random.default_rng(5)
    for _ in range(500):
        T = int(rng.integers(1, 9))
        y = rng.integers(0, 3, size=T).tolist()
        d = rng.integers(0, 3, size=T - 1).tolist()
        a = O.first_mismatch(d, y)
        # a is the largest k with d[0..k-1] == y[0..k-1]
        best = max(k for k in range(T) if d[:k] == y[:k])
        assert a == best


# ---------------------------------------------------------------- INT4 g64

def test_int4_pack_hand_example():
    g = _golden("int4_pack_hand.json")
    k = np.arange(64)
    w = ((k % 15 - 7) * 0.01).astype(np.float32)[None, :]
    packed, s = O.quantize_int4_g64(w)
    assert int(s[0, 0]) == g["scale_bits"]
    assert packed[0, :8].tolist() == g["first_bytes"]
    z, zs = O.quantize_int4_g64(np.zeros((1, 64), np.float32))
    assert set(z.ravel().tolist()) == {g["zero_group_byte"]} and int(zs[0, 0]) == 0


def test_int4_round_trip_bound_and_code_range():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((48, 256)) * 0.02).astype(np.float32)
    w[3, :64] = 0.0                              # an all-zero group
    packed, s_bits = O.quantize_int4_g64(w)
    deq = O.dequant_int4_g64(packed, s_bits)
    s = np.repeat(O.bf16_bits_to_f64(s_bits), 64, axis=1)
    err = np.abs(deq - w.astype(np.float64))
    assert np.all(err <= s / 2 + 1e-12)
    codes = np.round(deq / np.where(s > 0, s, 1)).astype(int)
    assert codes.min() >= -7 and codes.max() <= 7
    assert np.all(deq[3, :64] == 0)
    # dequantised values are exact multiples of the bf16 scale
    np.testing.assert_array_equal(deq, codes * s)


# ---------------------------------------------------------------- adaptive block

def test_adaptive_block_cap_hand_cases():
    cases = [(0.0, 16, 4), (1.49, 16, 4), (1.5, 16, 8), (4.49, 16, 8), (4.5, 16, 16),
             (15.0, 16, 16), (15.0, 8, 8), (0.0, 2, 2)]
    for ema, block, cap in cases:
        assert O.adaptive_block_cap(ema, block) == cap, (ema, block)


def test_adaptive_ema_is_the_halving_average():
    """ema_k = ema_{k-1}/2 + a_k/2 from block-1, checked in exact rationals
    over 20 rounds (every value is a dyadic rational fp32 holds exactly)."""
    from fractions import Fraction
    rng = np.random.default_rng(3)
    ema, exact = float(np.float32(15)), Fraction(15)
    for _ in range(20):
        a = int(rng.integers(0, 16))
        ema = O.adaptive_ema_update(ema, a)
        exact = exact / 2 + Fraction(a, 2)
        assert Fraction(ema) == exact
