"""Pins of the oracle's primitives against library routines and closed forms.

Each test checks an oracle function against something other than itself: a
torch library routine (F.rms_norm, F.silu, scaled_dot_product_attention), an
independent mathematical formulation (RoPE as a complex rotation), or an
invariant the definition implies (RoPE's relative-position property).
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import dflash_oracle as O

RNG = np.random.default_rng(1234)


def test_rms_norm_matches_torch():
    x = RNG.standard_normal((5, 3, 64))
    w = RNG.standard_normal(64)
    ref = F.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, w, 1e-6), ref, rtol=1e-13, atol=1e-13)


def test_silu_matches_torch():
    x = RNG.standard_normal(1000) * 6
    np.testing.assert_allclose(O.silu(x), F.silu(torch.from_numpy(x)).numpy(),
                               rtol=1e-13, atol=1e-15)


def test_linear_layout_is_nn_linear():
    x = RNG.standard_normal((3, 7))
    w = RNG.standard_normal((5, 7))
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(w)).numpy()
    np.testing.assert_allclose(O.linear(x, w), ref, rtol=1e-13, atol=1e-13)


def _rope_complex(x, positions, theta):
    """RoPE as a complex rotation of the pairs (x_i, x_{i+d/2})."""
    d = x.shape[-1]
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    i = np.arange(half)
    freq = 1.0 / (theta ** (2.0 * i / d))
    rot = np.exp(1j * np.asarray(positions, dtype=np.float64)[:, None, None] * freq)
    zr = z * rot
    return np.concatenate([zr.real, zr.imag], axis=-1)


@pytest.mark.parametrize("d", [4, 64, 128])
def test_rope_is_complex_rotation_of_half_pairs(d):
    x = RNG.standard_normal((6, 3, d))
    pos = [0, 1, 7, 100, 4097, 16383]
    # angles up to 16383 rad: the two formulations round them differently
    np.testing.assert_allclose(O.rope_rotate_half(x, pos, 1e6), _rope_complex(x, pos, 1e6),
                               rtol=1e-9, atol=1e-9)


def test_rope_position_zero_is_identity_and_norm_preserving():
    x = RNG.standard_normal((1, 2, 64))
    np.testing.assert_array_equal(O.rope_rotate_half(x, [0], 1e6), x)
    y = O.rope_rotate_half(np.repeat(x, 3, 0), [5, 900, 12000], 1e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1),
                               np.repeat(np.linalg.norm(x, axis=-1), 3, 0), rtol=1e-12)


def test_rope_scores_depend_only_on_relative_position():
    q = RNG.standard_normal((1, 1, 128))
    k = RNG.standard_normal((1, 1, 128))
    s = []
    for m, n in [(10, 3), (1010, 1003), (16000, 15993)]:
        qm = O.rope_rotate_half(q, [m], 1e6)
        kn = O.rope_rotate_half(k, [n], 1e6)
        s.append(float(np.sum(qm * kn)))
    np.testing.assert_allclose(s, s[0], rtol=1e-9)


def _sdpa_ref(q, k, v, visible, scale):
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]     # [1, Hq, Tq, d]
    kt = torch.from_numpy(k).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).permute(1, 0, 2)[None]
    out = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(visible),
                                         scale=scale, enable_gqa=True)
    return out[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("n_q,n_kv", [(4, 2), (32, 8), (4, 4)])
def test_attention_matches_sdpa_gqa_causal(n_q, n_kv):
    Tq, Tk, d = 5, 9, 16
    q = RNG.standard_normal((Tq, n_q, d))
    k = RNG.standard_normal((Tk, n_kv, d))
    v = RNG.standard_normal((Tk, n_kv, d))
    vis = O.causal_visible(range(Tk - Tq, Tk), range(Tk))
    np.testing.assert_allclose(O.attention(q, k, v, vis, 1 / math.sqrt(d)),
                               _sdpa_ref(q, k, v, vis, 1 / math.sqrt(d)), rtol=1e-11, atol=1e-12)


def test_attention_masked_keys_equal_dropped_keys():
    """Masking a key must be the same as removing it from the key set."""
    q = RNG.standard_normal((3, 4, 8))
    k = RNG.standard_normal((7, 2, 8))
    v = RNG.standard_normal((7, 2, 8))
    keep = np.array([1, 0, 1, 1, 0, 0, 1], dtype=bool)
    vis = np.tile(keep, (3, 1))
    full = O.attention(q, k, v, vis, 0.3)
    dropped = O.attention(q, k[keep], v[keep], np.ones((3, keep.sum()), bool), 0.3)
    np.testing.assert_allclose(full, dropped, rtol=1e-13, atol=1e-14)


def test_attention_zero_keys_closed_form():
    """n zero keys with zero values: out = out_blockonly * Zb / (Zb + n e^{-m})."""
    q = RNG.standard_normal((2, 1, 8))
    kb = RNG.standard_normal((3, 1, 8))
    vb = RNG.standard_normal((3, 1, 8))
    n0 = 5
    k = np.concatenate([np.zeros((n0, 1, 8)), kb])
    v = np.concatenate([np.zeros((n0, 1, 8)), vb])
    out = O.attention(q, k, v, np.ones((2, n0 + 3), bool), 1.0)
    s = q[:, 0, :] @ kb[:, 0, :].T
    m = np.maximum(s.max(1, keepdims=True), 0.0)
    zb = np.exp(s - m).sum(1, keepdims=True)
    ob = (np.exp(s - m) @ vb[:, 0, :]) / zb
    expect = ob * zb / (zb + n0 * np.exp(-m))
    np.testing.assert_allclose(out[:, 0, :], expect, rtol=1e-12, atol=1e-14)


def test_argmax_ties_go_to_lowest_index():
    row = np.array([0.0, 3.0, 1.0, 3.0, 3.0])
    assert O.argmax_lowest(row) == 1
    assert int(torch.argmax(torch.tensor([0.0, 3.0, 1.0, 3.0]))) == 1


def test_bf16_rounding_matches_torch():
    x = np.concatenate([RNG.standard_normal(20000).astype(np.float32) * 0.02,
                        np.float32([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0,
                                    65504.0, 1e-30])])
    ours = O.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
