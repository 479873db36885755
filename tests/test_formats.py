"""Number-format facts the GPU paths rely on, checked exhaustively on the CPU.

The dense INT4 paths (window ingest of an INT4 drafter, prompt prefill of an
INT4 target) dequantise each weight to f16 before the tcgen05 GEMM, which
takes one operand type for both sides: `f16(float(code) * scale)` with a
4-bit code in [-8, 7] and a bf16 group scale (the group-64 INT4 format of the
DFlash2 drafter commit, "Mference" page).  The claim is that this loses
nothing for every scale a real weight group produces, so the dense path and
the round's in-register bf16 dequantisation see the same weights.  These
tests model the kernel's arithmetic (an fp32 product, then one
round-to-nearest-even conversion to f16) over every positive finite bf16
scale and every code.
"""

import numpy as np

from oracle import dflash_oracle as O

CODES = np.arange(-8, 8, dtype=np.int32)
LO, HI = 2.0 ** -17, 8160.0   # the exact range of the scale (both ends bf16 values)


def _all_scales():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)     # every positive finite bf16
    return (bits << 16).view(np.float32)


def _products():
    s = _all_scales()
    with np.errstate(over="ignore"):
        p32 = CODES[None, :].astype(np.float32) * s[:, None]
    p64 = CODES[None, :].astype(np.float64) * s[:, None].astype(np.float64)
    return s, p32, p64


def test_code_times_bf16_scale_is_exact_in_fp32():
    # a 4-bit integer times an 8-bit significand needs at most 11 bits
    _, p32, p64 = _products()
    fin = np.isfinite(p32)
    assert fin[_all_scales() <= 2.0 ** 120].all()
    np.testing.assert_array_equal(p32[fin].astype(np.float64), p64[fin])


def test_f16_dequant_exact_inside_the_scale_range():
    s, p32, p64 = _products()
    with np.errstate(over="ignore"):
        h = p32.astype(np.float16).astype(np.float64)
    exact = h == p64
    inside = (s >= LO) & (s <= HI)
    assert inside.sum() > 0 and exact[inside].all()
    # both ends are tight: the next bf16 scale outside the range loses a code
    below = s[(s < LO)].max()
    above = s[(s > HI)].min()
    assert not exact[s == below].all() and not exact[s == above].all()
    # above the range the loss is overflow of the largest codes (8 * s > 65504)
    with np.errstate(over="ignore"):
        assert np.isinf(np.float16(np.float32(-8.0) * above))


def test_dequantised_f16_equals_the_oracle_dequantisation():
    # weights drawn as the workloads draw them (N(0, 0.02), plus wide groups
    # at the range's ends): the oracle's exact dequantisation survives f16
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    w[0, :64] *= 1e-2
    w[1, :64] *= 3e3
    w[2, :64] = 0.0
    packed, s_bits = O.quantize_int4_g64(w)
    s = O.bf16_bits_to_f64(s_bits)
    assert ((s == 0) | ((s >= LO) & (s <= HI))).all()
    deq = O.dequant_int4_g64(packed, s_bits)
    np.testing.assert_array_equal(deq.astype(np.float16).astype(np.float64), deq)


def _wide_fp32(n, seed, lo_exp, hi_exp):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(1.0, 2.0, n)
    exp = rng.integers(lo_exp, hi_exp, n)
    sign = rng.choice([-1.0, 1.0], n)
    return (sign * mant * np.exp2(exp)).astype(np.float32)


def test_bf16_hi_lo_planes_carry_16_bits():
    # GEMM inputs go in as hi = bf16(v), lo = bf16(v - hi): the fp32
    # difference is exact and hi + lo is within 2^-16 of v (two roundings
    # of an 8-bit significand), which is what puts the GEMM-input share of
    # the logits' error near 2e-5 instead of the ~1 % of plain bf16 inputs
    import torch
    v = _wide_fp32(200_000, 3, -60, 60)
    hi = torch.from_numpy(v).to(torch.bfloat16).float().numpy()
    r = v - hi                                              # fp32, as the kernel
    np.testing.assert_array_equal(r.astype(np.float64), v.astype(np.float64) - hi.astype(np.float64))
    lo = torch.from_numpy(r).to(torch.bfloat16).float().numpy()
    err = np.abs(v.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert (err <= 2.0 ** -16 * np.abs(v.astype(np.float64))).all()
    # plain bf16 is 2^8 times coarser: the bound is reached, not loose
    rel_hi = np.abs(v.astype(np.float64) - hi) / np.abs(v.astype(np.float64))
    assert rel_hi.max() > 2.0 ** -9.5 and (err / np.abs(v.astype(np.float64))).max() > 2.0 ** -18


def test_f16_hi_lo_planes_inside_their_range():
    # the INT4 dense paths carry activations as f16 hi/lo: within 2^-22
    # relative plus the subnormal floor 2^-25, for |v| up to 65504
    v = _wide_fp32(200_000, 4, -12, 16)
    v = v[np.abs(v) <= 65504]
    hi = v.astype(np.float16).astype(np.float32)
    r = v - hi
    np.testing.assert_array_equal(r.astype(np.float64), v.astype(np.float64) - hi.astype(np.float64))
    lo = r.astype(np.float16).astype(np.float64)
    err = np.abs(v.astype(np.float64) - hi.astype(np.float64) - lo)
    assert (err <= 2.0 ** -22 * np.abs(v.astype(np.float64)) + 2.0 ** -25).all()


def test_int4_code_to_f16_bit_tricks():
    """The INT4 GEMM turns codes into f16 without conversions: an even
    nibble u in the low mantissa bits, 0x6400 | u, is the f16 1024 + u, and
    1024 + u - 1032 = u - 8; an odd nibble left in bits 4..7, 0x6400 | 16 u,
    is 1024 + 16 u, and (1024 + 16 u) / 16 - 72 = u - 8.  Every step is exact
    in f16 (so one rounding, as in a fused multiply-add, changes nothing)."""
    for u in range(16):
        lo = np.array([0x6400 | u], dtype=np.uint16).view(np.float16)[0]
        hi = np.array([0x6400 | (u << 4)], dtype=np.uint16).view(np.float16)[0]
        assert float(lo) == 1024 + u
        assert float(hi) == 1024 + 16 * u
        assert np.float16(lo - np.float16(1032)) == u - 8
        prod = np.float16(hi * np.float16(0.0625))      # exact: a power-of-two scale
        assert float(prod) == 64 + u
        assert np.float16(prod + np.float16(-72)) == u - 8
        assert float(hi) * 0.0625 - 72 == u - 8           # the unrounded fma value
