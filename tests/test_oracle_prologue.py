"""Pins for the oracle's attention-input prologue (RMSNorm with channel gains,
rotary embedding), checked against properties that hold independently of how
the oracle writes them: textbook values of the rotary table, the rotation as
complex multiplication, the relative-position property of rotary embedding,
the unit RMS and scale invariance of RMSNorm, and the per-channel action of
the gains ("Delta-Matching for reliable FP8 attention training", section 02
on the query/key RMSNorm gains, section 05 on QK normalisation and RoPE)."""
import math

import numpy as np
import pytest

import oracle


def _x(shape, seed=0, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def test_rope_table_textbook_values():
    # d = 8, base 10^4: the frequencies are 10^0, 10^-1, 10^-2, 10^-3
    c, s = oracle.rope_table(3, 8)
    assert c.shape == s.shape == (3, 4)
    np.testing.assert_array_equal(c[0], np.ones(4))
    np.testing.assert_array_equal(s[0], np.zeros(4))
    # cos 1, sin 1, cos 0.1, sin 0.01, cos 0.002 to 16 digits
    assert c[1, 0] == pytest.approx(0.5403023058681398, rel=1e-15)
    assert s[1, 0] == pytest.approx(0.8414709848078965, rel=1e-15)
    assert c[1, 1] == pytest.approx(0.9950041652780258, rel=1e-15)
    assert s[1, 2] == pytest.approx(0.009999833334166665, rel=1e-13)
    assert c[2, 3] == pytest.approx(0.9999980000006667, rel=1e-15)


def test_rope_is_rotation_of_complex_pairs():
    B, H, N, d = 1, 2, 9, 16
    x = _x((B, H, N, d), 1)
    y0 = oracle.qk_prologue(x, rope=False)
    y1 = oracle.qk_prologue(x, rope=True)
    h = d // 2
    n = np.arange(N)[:, None]
    i = np.arange(h)[None, :]
    theta = n * (10000.0 ** (-2.0 * i / d))
    z = (y0[..., :h] + 1j * y0[..., h:]) * np.exp(1j * theta)
    np.testing.assert_allclose(y1[..., :h], z.real, rtol=0, atol=1e-13)
    np.testing.assert_allclose(y1[..., h:], z.imag, rtol=0, atol=1e-13)


def test_rope_position_zero_is_identity_and_norms_are_kept():
    x = _x((2, 1, 5, 32), 2)
    y0 = oracle.qk_prologue(x, rope=False)
    y1 = oracle.qk_prologue(x, rope=True)
    np.testing.assert_array_equal(y1[:, :, 0], y0[:, :, 0])
    h = 16
    np.testing.assert_allclose(y1[..., :h] ** 2 + y1[..., h:] ** 2, y0[..., :h] ** 2 + y0[..., h:] ** 2,
                               rtol=1e-13, atol=1e-15)


def test_rope_scores_depend_on_relative_position_only():
    # <rot(q, n), rot(k, m)> is a function of n - m: shifting both positions by
    # the same amount leaves every score unchanged.
    d, N, shift = 64, 40, 17
    base = _x((1, 1, 1, d), 3)
    other = _x((1, 1, 1, d), 4)
    q = np.repeat(base, N, axis=2)
    k = np.repeat(other, N, axis=2)
    rq = oracle.qk_prologue(q)[0, 0]
    rk = oracle.qk_prologue(k)[0, 0]
    for n, m in [(3, 1), (10, 10), (5, 12)]:
        assert rq[n] @ rk[m] == pytest.approx(rq[n + shift] @ rk[m + shift], rel=1e-11, abs=1e-12)
    # and it does depend on the offset
    assert abs(rq[3] @ rk[1] - rq[3] @ rk[2]) > 1e-3


def test_rmsnorm_unit_rms_scale_invariance_and_eps():
    x = _x((1, 3, 7, 128), 5, scale=3.0)
    y = oracle.qk_prologue(x, eps=0.0, rope=False)
    np.testing.assert_allclose(np.mean(y ** 2, axis=-1), 1.0, rtol=1e-13)
    y2 = oracle.qk_prologue(x * np.float32(0.125), eps=0.0, rope=False)
    np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-14)
    # rows far below eps: y -> x / sqrt(eps)
    tiny = _x((1, 1, 3, 64), 6, scale=1e-6)
    yt = oracle.qk_prologue(tiny, eps=1.0, rope=False)
    np.testing.assert_allclose(yt, tiny.astype(np.float64), rtol=1e-9)


def test_gains_scale_channels():
    d = 128
    g = np.ones(d)
    g[7] = 5.4
    g[:3] = 3.0
    x = _x((2, 2, 6, d), 7)
    y0 = oracle.qk_prologue(x, rope=False)
    yg = oracle.qk_prologue(x, gain=g, rope=False)
    np.testing.assert_allclose(yg, y0 * g, rtol=1e-15, atol=0)


def test_quantized_prologue_matches_tile_quantiser():
    x = _x((1, 2, 300, 64), 8)
    codes, scales, y = oracle.qk_prologue_quantized(x)
    c2, s2 = oracle.quantize(y.astype(np.float32), oracle.E4M3)
    np.testing.assert_array_equal(codes, c2)
    np.testing.assert_array_equal(scales, s2)
    # decoded values within half an E4M3 step (2^-4 relative, plus the FP32
    # rounding of y) of y, or half a subnormal step
    dec = oracle.dequantize(codes, scales, oracle.E4M3)
    s_row = np.repeat(scales, 128, axis=2)[:, :, :300, None].astype(np.float64)
    assert np.all(np.abs(dec - y) <= np.abs(y) * (2.0 ** -4 + 1e-6) + s_row * 2.0 ** -10 + 1e-12)


def test_bad_arguments():
    with pytest.raises(ValueError):
        oracle.qk_prologue(np.zeros((1, 1, 2, 5), np.float32))  # odd d
    with pytest.raises(ValueError):
        oracle.rope_table(4, 7)
    assert math.isfinite(oracle.ROPE_BASE)
