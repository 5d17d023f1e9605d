"""Pins for the oracle's FP8 codec and tile quantiser.

The pages name the formats (E4M3 forward, E5M2 backward -- "Delta-Matching
Reports FP8 LLM Training Parity...", section "The correction preserves FP8
through attention") and block scales (project page section 01, "What changes
in FP8?").  The codec is pinned against (a) the OCP OFP8 reference values in
tests/golden/ofp8_reference_values.txt, (b) torch's independent CPU float8
casts, exhaustively for decode and on every representable value, every
midpoint and random values for encode, and (c) saturation, which torch does
not implement, against the closed-form largest finite value.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ofp8_reference_values.txt")
TORCH_DT = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}
NAMES = {"E4M3": oracle.E4M3, "E5M2": oracle.E5M2}


def _torch_decode(codes, fmt):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(TORCH_DT[fmt]).to(torch.float64).numpy()


def _torch_encode(x, fmt):
    return torch.from_numpy(np.asarray(x, np.float32)).to(TORCH_DT[fmt]).view(torch.uint8).numpy()


def test_golden_values():
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        name, code, val = line.split()
        fmt, code = NAMES[name], int(code, 16)
        got = oracle.fp8_decode(np.array([code], np.uint8), fmt)[0]
        if val == "nan":
            assert np.isnan(got)
        else:
            want = float(val)
            assert got == want and np.signbit(got) == np.signbit(want), (name, hex(code), got, want)
            if np.isfinite(want):
                assert oracle.fp8_encode(np.array([want], np.float32), fmt)[0] == code


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_decode_exhaustive_vs_torch(fmt):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.fp8_decode(codes, fmt)
    ref = _torch_decode(codes, fmt)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_grid_midpoints_random_vs_torch(fmt):
    fmax = oracle.FMAX[fmt]
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.fp8_decode(codes, fmt)
    fin = np.isfinite(vals)
    # every finite value round-trips to its own code (both signs of zero)
    enc = oracle.fp8_encode(vals[fin].astype(np.float32), fmt)
    assert np.array_equal(enc, codes[fin])
    # midpoints between neighbours: round half to even, as torch does
    pos = np.unique(vals[fin & (vals >= 0)])
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[1:] + pos[:-1]) / 2)  # exact in fp32
    xs = np.concatenate([mids, -mids])
    assert np.array_equal(oracle.fp8_encode(xs, fmt), _torch_encode(xs, fmt))
    # random in-range values, log-uniform over the whole range incl. subnormals
    rng = np.random.default_rng(1)
    mag = np.exp(rng.uniform(np.log(2.0 ** -24), np.log(fmax), 200_000))
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    x = x[np.abs(x) <= fmax]
    assert np.array_equal(oracle.fp8_encode(x, fmt), _torch_encode(x, fmt))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_saturates(fmt):
    fmax = oracle.FMAX[fmt]
    top = oracle.fp8_encode(np.array([fmax], np.float32), fmt)[0]
    big = np.array([np.nextafter(np.float32(fmax), np.float32(np.inf)), fmax * 1.07, fmax * 1.2,
                    3e38, np.inf], np.float32)
    assert np.all(oracle.fp8_encode(big, fmt) == top)
    assert np.all(oracle.fp8_encode(-big, fmt) == (top | 0x80))
    nan = oracle.fp8_encode(np.array([np.nan], np.float32), fmt)
    assert np.isnan(oracle.fp8_decode(nan, fmt)[0])


def _torch_qz(x, fmt):
    """Per-tile amax quantiser written with torch primitives for an independent check."""
    fmax = np.float32(oracle.FMAX[fmt])
    amax = np.float32(np.max(np.abs(x)))
    if not amax >= np.float32(2.0 ** -96):
        return np.zeros(x.shape, np.uint8), np.float32(0)
    s = np.float32(amax / fmax)
    r = np.float32(fmax / amax)
    y = (x * r).astype(np.float32)
    y = np.clip(y, -fmax, fmax)  # values can exceed fmax by < 1 ulp; torch does not saturate
    return _torch_encode(y, fmt), s


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("N,d", [(256, 64), (200, 128), (77, 32), (1, 16)])
def test_quantize_tiles_vs_torch(fmt, N, d):
    rng = np.random.default_rng(N * d + fmt)
    x = (rng.standard_normal((2, 3, N, d)) * np.exp(rng.uniform(-8, 8, (2, 3, N, 1)))).astype(np.float32)
    x[0, 0, :min(N, 128)] = 0.0                  # an all-zero tile
    if N > 128:
        x[0, 1, 128:] *= np.float32(2.0 ** -110)  # a tile below the flush threshold
    codes, scales = oracle.quantize(x, fmt)
    T = (N + 127) // 128
    assert scales.shape == (2, 3, T)
    for b in range(2):
        for h in range(3):
            for t in range(T):
                tile = x[b, h, t * 128:(t + 1) * 128]
                c_ref, s_ref = _torch_qz(tile, fmt)
                assert scales[b, h, t] == s_ref
                assert np.array_equal(codes[b, h, t * 128:(t + 1) * 128], c_ref)
    assert scales[0, 0, 0] == 0 and not codes[0, 0, :min(N, 128)].any()
    if N > 128:
        assert scales[0, 1, 1] == 0


@pytest.mark.parametrize("fmt,rel", [(oracle.E4M3, 2.0 ** -4), (oracle.E5M2, 2.0 ** -3)])
def test_quantize_error_bound(fmt, rel):
    """|x^ - x| <= half a step: rel*|x| for normals, plus the subnormal half-step, of the scaled grid."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((1, 2, 384, 64)).astype(np.float32)
    codes, scales = oracle.quantize(x, fmt)
    xh = oracle.dequantize(codes, scales, fmt)
    s = np.repeat(scales, 128, axis=2)[:, :, :384, None].astype(np.float64)
    sub_half = {oracle.E4M3: 2.0 ** -10, oracle.E5M2: 2.0 ** -17}[fmt]
    bound = rel * np.abs(x) * (1 + 1e-6) + s * sub_half * (1 + 1e-6) + 1e-7 * np.abs(x)
    assert np.all(np.abs(xh - x) <= bound)
    # the tile's largest magnitude lands exactly on the largest code
    for t in range(3):
        tile = np.abs(x[0, 0, t * 128:(t + 1) * 128])
        i = np.unravel_index(np.argmax(tile), tile.shape)
        assert abs(oracle.fp8_decode(codes[0, 0, t * 128 + i[0], i[1]:i[1] + 1], fmt)[0]) == oracle.FMAX[fmt]
