"""Pins for the oracle's on-chip tile quantisation of the probabilities and of
dS: the backward's P^ (E4M3) and dS^ (E5M2) per 128x128 tile, and the
forward's one-pass P~ over several key tiles.

The project page ("Delta-Matching for reliable FP8 attention training",
section 01, "What changes in FP8?") puts every attention matmul on decoded
block-scaled FP8 operands: the backward's dV = P^T dO, dQ = sigma dS K and
dK = sigma dS^T Q use the quantised probabilities and the quantised dS, with
one FP32 scale per 128x128 tile (amax / FMAX; causally masked entries are not
part of a tile).  The forward quantises P~ = exp(S - running row max) per key
tile in one pass, so a later tile's amax is below one wherever its rows' maxima
sit below the running maximum, and partial sums are rescaled by
exp(m_old - m_new) when the maximum rises.

Each test below rebuilds those steps on its own from the definition: numpy for
the arithmetic, torch's float8 casts for the FP8 codes, libm's exp (the same
function the oracle calls) for the exponentials.  The inputs sit on coarse
binary grids so that every score and every dO^ V^T product is exact in FP64
whatever the summation order; the oracle and the emulation then take every
FP32 and FP8 rounding decision on identical values, and the tile-level
quantities must agree exactly.  A slip in the oracle (dV from unquantised P, a
dS amax over 128 x d, masked entries counted in a tile amax, a forward tile
amax fixed at one, quantising P~ after its rescale, the rescale on the wrong
side) changes codes and fails here.
"""
import math

import numpy as np
import pytest
import torch

import oracle

T = 128


def _grid(rng, shape, step, lim):
    """Values on the grid step * k, |value| <= lim: exact sums and products in FP64."""
    n = int(lim / step)
    return rng.integers(-n, n + 1, size=shape).astype(np.float64) * step


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _exp(a):
    """Elementwise libm exp (math.exp), the function the oracle's std::exp calls."""
    flat = np.asarray(a, dtype=np.float64).ravel()
    return np.array([math.exp(v) for v in flat]).reshape(np.shape(a))


def _qz_tile(x, valid, fmt):
    """One 128x128 tile quantised by the amax rule: returns (decoded, scale).
    x holds FP32 values; entries outside `valid` are absent (code 0)."""
    fmax = 448.0 if fmt == 0 else 57344.0
    dtype = torch.float8_e4m3fn if fmt == 0 else torch.float8_e5m2
    a = np.abs(x[valid]).max() if valid.any() else 0.0
    amax = np.float32(a)
    if not amax >= np.float32(2.0 ** -96):
        return np.zeros_like(x), 0.0
    s = np.float32(amax / np.float32(fmax))
    r = np.float32(np.float32(fmax) / amax)
    xr = np.where(valid, (x.astype(np.float32) * r), np.float32(0.0)).astype(np.float32)
    xr = np.clip(xr, -fmax, fmax)   # satfinite (torch's E4M3 cast is not saturating)
    dec = torch.from_numpy(xr).to(dtype).to(torch.float64).numpy()
    return dec * float(s), float(s)


# ------------------------------------------------------------------ backward
def _bwd_emulation(Q, K, V, dO, LSE, delta, sigma, causal):
    """P, P^, dS, dS^ per 128x128 tile and dQ, dK, dV for one (b, kv head)
    group of G query heads.  Q [G][N][d], K [N][d], V [N][dv], dO [G][N][dv]."""
    G, N, d = Q.shape
    Tn = (N + T - 1) // T
    out = {k: [] for k in ("P", "Ph", "dS", "dSh")}
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    diag = np.zeros((4, G, N))
    for h in range(G):
        S = sigma * (Q[h] @ K.T)                               # exact (grid inputs)
        vis = np.ones((N, N), bool) if not causal else np.tril(np.ones((N, N), bool))
        P = np.where(vis, _f32(_exp(np.where(vis, S, 0.0) - LSE[h][:, None])), 0.0)
        dP = dO[h] @ V.T                                        # exact (grid inputs)
        dS = np.where(vis, _f32(P * (dP - delta[h][:, None])), 0.0)
        Ph = np.zeros_like(P)
        dSh = np.zeros_like(dS)
        for qt in range(Tn):
            for kt in range(Tn):
                rs, cs = slice(qt * T, min(N, qt * T + T)), slice(kt * T, min(N, kt * T + T))
                v = vis[rs, cs]
                if not v.any():
                    continue
                Ph[rs, cs], _ = _qz_tile(P[rs, cs], v, 0)
                dSh[rs, cs], _ = _qz_tile(dS[rs, cs], v, 1)
        dV += Ph.T @ dO[h]
        dQ[h] = sigma * (dSh @ K)
        dK += sigma * (dSh.T @ Q[h])
        diag[:, h] = dS.sum(1), np.abs(dS).sum(1), dSh.sum(1), np.abs(dSh).sum(1)
        for key, val in (("P", P), ("Ph", Ph), ("dS", dS), ("dSh", dSh)):
            out[key].append(val)
    out = {k: np.stack(v) for k, v in out.items()}
    out.update(dQ=dQ, dK=dK, dV=dV, diag=diag)
    return out


@pytest.mark.parametrize("causal", [True, False])
def test_backward_tile_quantisation_matches_torch_cast_emulation(causal):
    """Two query and two key tiles (so one masked diagonal tile, one full
    off-diagonal tile and, non-causal, an upper tile), a ragged tail, two query
    heads of one kv head: P^, dS^ and every gradient against the emulation."""
    rng = np.random.default_rng(2024 + causal)
    G, N, d, dv = 2, 250, 16, 16
    sigma = 0.25                                                # 1/sqrt(16), exact
    Q = _grid(rng, (1, G, N, d), 0.125, 2.0)
    K = _grid(rng, (1, 1, N, d), 0.125, 2.0)
    V = _grid(rng, (1, 1, N, dv), 0.0625, 1.0)
    dO = _grid(rng, (1, G, N, dv), 2.0 ** -12, 2.0 ** -8)      # small like the workloads' dO
    # the stored LSE (FP32, from the exact forward) and an arbitrary delta: the
    # backward takes both as inputs, so any values pin its tile steps
    _, LSE = oracle.attn_fwd(Q, K, V, causal, sigma, oracle.EXACT)
    LSE = _f32(LSE)
    delta = _f32(rng.standard_normal((1, G, N)) * 2.0 ** -10)
    got = oracle.attn_bwd(Q, K, V, dO, LSE, delta, causal, sigma, oracle.GPU_CONTRACT,
                          want_diag=True, want_tiles=True)
    want = _bwd_emulation(Q[0], K[0, 0], V[0, 0], dO[0], LSE[0], delta[0], sigma, causal)
    # tile-level values: identical rounding decisions on identical inputs
    np.testing.assert_array_equal(got["Phat"][0], want["Ph"])
    np.testing.assert_array_equal(got["dS"][0], want["dS"])
    np.testing.assert_array_equal(got["dShat"][0], want["dSh"])
    # the quantisation really acted: P^ != P and dS^ != dS somewhere, masked entries zero
    assert np.abs(want["Ph"] - want["P"]).max() > 0 and np.abs(want["dSh"] - want["dS"]).max() > 0
    if causal:
        iu = np.triu_indices(N, 1)
        assert np.all(got["Phat"][0][:, iu[0], iu[1]] == 0)
    for key in ("dQ", "dK", "dV"):
        w = want[key] if key == "dQ" else want[key][None]
        np.testing.assert_allclose(got[key][0], w, rtol=0, atol=1e-12 * np.abs(w).max(), err_msg=key)
    np.testing.assert_allclose(got["diag"][:, 0], want["diag"], rtol=0,
                               atol=1e-12 * np.abs(want["diag"]).max())


def test_backward_pin_fails_on_planted_slips():
    """The emulation is sensitive to the slips it guards against: dV from the
    unquantised P, and a dS amax over 128 x d instead of 128 x 128, both move
    the results far beyond the 1e-12 the pin asks for."""
    rng = np.random.default_rng(7)
    G, N, d = 1, 256, 16
    sigma = 0.25
    Q = _grid(rng, (G, N, d), 0.125, 2.0)
    K = _grid(rng, (N, d), 0.125, 2.0)
    V = _grid(rng, (N, d), 0.0625, 1.0)
    dO = _grid(rng, (G, N, d), 2.0 ** -12, 2.0 ** -8)
    S = sigma * Q[0] @ K.T
    LSE = _f32(np.log(np.exp(np.where(np.tril(np.ones((N, N), bool)), S, -np.inf)).sum(1)))[None]
    delta = _f32(rng.standard_normal((G, N)) * 2.0 ** -10)
    ref = _bwd_emulation(Q, K, V, dO, LSE, delta, sigma, True)
    dV_unquantised = ref["P"][0].T @ dO[0]
    assert np.abs(dV_unquantised - ref["dV"]).max() > 1e-6 * np.abs(ref["dV"]).max()
    # dS tiles of query tile 1 quantised with one scale for the whole 128-row
    # strip (both key tiles) instead of one per 128x128 tile
    strip = ref["dS"][0][T:]
    wide, _ = _qz_tile(strip, np.tril(np.ones((N, N), bool))[T:], 1)
    assert np.abs(wide - ref["dSh"][0][T:]).max() > 0


# ------------------------------------------------------------------- forward
def _fwd_emulation(Q, K, V, sigma, causal):
    """One-pass forward for one query head: key tiles ascending, running max,
    P~ = fl32(exp(S - m_t)) quantised per 128x128 tile, l from the unquantised
    P~, the accumulator and l rescaled by exp(m_old - m_new).  Returns
    (O, LSE, per-tile amax of P~ [query tile][key tile])."""
    N = Q.shape[0]
    Tn = (N + T - 1) // T
    S = sigma * (Q @ K.T)
    vis = np.ones((N, N), bool) if not causal else np.tril(np.ones((N, N), bool))
    O = np.zeros((N, V.shape[1]))
    LSE = np.zeros(N)
    amaxes = np.zeros((Tn, Tn))
    for qt in range(Tn):
        rs = slice(qt * T, min(N, qt * T + T))
        rows = rs.stop - rs.start
        m = np.full(rows, -np.inf)
        l = np.zeros(rows)
        acc = np.zeros((rows, V.shape[1]))
        for kt in range(Tn):
            cs = slice(kt * T, min(N, kt * T + T))
            v = vis[rs, cs]
            if not v.any():
                continue
            St = np.where(v, S[rs, cs], -np.inf)
            m_new = np.maximum(m, St.max(1))
            pt = np.where(v, _f32(_exp(np.where(v, St, 0.0) - m_new[:, None])), 0.0)
            amaxes[qt, kt] = pt[v].max()
            ph, _ = _qz_tile(pt, v, 0)
            alpha = _exp(m - m_new)                     # 0 on the first tile (exp(-inf))
            l = alpha * l + pt.sum(1)
            acc = alpha[:, None] * acc + ph @ V[cs]
            m = m_new
        O[rs] = acc / l[:, None]
        LSE[rs] = m + np.log(l)
    return O, LSE, amaxes


def _planted_scores(rng, N, d, shifts):
    """Q, K on a grid whose scores put each row's maximum over key tile 1 at
    shifts[row] (in score units) relative to its maximum over key tile 0:
    channel 0 of every key is a per-tile anchor, the other channels are small
    noise that moves no maximum."""
    Q = np.zeros((N, d))
    K = _grid(rng, (N, d), 2.0 ** -6, 2.0 ** -3)
    Q[:, 1:] = _grid(rng, (N, d - 1), 2.0 ** -6, 2.0 ** -3)
    K[:, 0] = 0.0
    K[0, :] = 0.0
    K[T, :] = 0.0
    K[0, 0] = 8.0             # anchor key of tile 0
    K[T, 0] = 8.0             # anchor key of tile 1
    Q[:, 0] = 1.0
    # row i sees the tile-1 anchor shifted by shifts[i]: carry it in channel 1
    K[0, 1] = 0.0
    K[T, 1] = 1.0
    Q[:, 1] = shifts
    return Q, K


@pytest.mark.parametrize("rise", [False, True])
def test_one_pass_forward_two_tiles_vs_torch_cast(rise):
    """Two key tiles, non-causal, V = identity (so O is the effective
    probability matrix P^fwd itself).  rise=False: every row's maximum over
    tile 1 lies below its tile-0 maximum by a planted gap, so tile 1's P~ amax
    is exp(-smallest gap) < 1 in closed form.  rise=True: the maximum rises in
    tile 1 for some rows, so tile 0's quantised partial sums must be rescaled
    by exp(m_0 - m_1) after they were quantised."""
    rng = np.random.default_rng(99 + rise)
    N, d = 256, 8
    sigma = 0.5
    gaps = _grid(rng, (N,), 0.25, 3.0)
    gaps = -(np.abs(gaps) + 0.5) if not rise else gaps       # score units before sigma
    Q, K = _planted_scores(rng, N, d, gaps)
    V = np.eye(N)
    O, LSE = oracle.attn_fwd(Q[None, None], K[None, None], V[None, None], False, sigma,
                             oracle.QUANT_P_FWD | oracle.ROUND32)
    Ow, LSEw, amaxes = _fwd_emulation(Q, K, V, sigma, False)
    # the scores are exact, so the maxima are exactly the anchors
    S = sigma * Q @ K.T
    np.testing.assert_array_equal(S[:, :T].max(1), sigma * 8.0 + 0 * gaps)
    if not rise:
        assert np.all(S[:, T:].max(1) == sigma * (8.0 + gaps))
        # tile 1's amax in closed form, exp(-sigma * smallest gap) < 1 for the query tiles
        for qt in range(2):
            g = -gaps[qt * T:(qt + 1) * T].max()
            assert amaxes[qt, 1] == np.float32(math.exp(-sigma * g)) < 1.0
    else:
        assert np.any(gaps > 0) and np.any(gaps < 0)
    np.testing.assert_allclose(O[0, 0], Ow, rtol=0, atol=1e-13)
    np.testing.assert_allclose(LSE[0, 0], LSEw, rtol=1e-15, atol=1e-14)
    # O = P^fwd: its tile-1 block is the tile's decoded codes divided by l
    # (the maximum never moved); with amax < 1 those codes differ from the
    # ones an amax fixed at one would give
    if not rise:
        l = np.exp(LSEw - sigma * 8.0)
        used = O[0, 0][:, T:] * l[:, None]
        pt1 = _f32(_exp(S[:, T:] - sigma * 8.0)).astype(np.float32)
        fixed_one = torch.from_numpy(pt1 * np.float32(448.0)).to(torch.float8_e4m3fn).to(
            torch.float64).numpy() * float(np.float32(1.0) / np.float32(448.0))
        assert np.abs(used - fixed_one).max() > 1e-6


def test_one_pass_forward_causal_multi_tile_vs_emulation():
    """Causal, three query/key tiles with a ragged tail, random grid scores:
    every tile's running-max rescale and amax as in the emulation."""
    rng = np.random.default_rng(5)
    N, d = 300, 16
    sigma = 0.25
    Q = _grid(rng, (N, d), 0.25, 3.0)
    K = _grid(rng, (N, d), 0.25, 3.0)
    K[200:] *= 1.5           # larger scores in the last tile: the maximum rises late
    V = _grid(rng, (N, 12), 0.125, 2.0)
    O, LSE = oracle.attn_fwd(Q[None, None], K[None, None], V[None, None], True, sigma,
                             oracle.QUANT_P_FWD | oracle.ROUND32)
    Ow, LSEw, amaxes = _fwd_emulation(Q, K, V, sigma, True)
    # the running maximum rises in the last key tile for some rows of the last query tile
    S = sigma * Q @ K.T
    assert np.any(S[256:, 256:].max(1) > np.where(np.tril(np.ones((N, N), bool)), S, -np.inf)[256:, :256].max(1))
    np.testing.assert_allclose(O[0, 0], Ow, rtol=0, atol=1e-12 * np.abs(Ow).max())
    np.testing.assert_allclose(LSE[0, 0], LSEw, rtol=1e-15, atol=1e-13)
