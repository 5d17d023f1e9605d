"""Pins for the oracle's attention forward, delta and backward.

What the pages fix, and the test that holds the oracle to it:

* definition of attention and its backward (project page "Delta-Matching for
  reliable FP8 attention training", section 01, "Write down softmax
  backward"): exact mode against torch's scaled-dot-product attention and
  autograd in FP64 (a library), and against central finite differences of
  L = sum(dO * O) on tiny inputs (brute force);
* the saved-output shortcut sum_j P dP = <dO, O> (section 01, "Why can we reuse
  the forward output?");
* shift invariance and the zero row sum of dS (section 01);
* the matched correction restores the zero row sum under quantisation
  (section 03), and the stale one does not;
* the stale residual splits into a probability term and a dO term (section
  01, "Separate the two mismatches"), each vanishing in its special case;
  matching only dO leaves the probability term (section 03);
* dS_stale = dS_centered + eps * P (section 02);
* GQA: the kv head's gradients are the sum over its query heads;
* the one-pass quantised forward: a single key tile reproduces a torch-cast
  emulation, O = Pfwd V exactly, rescaling across tiles keeps O within the
  FP8 error of exact attention.
"""
import numpy as np
import pytest
import torch

import oracle

EX = oracle.EXACT


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _case(B=1, Hq=2, Hkv=1, N=40, d=8, seed=0, qscale=1.0, dv=None):
    dv = d if dv is None else dv
    Q = _rand((B, Hq, N, d), seed, qscale)
    K = _rand((B, Hkv, N, d), seed + 1, qscale)
    V = _rand((B, Hkv, N, dv), seed + 2)
    dO = _rand((B, Hq, N, dv), seed + 3)
    return Q, K, V, dO


def _torch_attn(Q, K, V, causal, sigma=None):
    G = Q.shape[1] // K.shape[1]
    q = torch.tensor(Q, dtype=torch.float64, requires_grad=True)
    k = torch.tensor(K, dtype=torch.float64, requires_grad=True)
    v = torch.tensor(V, dtype=torch.float64, requires_grad=True)
    kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=causal, scale=sigma)
    return q, k, v, o


def _exact_all(Q, K, V, dO, causal, mode=oracle.DELTA_MATCHED, sigma=0.0):
    O, LSE = oracle.attn_fwd(Q, K, V, causal, sigma, EX)
    delta = oracle.attn_delta(Q, K, V, dO, LSE, mode, dO=dO, O=O, causal=causal, sigma=sigma, flags=EX)
    g = oracle.attn_bwd(Q, K, V, dO, LSE, delta, causal, sigma, EX, want_diag=True, want_tiles=True)
    return O, LSE, delta, g


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(1, 2, 1, 40, 8), (2, 4, 2, 150, 16), (1, 1, 1, 1, 4), (1, 2, 2, 257, 32),
                                   (1, 2, 1, 24, 256)])
def test_exact_matches_torch(causal, shape):
    B, Hq, Hkv, N, d = shape
    Q, K, V, dO = _case(B, Hq, Hkv, N, d, seed=N)
    O, LSE, delta, g = _exact_all(Q, K, V, dO, causal)
    q, k, v, o = _torch_attn(Q, K, V, causal)
    o.backward(torch.tensor(dO))
    np.testing.assert_allclose(O, o.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dQ"], q.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(g["dK"], k.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(g["dV"], v.grad.numpy(), rtol=1e-10, atol=1e-11)
    # LSE against its definition via torch.logsumexp
    s = torch.tensor(Q) @ torch.tensor(K).repeat_interleave(Hq // Hkv, 1).transpose(-1, -2) / np.sqrt(d)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(LSE, torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [(1, 2, 1, 40, 24, 16), (2, 4, 2, 150, 16, 40), (1, 2, 1, 20, 192, 128)])
def test_value_width_differs_matches_torch(causal, shape):
    """Heads whose value dimension differs from the query/key one (multi-head
    latent attention shapes): exact mode against torch's attention and
    autograd, and the saved-output shortcut sum_j P dP = <dO, O> over dv."""
    B, Hq, Hkv, N, d, dv = shape
    Q, K, V, dO = _case(B, Hq, Hkv, N, d, seed=N + d, dv=dv)
    O, LSE, delta, g = _exact_all(Q, K, V, dO, causal)
    assert O.shape == (B, Hq, N, dv) and g["dV"].shape == V.shape and g["dK"].shape == K.shape
    q, k, v, o = _torch_attn(Q, K, V, causal)
    o.backward(torch.tensor(dO))
    np.testing.assert_allclose(O, o.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(g["dQ"], q.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(g["dK"], k.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(g["dV"], v.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(delta, np.sum(dO * O, axis=-1), rtol=1e-10, atol=1e-12)


def test_explicit_sigma_matches_torch():
    Q, K, V, dO = _case(N=30, d=8, seed=3)
    O, _ = oracle.attn_fwd(Q, K, V, True, 0.3, EX)
    _, _, _, o = _torch_attn(Q, K, V, True, sigma=0.3)
    np.testing.assert_allclose(O, o.detach().numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_finite_differences(causal):
    """Central differences of L = sum(dO * O(Q, K, V)) on a tiny GQA case."""
    Q, K, V, dO = _case(1, 2, 1, 7, 3, seed=11)
    _, _, _, g = _exact_all(Q, K, V, dO, causal)
    h = 1e-6

    def loss(Qx, Kx, Vx):
        O, _ = oracle.attn_fwd(Qx, Kx, Vx, causal, 0.0, EX)
        return float(np.sum(O * dO))

    for name, X, grad in (("Q", Q, g["dQ"]), ("K", K, g["dK"]), ("V", V, g["dV"])):
        fd = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += h
            Xm[idx] -= h
            args_p = {"Q": (Xp, K, V), "K": (Q, Xp, V), "V": (Q, K, Xp)}[name]
            args_m = {"Q": (Xm, K, V), "K": (Q, Xm, V), "V": (Q, K, Xm)}[name]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=name)


@pytest.mark.parametrize("causal", [True, False])
def test_saved_output_shortcut(causal):
    """Exact arithmetic: sum_j P_ij dP_ij equals <dO_i, O_i> (section 01)."""
    Q, K, V, dO = _case(1, 2, 2, 300, 16, seed=5)
    O, LSE = oracle.attn_fwd(Q, K, V, causal, 0.0, EX)
    dm = oracle.attn_delta(Q, K, V, dO, LSE, oracle.DELTA_MATCHED, causal=causal, flags=EX)
    ds = oracle.attn_delta(Q, K, V, dO, LSE, oracle.DELTA_STALE_DO, dO=dO, O=O, causal=causal, flags=EX)
    np.testing.assert_allclose(dm, ds, rtol=1e-11, atol=1e-13)
    # the shortcut computed by hand from O: an independent dot product
    np.testing.assert_allclose(ds, np.sum(dO * O, -1), rtol=1e-14, atol=1e-15)


def test_shift_invariance_and_zero_row_sum():
    """Adding c_i to row i of S leaves P unchanged, shifts LSE by c_i, and sum_j dS_ij = 0."""
    Q, K, V, dO = _case(1, 2, 1, 140, 8, seed=9)
    sigma = 1 / np.sqrt(8)
    c = _rand((1, 2, 140, 1), 17, 3.0)
    Q2 = np.concatenate([Q, c / sigma], -1)           # S'_ij = S_ij + c_i
    K2 = np.concatenate([K, np.ones((1, 1, 140, 1))], -1)
    V2 = np.concatenate([V, np.zeros((1, 1, 140, 1))], -1)
    dO2 = np.concatenate([dO, np.zeros((1, 2, 140, 1))], -1)
    O, LSE, delta, g = _exact_all(Q, K, V, dO, True, sigma=sigma)
    O2, LSE2, delta2, g2 = _exact_all(Q2, K2, V2, dO2, True, sigma=sigma)
    np.testing.assert_allclose(O2[..., :8], O, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(delta2, delta, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(LSE2, LSE + c[..., 0], rtol=1e-12, atol=1e-11)
    for gg in (g, g2):
        rs, ab = gg["diag"][0], gg["diag"][1]
        assert np.all(np.abs(rs) <= 1e-12 * ab + 1e-300)
        assert np.all(np.abs(gg["dS"].sum(-1)) <= 1e-12 * np.abs(gg["dS"]).sum(-1) + 1e-300)
    # the extra column of dQ' is sigma * sum_j dS_ij * 1 = 0
    assert np.all(np.abs(g2["dQ"][..., -1]) <= 1e-12 * np.abs(g2["dQ"]).max())


def _quantised_operands(Q, K, V, dO):
    dec = {}
    for name, x, fmt in (("Q", Q, 0), ("K", K, 0), ("V", V, 0), ("dO", dO, 1)):
        c, s = oracle.quantize(x.astype(np.float32), fmt)
        dec[name] = oracle.dequantize(c, s, fmt)
    return dec


QFLAGS = oracle.QUANT_P_FWD | oracle.QUANT_P_BWD | oracle.QUANT_DS


@pytest.mark.parametrize("causal", [True, False])
def test_matched_zero_row_sum_quantised(causal):
    """Section 03: delta from the backward's own operands gives sum_j dS_ij = 0 (P normalised)."""
    Q, K, V, dO = _case(1, 2, 1, 300, 32, seed=21, qscale=1.5)
    q = _quantised_operands(Q, K, V, dO)
    O, LSE = oracle.attn_fwd(q["Q"], q["K"], q["V"], causal, 0.0, QFLAGS)
    for mode, want_zero in ((oracle.DELTA_MATCHED, True), (oracle.DELTA_STALE_DO, False),
                            (oracle.DELTA_STALE_DOHAT, False)):
        delta = oracle.attn_delta(q["Q"], q["K"], q["V"], q["dO"], LSE, mode, dO=dO, O=O,
                                  causal=causal, flags=QFLAGS)
        g = oracle.attn_bwd(q["Q"], q["K"], q["V"], q["dO"], LSE, delta, causal, 0.0, QFLAGS,
                            want_diag=True)
        rs, ab = np.abs(g["diag"][0]), g["diag"][1]
        if want_zero:
            assert np.all(rs <= 1e-12 * ab)   # rows with a single key have dS = 0 exactly
        else:
            rel = rs[ab > 0] / ab[ab > 0]
            assert np.median(rel) > 1e-4   # the stale corrections leave a visible residual
    # with P held in FP32 and LSE stored in FP32, sum_j P_ij = 1 + eta: the matched
    # delta divides by sum_j P_ij, so the pre-cast row sum is only the FP32
    # rounding of the dS elements themselves (<= 2^-24 per element)
    fl = QFLAGS | oracle.ROUND32
    LSE32 = LSE.astype(np.float32).astype(np.float64)
    delta = oracle.attn_delta(q["Q"], q["K"], q["V"], q["dO"], LSE32, oracle.DELTA_MATCHED, causal=causal, flags=fl)
    g = oracle.attn_bwd(q["Q"], q["K"], q["V"], q["dO"], LSE32, delta, causal, 0.0, fl, want_diag=True)
    assert np.all(np.abs(g["diag"][0]) <= 2.0 ** -23 * g["diag"][1])
    # dividing by sum_j P_ij is what makes this hold: the undivided sum misses by eta * delta
    eta_delta = np.abs(g["diag"][0]).max()
    assert eta_delta <= 1e-6 * np.abs(delta).max()


@pytest.mark.parametrize("quant", ["both", "p_only", "do_only"])
def test_stale_residual_decomposition(quant):
    """eps_i = <dO^_i, (P_i - P^_i) V^> + <dO^_i - dO_i, P^_i V^> (section 01)."""
    Q, K, V, dO = _case(1, 2, 1, 260, 16, seed=31, qscale=1.5)
    q = _quantised_operands(Q, K, V, dO)
    Vh = q["V"]
    dOh = q["dO"] if quant in ("both", "do_only") else dO
    fwd_flags = oracle.QUANT_P_FWD if quant in ("both", "p_only") else EX
    O, LSE, Pf = oracle.attn_fwd(q["Q"], q["K"], Vh, True, 0.0, fwd_flags, want_pfwd=True)
    np.testing.assert_allclose(O, Pf @ np.repeat(Vh, 2, 1), rtol=1e-12, atol=1e-14)  # O = P^fwd V^
    d_dm = oracle.attn_delta(q["Q"], q["K"], Vh, dOh, LSE, oracle.DELTA_MATCHED, flags=EX)
    d_st = oracle.attn_delta(q["Q"], q["K"], Vh, dOh, LSE, oracle.DELTA_STALE_DO, dO=dO, O=O, flags=EX)
    d_sh = oracle.attn_delta(q["Q"], q["K"], Vh, dOh, LSE, oracle.DELTA_STALE_DOHAT, O=O, flags=EX)
    g = oracle.attn_bwd(q["Q"], q["K"], Vh, dOh, LSE, d_dm, True, 0.0, EX, want_tiles=True)
    P = g["Phat"]                                     # backward P, unquantised here
    Vr = np.repeat(Vh, 2, 1)
    term1 = np.einsum("bhik,bhik->bhi", dOh, (P - Pf) @ Vr)
    term2 = np.einsum("bhik,bhik->bhi", dOh - dO, Pf @ Vr)
    eps = d_dm - d_st
    scale = np.abs(eps).max()
    np.testing.assert_allclose(eps, term1 + term2, rtol=0, atol=1e-10 * scale)
    if quant == "p_only":
        assert np.abs(term2).max() == 0.0
    if quant == "do_only":
        assert np.abs(term1).max() <= 1e-12 * scale
    # matching dO only (delta = <dO^, O>) leaves exactly the probability term
    np.testing.assert_allclose(d_dm - d_sh, term1, rtol=0, atol=1e-10 * scale)
    assert np.abs(eps).max() > 0


def test_stale_gradient_is_centered_plus_eps_p():
    """Section 02: dS_stale = dS_centered + eps_i * P_ij, elementwise, before the cast."""
    Q, K, V, dO = _case(1, 2, 1, 200, 16, seed=41)
    q = _quantised_operands(Q, K, V, dO)
    O, LSE = oracle.attn_fwd(q["Q"], q["K"], q["V"], True, 0.0, oracle.QUANT_P_FWD)
    d_c = oracle.attn_delta(q["Q"], q["K"], q["V"], q["dO"], LSE, oracle.DELTA_MATCHED, flags=EX)
    d_s = oracle.attn_delta(q["Q"], q["K"], q["V"], q["dO"], LSE, oracle.DELTA_STALE_DO, dO=dO, O=O, flags=EX)
    gc = oracle.attn_bwd(q["Q"], q["K"], q["V"], q["dO"], LSE, d_c, True, 0.0, EX, want_tiles=True)
    gs = oracle.attn_bwd(q["Q"], q["K"], q["V"], q["dO"], LSE, d_s, True, 0.0, EX, want_tiles=True)
    eps = (d_c - d_s)[..., None]
    diff = gs["dS"] - gc["dS"]
    np.testing.assert_allclose(diff, eps * gc["Phat"], rtol=0, atol=1e-12 * np.abs(gc["dS"]).max())
    # the sign argument: rows with eps < 0 get a negative row sum pushed onto their largest P
    assert np.all(np.sign(diff.sum(-1)[np.abs(eps[..., 0]) > 1e-9]) ==
                  np.sign(eps[..., 0][np.abs(eps[..., 0]) > 1e-9]))


def test_gqa_is_sum_over_query_heads():
    Q, K, V, dO = _case(1, 4, 2, 150, 16, seed=51)
    q = _quantised_operands(Q, K, V, dO)
    res = oracle.pipeline(Q.astype(np.float32), K.astype(np.float32), V.astype(np.float32),
                          dO.astype(np.float32))
    # MHA with each kv head repeated for its query heads, run head by head
    Kr, Vr = np.repeat(q["K"], 2, 1), np.repeat(q["V"], 2, 1)
    O, LSE = oracle.attn_fwd(q["Q"], Kr, Vr, True, 0.0, oracle.GPU_CONTRACT)
    LSE32 = LSE.astype(np.float32).astype(np.float64)
    delta = oracle.attn_delta(q["Q"], Kr, Vr, q["dO"], LSE32, flags=oracle.GPU_CONTRACT)
    g = oracle.attn_bwd(q["Q"], Kr, Vr, q["dO"], LSE32, delta, True, 0.0, oracle.GPU_CONTRACT)
    np.testing.assert_array_equal(res["dQ"], g["dQ"])
    for key in ("dK", "dV"):
        want = g[key].reshape(1, 2, 2, 150, 16).sum(2)
        np.testing.assert_allclose(res[key], want, rtol=0, atol=1e-13 * np.abs(want).max())


def test_one_pass_forward_single_tile_vs_torch_cast():
    """One key tile: P~ = exp(S - rowmax), tile amax 1, codes = enc(fl32(P~ * 448))."""
    Q, K, V, _ = _case(1, 1, 1, 100, 16, seed=61, qscale=2.0)
    O, LSE = oracle.attn_fwd(Q, K, V, True, 0.0, oracle.QUANT_P_FWD | oracle.ROUND32)
    S = (Q[0, 0] @ K[0, 0].T) / 4.0
    S[np.triu_indices(100, 1)] = -np.inf
    m = S.max(-1, keepdims=True)
    pt = np.exp(S - m).astype(np.float32)
    codes = torch.from_numpy(pt * np.float32(448.0)).to(torch.float8_e4m3fn)
    sP = np.float64(np.float32(1.0) / np.float32(448.0))
    ph = codes.to(torch.float64).numpy() * sP
    l = pt.astype(np.float64).sum(-1, keepdims=True)
    np.testing.assert_allclose(O[0, 0], (ph @ V[0, 0]) / l, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(LSE[0, 0], m[:, 0] + np.log(l[:, 0]), rtol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_one_pass_forward_properties(causal):
    """Multi-tile one-pass forward: O = Pfwd V, rows of Pfwd sum to 1 within FP8 error,
    O within FP8 error of exact attention even when the running max rises in late tiles."""
    Q, K, V, _ = _case(1, 2, 1, 400, 16, seed=71)
    K[0, 0, 300:] *= 3.0        # later key tiles hold larger scores: the running max must be rescaled
    O, LSE, Pf = oracle.attn_fwd(Q, K, V, causal, 0.0, oracle.GPU_CONTRACT, want_pfwd=True)
    Oe, LSEe = oracle.attn_fwd(Q, K, V, causal, 0.0, EX)
    np.testing.assert_allclose(O, Pf @ np.repeat(V, 2, 1), rtol=1e-12, atol=1e-13)
    assert np.abs(Pf.sum(-1) - 1).max() < 0.04
    np.testing.assert_allclose(LSE, LSEe, rtol=0, atol=1e-5)   # l uses the unquantised P~
    rel = np.linalg.norm(O - Oe) / np.linalg.norm(Oe)
    assert 1e-4 < rel < 0.05
    if causal:
        assert np.all(Pf[..., np.triu_indices(400, 1)[0], np.triu_indices(400, 1)[1]] == 0)


def test_tile_selection_matches_full_run():
    Q, K, V, dO = _case(2, 4, 2, 300, 16, seed=81)
    full = oracle.pipeline(Q, K, V, dO, want_diag=True)
    part = oracle.pipeline(Q, K, V, dO, q_tiles=[0, 2], kv_tiles=[1, 2], groups=[(1, 0), (0, 1)], want_diag=True)
    for b, g in ((1, 0), (0, 1)):
        hs = slice(2 * g, 2 * g + 2)
        for t in (0, 2):
            rs = slice(128 * t, 128 * t + 128)
            for key in ("O", "LSE", "delta", "dQ"):
                np.testing.assert_array_equal(part[key][b, hs, rs], full[key][b, hs, rs])
            np.testing.assert_array_equal(part["diag"][:, b, hs, rs], full["diag"][:, b, hs, rs])
        for t in (1, 2):
            rs = slice(128 * t, 128 * t + 128)
            np.testing.assert_array_equal(part["dK"][b, g, rs], full["dK"][b, g, rs])
            np.testing.assert_array_equal(part["dV"][b, g, rs], full["dV"][b, g, rs])
