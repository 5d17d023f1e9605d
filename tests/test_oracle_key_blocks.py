"""Pins for the oracle's key-block (context-parallel) functions.

The project page ("Delta-Matching for reliable FP8 attention training",
section 06) extends the context from 8K to 64K tokens, where attention is
split over the sequence; it does not say how.  The reading taken here: the keys
are split into blocks, every block's attention is computed for every query row
(O_r, LSE_r), the blocks are merged by the log-sum-exp rule, the matched delta
adds the blocks' partial sums sum_j P dP^ and sum_j P before its one division
(section 03's delta over all keys), and the backward runs per block with the
merged LSE and delta, its dQ summed over blocks.

Pins, each against something other than the oracle's own formula:
* a key range against torch's scaled-dot-product attention with the block's
  mask (a library routine), causal and not, rows seeing no key excluded;
* the merge against torch.logsumexp and a weighted sum written out;
* the whole split pipeline in exact arithmetic against torch autograd of
  plain attention (a library), for two and three blocks;
* the quantised one-pass forward over a key range against the unsplit
  quantised forward on the block's keys alone (non-causal: the same problem);
* the blocks' partial delta sums and dQ adding up to the unsplit values.
"""
import numpy as np
import pytest
import torch

import oracle

EX = oracle.EXACT


def _case(B=1, Hq=2, Hkv=1, N=300, d=16, seed=0, dv=None):
    rng = np.random.default_rng(seed)
    dv = d if dv is None else dv
    return (rng.standard_normal((B, Hq, N, d)), rng.standard_normal((B, Hkv, N, d)),
            rng.standard_normal((B, Hkv, N, dv)), rng.standard_normal((B, Hq, N, dv)))


def _torch_block(Q, K, V, causal, kb, ke):
    """Attention over keys [kb, ke) by torch SDPA with an explicit boolean mask."""
    G = Q.shape[1] // K.shape[1]
    N = Q.shape[2]
    q = torch.tensor(Q)
    k = torch.tensor(K).repeat_interleave(G, 1)
    v = torch.tensor(V).repeat_interleave(G, 1)
    j = torch.arange(N)
    allowed = ((j >= kb) & (j < ke))[None, :].expand(N, N).clone()
    if causal:
        allowed &= j[None, :] <= j[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed)
    s = (q @ k.transpose(-1, -2)) / np.sqrt(Q.shape[-1])
    lse = torch.logsumexp(s.masked_fill(~allowed, float("-inf")), -1)
    return o.numpy(), lse.numpy(), allowed.any(-1).numpy()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("kb,ke", [(0, 128), (128, 300), (128, 256), (256, 300)])
def test_key_range_forward_matches_masked_sdpa(causal, kb, ke):
    Q, K, V, _ = _case(1, 4, 2, 300, 16, seed=kb + ke)
    O, LSE = oracle.attn_fwd(Q, K, V, causal, 0.0, EX, kv_range=(kb, ke))
    Ot, Lt, seen = _torch_block(Q, K, V, causal, kb, ke)
    np.testing.assert_allclose(O[..., seen, :], Ot[..., seen, :], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(LSE[..., seen], Lt[..., seen], rtol=1e-12, atol=1e-12)
    assert np.all(O[..., ~seen, :] == 0) and np.all(LSE[..., ~seen] == -np.inf)
    if causal and kb > 0:
        assert (~seen).any()


def test_merge_matches_logsumexp():
    rng = np.random.default_rng(3)
    S, rows, dv = 3, 50, 8
    Op = rng.standard_normal((S, 1, 1, rows, dv))
    Lp = rng.standard_normal((S, 1, 1, rows)) * 5
    Lp[0, 0, 0, :10] = -np.inf            # block 0 sees nothing in these rows
    Lp[:, 0, 0, 10:12] = -np.inf          # no block sees anything
    O, LSE = oracle.attn_merge(Op, Lp)
    lt = torch.logsumexp(torch.tensor(Lp), 0).numpy()
    np.testing.assert_allclose(LSE[..., 12:], lt[..., 12:], rtol=1e-14, atol=1e-14)
    with np.errstate(invalid="ignore"):
        w = np.exp(Lp - lt[None])
    want = (w[..., None] * Op).sum(0)
    np.testing.assert_allclose(O[..., 12:, :], want[..., 12:, :], rtol=1e-13, atol=1e-14)
    assert np.all(O[..., 10:12, :] == 0) and np.all(LSE[..., 10:12] == -np.inf)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("bounds", [(0, 128, 300), (0, 128, 256, 300)])
def test_split_pipeline_exact_matches_torch_autograd(causal, bounds):
    """Exact arithmetic: merged forward, summed delta parts and summed dQ equal
    plain attention and its autograd gradients."""
    Q, K, V, dO = _case(1, 4, 2, 300, 16, seed=len(bounds))
    res = oracle.pipeline_key_blocks(Q, K, V, dO, list(bounds), causal=causal, flags=EX)
    G = 2
    # exact mode still quantises the inputs to FP8 first (as the GPU does): use the decoded operands
    dq = oracle.dequantize(res["q_codes"], res["q_scales"], oracle.E4M3)
    dk = oracle.dequantize(res["k_codes"], res["k_scales"], oracle.E4M3)
    dvv = oracle.dequantize(res["v_codes"], res["v_scales"], oracle.E4M3)
    ddo = oracle.dequantize(res["do_codes"], res["do_scales"], oracle.E5M2)
    q = torch.tensor(dq, requires_grad=True)
    k = torch.tensor(dk, requires_grad=True)
    v = torch.tensor(dvv, requires_grad=True)
    o = torch.nn.functional.scaled_dot_product_attention(q, k.repeat_interleave(G, 1), v.repeat_interleave(G, 1),
                                                         is_causal=causal)
    o.backward(torch.tensor(ddo))
    # O and LSE as stored (fp32): compare within fp32 rounding
    np.testing.assert_allclose(res["O"], o.detach().numpy(), rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(res["delta"], np.sum(ddo * o.detach().numpy(), -1), rtol=1e-5, atol=1e-7)
    for key, t in (("dQ", q), ("dK", k), ("dV", v)):
        np.testing.assert_allclose(res[key], t.grad.numpy(), rtol=1e-4, atol=1e-5 * np.abs(t.grad.numpy()).max(),
                                   err_msg=key)


def test_quantised_key_range_is_the_forward_on_the_block():
    """Non-causal: the quantised one-pass forward over keys [128, 384) is the
    unsplit quantised forward on K, V cut to those keys (its running maximum
    starts at the block's first tile)."""
    Q, K, V, _ = _case(1, 2, 1, 400, 16, seed=9)
    O, LSE = oracle.attn_fwd(Q, K, V, False, 0.0, oracle.GPU_CONTRACT, kv_range=(128, 384))
    # the same query rows against the cut keys: one problem of 256 rows whose
    # query tiles are the original tiles 1 and 2 (a non-causal row sees only keys)
    cut = lambda x: np.ascontiguousarray(x[:, :, 128:384])
    Oc, LSEc = oracle.attn_fwd(cut(Q), cut(K), cut(V), False, 0.0, oracle.GPU_CONTRACT)
    np.testing.assert_array_equal(O[:, :, 128:384], Oc)
    np.testing.assert_array_equal(LSE[:, :, 128:384], LSEc)


@pytest.mark.parametrize("causal", [True, False])
def test_partial_delta_and_dq_add_up(causal):
    """With one LSE, the blocks' partial sums give the unsplit matched delta and
    the blocks' dQ add up to the unsplit dQ; dK, dV of a block are the unsplit
    rows (the per-tile work is the same)."""
    Q, K, V, dO = _case(2, 4, 2, 300, 16, seed=21)
    flags = oracle.GPU_CONTRACT
    _, LSE = oracle.attn_fwd(Q, K, V, causal, 0.0, EX)
    LSE = LSE.astype(np.float32).astype(np.float64)
    full = oracle.attn_delta(Q, K, V, dO, LSE, causal=causal, flags=flags)
    num = np.zeros_like(full)
    den = np.zeros_like(full)
    blocks = [(0, 128), (128, 256), (256, 300)]
    for b in blocks:
        n_r, d_r = oracle.attn_delta(Q, K, V, dO, LSE, causal=causal, flags=flags, kv_range=b, partial=True)
        num += n_r
        den += d_r
    np.testing.assert_allclose(num / den, full, rtol=1e-12, atol=1e-15)
    # sum_j P_ij over all keys from torch, against the summed denominators
    s = torch.tensor(Q) @ torch.tensor(K).repeat_interleave(2, 1).transpose(-1, -2) / 4.0
    if causal:
        s = s.masked_fill(torch.ones(300, 300, dtype=torch.bool).triu(1), float("-inf"))
    psum = torch.exp(s - torch.tensor(LSE)[..., None]).sum(-1).numpy()
    np.testing.assert_allclose(den, psum, rtol=1e-6)      # P rounded to FP32 in the contract
    g = oracle.attn_bwd(Q, K, V, dO, LSE, full, causal, 0.0, flags)
    dq = np.zeros_like(g["dQ"])
    for b in blocks:
        gb = oracle.attn_bwd(Q, K, V, dO, LSE, full, causal, 0.0, flags, kv_range=b)
        dq += gb["dQ"]
        np.testing.assert_array_equal(gb["dK"][:, :, b[0]:b[1]], g["dK"][:, :, b[0]:b[1]])
        np.testing.assert_array_equal(gb["dV"][:, :, b[0]:b[1]], g["dV"][:, :, b[0]:b[1]])
        outside = np.ones(300, bool)
        outside[b[0]:b[1]] = False
        assert np.all(gb["dK"][:, :, outside] == 0) and np.all(gb["dV"][:, :, outside] == 0)
    np.testing.assert_allclose(dq, g["dQ"], rtol=0, atol=1e-13 * np.abs(g["dQ"]).max())
