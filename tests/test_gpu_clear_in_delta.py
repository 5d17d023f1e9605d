"""The one-call backward starts its outputs at zero without a fill launch.

dm_attn_bwd with delta NULL and the matched mode computes delta itself, and
that kernel also clears dQ, dK, dV and the diagnostics rows, which the
backward then adds into (bulk reduce-adds, atomics).  Here every output
holds NaN before the call.  The results must match the oracle within the
usual 2e-3, and the two-call path (dm_attn_delta, then dm_attn_bwd with that
delta, whose outputs a fill launch clears) up to the order of the fp32
reduce-adds.  The shapes cover a GQA group (only its first query head's
CTAs clear dK and dV), a ragged last tile, no mask, d = 64, 128, 256 and
heads with a narrower value dimension (dV rows d_v wide).
"""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
from fp8_attention_gb300.inputs import custom, make_inputs
from gpu_common import DEV, TOL, np32, oracle_pipeline, rel_err

pytestmark = pytest.mark.gpu

DIAG = ("rowsum_pre", "abssum_pre", "rowsum_post", "abssum_post")


@pytest.mark.parametrize("shape,causal", [
    ((1, 4, 2, 384, 128, 128), True),
    ((2, 4, 1, 300, 64, 64), False),
    ((1, 2, 2, 260, 256, 256), True),
    ((1, 2, 2, 200, 192, 128), True),
])
def test_outputs_cleared_by_the_delta_pass(shape, causal):
    B, Hq, Hkv, N, d, dv = shape
    w = custom(B, Hq, Hkv, N, d, causal=causal, seed=N + d, dv=dv)
    q, k, v, do = make_inputs(w)
    p = dm.AttnParams(B, Hq, Hkv, N, d, causal=causal, d_v=dv)
    qh = dm.dm_quantize(q.to(DEV), dm.DM_E4M3)
    kh = dm.dm_quantize(k.to(DEV), dm.DM_E4M3)
    vh = dm.dm_quantize(v.to(DEV), dm.DM_E4M3)
    doh = dm.dm_quantize(do.to(DEV), dm.DM_E5M2)
    O, lse = dm.dm_attn_fwd(p, qh, kh, vh)
    nan = lambda *sh: torch.full(sh, float("nan"), dtype=torch.float32, device=DEV)
    diag = {n: nan(B, Hq, N) for n in DIAG}
    one = dm.dm_attn_bwd(p, dm.DM_DELTA_MATCHED, qh, kh, vh, doh, lse, None, dQ=nan(B, Hq, N, d),
                         dK=nan(B, Hkv, N, d), dV=nan(B, Hkv, N, dv), diag=diag)
    delta = dm.dm_attn_delta(p, dm.DM_DELTA_MATCHED, qh, kh, vh, doh, lse)
    two = dm.dm_attn_bwd(p, dm.DM_DELTA_MATCHED, qh, kh, vh, doh, lse, delta, diag=True)
    assert dm.dm_get_status() == dm.DM_OK
    for key in ("dQ", "dK", "dV") + DIAG:
        got, want = np32(one[key]), np32(two[key])
        assert np.isfinite(got).all(), key
        if key.startswith("rowsum"):  # near-cancelling sums: bound by the absolute sums
            scale = np.abs(np32(two["abssum" + key[6:]])).max()
            assert np.abs(got - want).max() <= 1e-5 * scale, key
        else:
            err = rel_err(got, want)
            assert err <= 1e-5, (key, err)
    r = oracle_pipeline(q, k, v, do, causal=causal)
    for key in ("dQ", "dK", "dV"):
        err = rel_err(np32(one[key]), r[key])
        assert err <= TOL, (key, err)


def test_one_call_backward_on_a_side_stream():
    """The one-call backward on a stream other than the current one, with the
    workspace allocated by the binding: the same gradients as on the current
    stream, also when the current stream allocates and writes right after."""
    B, Hq, Hkv, N, d = 1, 4, 2, 384, 128
    w = custom(B, Hq, Hkv, N, d, causal=True, seed=71)
    q, k, v, do = make_inputs(w)
    p = dm.AttnParams(B, Hq, Hkv, N, d, causal=True)
    qh = dm.dm_quantize(q.to(DEV), dm.DM_E4M3)
    kh = dm.dm_quantize(k.to(DEV), dm.DM_E4M3)
    vh = dm.dm_quantize(v.to(DEV), dm.DM_E4M3)
    doh = dm.dm_quantize(do.to(DEV), dm.DM_E5M2)
    _, lse = dm.dm_attn_fwd(p, qh, kh, vh)
    ref = dm.dm_attn_bwd(p, dm.DM_DELTA_MATCHED, qh, kh, vh, doh, lse, None)
    torch.cuda.synchronize()
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream())
    got = dm.dm_attn_bwd(p, dm.DM_DELTA_MATCHED, qh, kh, vh, doh, lse, None, stream=side)
    junk = torch.full((dm.dm_attn_bwd_workspace_size(p) // 4,), float("nan"), device=DEV)  # may not take its place
    torch.cuda.synchronize()
    assert dm.dm_get_status() == dm.DM_OK
    for key in ("dQ", "dK", "dV"):
        assert rel_err(np32(got[key]), np32(ref[key])) <= 1e-5, key
    del junk
