"""The no-allocation backward entry point, for callers that cannot allocate
device memory (a runtime that plans every device byte ahead of the training
step, or a host program that only reaches this library through its C ABI and
has no device allocator): it must give the same gradients as dm_attn_bwd with
a caller-provided workspace, on two calls in a row sharing its fixed array,
and must reject problems larger than that array before launching anything.

Kept in a file of its own that pytest collects last."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
from fp8_attention_gb300.inputs import custom, make_inputs
from gpu_common import DEV, TOL, rel_err

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, N, d, seed):
    q, k, v, do = make_inputs(custom(B, Hq, Hkv, N, d, seed=seed))
    p = dm.AttnParams(B, Hq, Hkv, N, d)
    qh = dm.dm_quantize(q.to(DEV), dm.DM_E4M3)
    kh = dm.dm_quantize(k.to(DEV), dm.DM_E4M3)
    vh = dm.dm_quantize(v.to(DEV), dm.DM_E4M3)
    doh = dm.dm_quantize(do.to(DEV), dm.DM_E5M2)
    O, lse = dm.dm_attn_fwd(p, qh, kh, vh)
    return p, qh, kh, vh, doh, lse, do.to(DEV), O


@pytest.mark.parametrize("mode", [dm.DM_DELTA_MATCHED, dm.DM_DELTA_STALE_DO])
def test_noalloc_matches_workspace_backward_twice(mode):
    cases = [(1, 4, 2, 384, 128, 11), (2, 2, 1, 200, 64, 12)]   # second call: a different, ragged problem
    for B, Hq, Hkv, N, d, seed in cases:
        p, qh, kh, vh, doh, lse, do, O = _inputs(B, Hq, Hkv, N, d, seed)
        ref = dm.dm_attn_bwd(p, mode, qh, kh, vh, doh, lse, None, dO=do, O=O, diag=True)   # workspace path
        got = dm.dm_attn_bwd_noalloc(p, mode, qh, kh, vh, doh, lse, dO=do, O=O, diag=True)
        assert dm.dm_get_status() == dm.DM_OK
        for key in ("dQ", "dK", "dV", "abssum_pre", "abssum_post"):
            err = rel_err(got[key].double().cpu().numpy(), ref[key].double().cpu().numpy())
            assert err <= TOL, (key, err)


def test_noalloc_rejects_oversize_before_launch():
    L = dm.lib()
    rows = dm.DM_NOALLOC_MAX_DELTA_ROWS
    p = dm.AttnParams(1, 16, 4, rows // 16 + 128, 128).c()
    A = 0x10000
    f = dm._Fp8(A, A)
    rc = L.dm_attn_bwd_noalloc(ctypes.byref(p), 0, f, f, f, f, A, None, 0, None, 0, A, A, A, None, None)
    assert rc == dm.DM_ERR_SHAPE
    ok = dm.AttnParams(1, 16, 4, rows // 16, 128).c()   # at the limit: accepted by the size check
    rc = L.dm_attn_bwd_noalloc(ctypes.byref(ok), 0, f, f, f, dm._Fp8(None, None), A, None, 0, None, 0, A, A, A,
                               None, None)
    assert rc == dm.DM_ERR_INVALID_ARG  # rejected later, on the missing dO^ pointer, still before any launch
    assert dm.dm_get_status() == dm.DM_OK
