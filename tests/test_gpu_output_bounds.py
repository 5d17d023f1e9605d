"""Every output stays inside its tensor.

O is written by TMA tile stores of whole 128-row boxes, dQ, dK and dV by bulk
reduce-adds of 128-row boxes, and the one-call backward's delta kernel clears
the gradients row by row; on a ragged last query or key tile the boxes reach
past row N, where the tensor maps must clip them.  Each output here is the
front of a larger buffer whose tail holds a sentinel, on shapes whose last
tile is ragged (and heads with a narrower value dimension, whose rows are
d_v wide); the tail must be untouched and the results finite.
"""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
from fp8_attention_gb300.inputs import custom, make_inputs
from gpu_common import DEV

pytestmark = pytest.mark.gpu

SENTINEL = 12345.0
PAD = 4096


def _padded(shape, dtype=torch.float32):
    n = int(np.prod(shape))
    buf = torch.full((n + PAD,), SENTINEL, dtype=dtype, device=DEV)
    return buf, buf[:n].view(shape)


def _tail_intact(buf, n):
    return bool(torch.all(buf[n:] == SENTINEL))


@pytest.mark.parametrize("shape", [(1, 4, 2, 300, 128, 128), (2, 2, 1, 200, 64, 64), (1, 2, 2, 260, 192, 128),
                                   (1, 2, 1, 130, 256, 256)])
@pytest.mark.parametrize("o_dtype", [torch.float32, torch.bfloat16])
def test_outputs_stay_inside_their_tensors(shape, o_dtype):
    B, Hq, Hkv, N, d, dv = shape
    w = custom(B, Hq, Hkv, N, d, causal=True, seed=N + d + dv, dv=dv)
    q, k, v, do = make_inputs(w)
    p = dm.AttnParams(B, Hq, Hkv, N, d, causal=True, d_v=dv)
    qh = dm.dm_quantize(q.to(DEV), dm.DM_E4M3)
    kh = dm.dm_quantize(k.to(DEV), dm.DM_E4M3)
    vh = dm.dm_quantize(v.to(DEV), dm.DM_E4M3)
    doh = dm.dm_quantize(do.to(DEV), dm.DM_E5M2)
    obuf, O = _padded((B, Hq, N, dv), o_dtype)
    _, lse = dm.dm_attn_fwd(p, qh, kh, vh, O=O)
    torch.cuda.synchronize()
    assert _tail_intact(obuf, O.numel()), "O written past its tensor"
    assert bool(torch.isfinite(O.float()).all())
    for delta_in_bwd in (False, True):
        delta = None if delta_in_bwd else dm.dm_attn_delta(p, dm.DM_DELTA_MATCHED, qh, kh, vh, doh, lse)
        bufs = {"dQ": _padded((B, Hq, N, d)), "dK": _padded((B, Hkv, N, d)), "dV": _padded((B, Hkv, N, dv))}
        g = dm.dm_attn_bwd(p, dm.DM_DELTA_MATCHED, qh, kh, vh, doh, lse, delta,
                           **{name: t for name, (_, t) in bufs.items()})
        torch.cuda.synchronize()
        assert dm.dm_get_status() == dm.DM_OK
        for name, (buf, t) in bufs.items():
            assert _tail_intact(buf, t.numel()), f"{name} written past its tensor (delta in backward: {delta_in_bwd})"
            assert bool(torch.isfinite(g[name]).all()), name
