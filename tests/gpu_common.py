"""Shared helpers for the GPU parity tests: run the CUDA path and the oracle
on the same seeded inputs and compare."""
from __future__ import annotations

import numpy as np
import torch

import fp8_attention_gb300 as dm
import oracle

TOL = 2e-3          # relative Frobenius error bound for O, LSE, delta, dQ, dK, dV
ROWSUM_TOL = 1e-4   # matched-delta rows: |sum_j dS_ij| <= 1e-4 * sum_j |dS_ij| (before the E5M2 cast)

DEV = torch.device("cuda:0")


def rel_err(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / den) if den > 0 else float(np.linalg.norm(got))


def gpu_pipeline(q, k, v, do, causal=True, mode=dm.DM_DELTA_MATCHED, o_dtype=torch.float32, sigma=0.0,
                 diag=False, delta_in_bwd=False):
    """Quantise, forward, delta and backward on the GPU; returns torch tensors on the GPU."""
    B, Hq, N, d = q.shape
    p = dm.AttnParams(B, Hq, k.shape[1], N, d, causal=causal, softmax_scale=sigma, d_v=v.shape[-1])
    res = {"p": p}
    qh = dm.dm_quantize(q.to(DEV), dm.DM_E4M3)
    kh = dm.dm_quantize(k.to(DEV), dm.DM_E4M3)
    vh = dm.dm_quantize(v.to(DEV), dm.DM_E4M3)
    doh = dm.dm_quantize(do.to(DEV), dm.DM_E5M2)
    do_dev = do.to(DEV)
    O, lse = dm.dm_attn_fwd(p, qh, kh, vh, o_dtype=o_dtype)
    if delta_in_bwd:
        delta = None
    else:
        delta = dm.dm_attn_delta(p, mode, qh, kh, vh, doh, lse, dO=do_dev, O=O)
    g = dm.dm_attn_bwd(p, mode, qh, kh, vh, doh, lse, delta, dO=do_dev, O=O, diag=diag)
    st = dm.dm_get_status()
    assert st == 0, dm.dm_status_string(st)
    res.update(g)
    res.update(O=O, LSE=lse, delta=delta, q=qh, k=kh, v=vh, do=doh)
    return res


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def oracle_pipeline(q, k, v, do, causal=True, mode=oracle.DELTA_MATCHED, o_bf16=False, sigma=0.0, **kw):
    return oracle.pipeline(np32(q), np32(k), np32(v), np32(do), causal=causal, sigma=sigma, mode=mode,
                           o_bf16=o_bf16, **kw)
