"""Context-parallel attention with the Delta-Matching correction over a process group.

The project page ("Delta-Matching for reliable FP8 attention training",
section 06) extends the context from 8K to 64K tokens.  Here the sequence's
keys are split over the ranks of a torch.distributed group: rank r holds every
query row (Q, dO) and one 128-aligned key block (K, V rows [kv_offset,
kv_offset + kv_len), given by its AttnParams).  Per step:

* forward: each rank's block attention (O_r, LSE_r), an all-gather of both and
  the log-sum-exp merge (dm_attn_merge) into the whole sequence's O and LSE;
* matched delta: each rank's sums over its keys of P dP^ and of P
  (dm_attn_delta_partial, P from the merged LSE), one sum all-reduce of the
  pair, then the one division (dm_attn_delta_combine);
* backward: each rank's block backward with the merged LSE and delta gives
  dK, dV of its keys (complete: all query rows are local) and its share of
  dQ, which one sum all-reduce completes.

The collectives are the only exchange; every arithmetic step is one of the
library's kernels (``ops``).  The per-rank steps are injectable so that the
exchange logic can be exercised with any implementation of them.
"""
from __future__ import annotations

from dataclasses import replace
from typing import Optional

import torch
import torch.distributed as dist

from . import (DM_DELTA_MATCHED, AttnParams, Fp8, dm_attn_bwd, dm_attn_delta_combine, dm_attn_delta_partial,
               dm_attn_fwd, dm_attn_merge)


class LibraryOps:
    """The per-rank steps as the library's calls (the GPU path)."""

    @staticmethod
    def fwd(p: AttnParams, q: Fp8, k: Fp8, v: Fp8):
        return dm_attn_fwd(p, q, k, v)

    @staticmethod
    def merge(p: AttnParams, O_parts, lse_parts):
        return dm_attn_merge(p, O_parts, lse_parts)

    @staticmethod
    def delta_partial(p: AttnParams, q: Fp8, k: Fp8, v: Fp8, do_hat: Fp8, lse, nd):
        dm_attn_delta_partial(p, q, k, v, do_hat, lse, num=nd[0], den=nd[1])

    @staticmethod
    def delta_combine(p: AttnParams, nd):
        return dm_attn_delta_combine(p, nd[0:1], nd[1:2])

    @staticmethod
    def bwd(p: AttnParams, q: Fp8, k: Fp8, v: Fp8, do_hat: Fp8, lse, delta):
        return dm_attn_bwd(p, DM_DELTA_MATCHED, q, k, v, do_hat, lse, delta)


def whole(p: AttnParams) -> AttnParams:
    """The same problem without a key block (the whole sequence's shapes)."""
    return replace(p, kv_offset=0, kv_len=0)


def forward(p: AttnParams, q: Fp8, k: Fp8, v: Fp8, group: Optional[dist.ProcessGroup] = None, ops=LibraryOps):
    """O [B][Hq][N][d_v] and LSE [B][Hq][N] of the whole sequence from this rank's key block."""
    S = dist.get_world_size(group)
    O_r, lse_r = ops.fwd(p, q, k, v)
    O_all = torch.empty((S,) + tuple(O_r.shape), dtype=O_r.dtype, device=O_r.device)
    lse_all = torch.empty((S,) + tuple(lse_r.shape), dtype=lse_r.dtype, device=lse_r.device)
    dist.all_gather_into_tensor(O_all.view(-1), O_r.reshape(-1), group=group)
    dist.all_gather_into_tensor(lse_all.view(-1), lse_r.reshape(-1), group=group)
    return ops.merge(whole(p), O_all, lse_all)


def delta(p: AttnParams, q: Fp8, k: Fp8, v: Fp8, do_hat: Fp8, lse, group: Optional[dist.ProcessGroup] = None,
          ops=LibraryOps):
    """The matched delta [B][Hq][N] of the whole sequence (lse: the merged one)."""
    nd = torch.empty((2, p.B, p.Hq, p.N), dtype=lse.dtype, device=lse.device)
    ops.delta_partial(p, q, k, v, do_hat, lse, nd)
    dist.all_reduce(nd, op=dist.ReduceOp.SUM, group=group)
    return ops.delta_combine(whole(p), nd)


def backward(p: AttnParams, q: Fp8, k: Fp8, v: Fp8, do_hat: Fp8, lse, delta_, group: Optional[dist.ProcessGroup] = None,
             ops=LibraryOps):
    """dQ of the whole sequence (summed over the ranks) and dK, dV of this rank's keys."""
    g = ops.bwd(p, q, k, v, do_hat, lse, delta_)
    dist.all_reduce(g["dQ"], op=dist.ReduceOp.SUM, group=group)
    return g


def step(p: AttnParams, q: Fp8, k: Fp8, v: Fp8, do_hat: Fp8, group: Optional[dist.ProcessGroup] = None,
         ops=LibraryOps):
    """Forward, matched delta and backward of one training step; returns a dict
    with O, LSE, delta, dQ (whole sequence) and dK, dV (this rank's keys)."""
    O, lse = forward(p, q, k, v, group, ops)
    d = delta(p, q, k, v, do_hat, lse, group, ops)
    g = backward(p, q, k, v, do_hat, lse, d, group, ops)
    return {"O": O, "LSE": lse, "delta": d, **g}
