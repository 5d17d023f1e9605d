"""Key blocks (context parallelism over the sequence) on one GPU, against the oracle.

The project page ("Delta-Matching for reliable FP8 attention training",
section 06) extends the context from 8K to 64K tokens; splitting the sequence
over devices needs each device's share of attention to merge exactly.  Here
the keys are split into 128-aligned blocks, each block runs as its own calls
one after the other on one GPU (as one rank of a context-parallel group would):
K and V of the block quantised on their own, dm_attn_fwd over the block,
dm_attn_merge of the stacked O/LSE, dm_attn_delta_partial per block and
dm_attn_delta_combine, dm_attn_bwd per block with the merged LSE and delta,
dQ summed over the blocks.

Bars: K/V codes and scales of each block bit-exact with the whole tensor's;
every result (the blocks' own O and LSE too) within 2e-3 of the oracle's split
pipeline; LSE, delta, dQ, dK and dV also within 2e-3 of the unsplit oracle
(the merged O differs from a single pass by the FP8 rounding of P~ against
each block's own running maximum, a few 1e-3 relative).
"""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
import oracle
from fp8_attention_gb300.inputs import WORKLOADS, custom, make_inputs
from gpu_common import DEV, TOL, np32, rel_err

pytestmark = pytest.mark.gpu


def gpu_key_blocks(q, k, v, do, bounds, causal=True, d_v=0):
    """The whole split pipeline on the GPU; returns a dict of GPU tensors."""
    B, Hq, N, d = q.shape
    Hkv, dv = k.shape[1], v.shape[-1]
    S = len(bounds) - 1
    qh = dm.dm_quantize(q.to(DEV), dm.DM_E4M3)
    doh = dm.dm_quantize(do.to(DEV), dm.DM_E5M2)
    full = dm.AttnParams(B, Hq, Hkv, N, d, causal=causal, d_v=d_v)
    blocks = []
    for kb, ke in zip(bounds[:-1], bounds[1:]):
        p = dm.AttnParams(B, Hq, Hkv, N, d, causal=causal, d_v=d_v, kv_offset=kb, kv_len=ke - kb)
        kh = dm.dm_quantize(k[:, :, kb:ke].contiguous().to(DEV), dm.DM_E4M3)
        vh = dm.dm_quantize(v[:, :, kb:ke].contiguous().to(DEV), dm.DM_E4M3)
        blocks.append((p, kh, vh))
    O_parts = torch.empty((S, B, Hq, N, dv), dtype=torch.float32, device=DEV)
    L_parts = torch.empty((S, B, Hq, N), dtype=torch.float32, device=DEV)
    for r, (p, kh, vh) in enumerate(blocks):
        dm.dm_attn_fwd(p, qh, kh, vh, O=O_parts[r], lse=L_parts[r])
    O, lse = dm.dm_attn_merge(full, O_parts, L_parts)
    num = torch.empty((S, B, Hq, N), dtype=torch.float32, device=DEV)
    den = torch.empty_like(num)
    for r, (p, kh, vh) in enumerate(blocks):
        dm.dm_attn_delta_partial(p, qh, kh, vh, doh, lse, num=num[r], den=den[r])
    delta = dm.dm_attn_delta_combine(full, num, den)
    dQ = torch.zeros((B, Hq, N, d), dtype=torch.float32, device=DEV)
    dK = torch.empty((B, Hkv, N, d), dtype=torch.float32, device=DEV)
    dV = torch.empty((B, Hkv, N, dv), dtype=torch.float32, device=DEV)
    for (p, kh, vh), kb, ke in zip(blocks, bounds[:-1], bounds[1:]):
        g = dm.dm_attn_bwd(p, dm.DM_DELTA_MATCHED, qh, kh, vh, doh, lse, delta)
        dQ += g["dQ"]                      # the blocks' partial dQ (a reduction across ranks)
        dK[:, :, kb:ke] = g["dK"]
        dV[:, :, kb:ke] = g["dV"]
    st = dm.dm_get_status()
    assert st == 0, dm.dm_status_string(st)
    return {"O_parts": O_parts, "LSE_parts": L_parts, "O": O, "LSE": lse, "delta": delta, "dQ": dQ, "dK": dK,
            "dV": dV, "blocks": blocks, "q": qh, "do": doh}


def _check(g, r, rf, bounds, keys_unsplit=("LSE", "delta", "dQ", "dK", "dV")):
    for name in ("q", "do"):
        assert np.array_equal(g[name].codes.cpu().numpy(), r[name + "_codes"]), name
        assert np.array_equal(g[name].scales.cpu().numpy(), r[name + "_scales"]), name
    for (p, kh, vh), kb, ke in zip(g["blocks"], bounds[:-1], bounds[1:]):
        for t, name in ((kh, "k"), (vh, "v")):
            assert np.array_equal(t.codes.cpu().numpy(), r[name + "_codes"][:, :, kb:ke]), name
            T0, T1 = kb // 128, (ke + 127) // 128
            assert np.array_equal(t.scales.cpu().numpy(), r[name + "_scales"][:, :, T0:T1]), name
    errs, errs_full = {}, {}
    for key in ("O_parts", "LSE_parts", "O", "LSE", "delta", "dQ", "dK", "dV"):
        got = np32(g[key]).astype(np.float64)
        want = r[key]
        mask = np.isfinite(want)        # rows a block does not see hold LSE = -inf on both sides
        if key == "LSE_parts":  # the same rows see no key of a block on both sides
            sel = ~np.isnan(want)
            assert np.array_equal(np.isneginf(got[sel]), np.isneginf(want[sel]))
        errs[key] = rel_err(got[mask], want[mask])
    for key in keys_unsplit:
        got = np32(g[key]).astype(np.float64)
        mask = ~np.isnan(rf[key])
        errs_full[key] = rel_err(got[mask], rf[key][mask])
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    bad.update({"unsplit " + k: v for k, v in errs_full.items() if not v <= TOL})
    assert not bad, f"errors above {TOL}: {bad}; split {errs}; unsplit {errs_full}"
    return errs, errs_full


@pytest.mark.parametrize("shape,causal,bounds", [
    ((1, 4, 2, 512, 128), True, (0, 256, 512)),
    ((1, 4, 2, 512, 128), False, (0, 128, 384, 512)),
    ((2, 2, 1, 300, 64), True, (0, 128, 300)),          # ragged last block
    ((1, 3, 1, 260, 128), False, (0, 256, 260)),        # a 4-key last block
    ((1, 4, 2, 384, 256), True, (0, 128, 384)),         # head dimension 256 (split backward)
])
def test_key_blocks_match_oracle(shape, causal, bounds):
    B, Hq, Hkv, N, d = shape
    w = custom(B, Hq, Hkv, N, d, causal=causal, seed=N + d + len(bounds))
    q, k, v, do = make_inputs(w)
    g = gpu_key_blocks(q, k, v, do, list(bounds), causal=causal)
    a = [np32(t) for t in (q, k, v, do)]
    r = oracle.pipeline_key_blocks(*a, list(bounds), causal=causal)
    rf = oracle.pipeline(*a, causal=causal)
    errs, errs_full = _check(g, r, rf, bounds)
    print(shape, causal, bounds, "split", errs, "unsplit", errs_full,
          "O vs unsplit", rel_err(np32(g["O"]), rf["O"]))


def test_key_blocks_value_width():
    """Heads shaped like multi-head latent attention (d = 192, d_v = 128)."""
    w = custom(1, 2, 2, 384, 192, causal=True, seed=19, dv=128)
    q, k, v, do = make_inputs(w)
    bounds = [0, 256, 384]
    g = gpu_key_blocks(q, k, v, do, bounds, causal=True, d_v=128)
    a = [np32(t) for t in (q, k, v, do)]
    _check(g, oracle.pipeline_key_blocks(*a, bounds), oracle.pipeline(*a), bounds)


def test_key_blocks_8k_workload_sampled():
    """The 8K workload split into two blocks of 4096 keys (two ranks' share),
    checked on sampled whole tiles at full size."""
    w = WORKLOADS["gqa_b1_n8192_d128"]
    q, k, v, do = make_inputs(w)
    bounds = [0, 4096, 8192]
    g = gpu_key_blocks(q, k, v, do, bounds)
    T = w.N // 128
    q_tiles = [0, 31, 32, 63]
    kv_tiles = [30, 31, 62, 63]
    a = [np32(t) for t in (q, k, v, do)]
    r = oracle.pipeline_key_blocks(*a, bounds, q_tiles=q_tiles, kv_tiles=kv_tiles, groups=[(0, 0)])
    rf = oracle.pipeline(*a, q_tiles=q_tiles, kv_tiles=kv_tiles, groups=[(0, 0)])
    assert T == 64
    errs, errs_full = _check(g, r, rf, bounds)
    print("8k split", errs, "unsplit", errs_full)


def test_key_block_argument_errors():
    w = custom(1, 2, 1, 256, 64)
    q, k, v, do = make_inputs(w)
    qh = dm.dm_quantize(q.to(DEV), dm.DM_E4M3)
    kh = dm.dm_quantize(k[:, :, 128:].contiguous().to(DEV), dm.DM_E4M3)
    for kv_offset, kv_len in ((64, 128), (256, 0), (128, 200), (-128, 0)):
        with pytest.raises(dm.DMError) as e:
            dm.dm_attn_fwd(dm.AttnParams(1, 2, 1, 256, 64, kv_offset=kv_offset, kv_len=kv_len), qh, kh, kh)
        assert e.value.code == dm.DM_ERR_SHAPE
    p = dm.AttnParams(1, 2, 1, 256, 64, kv_offset=128)
    O, lse = dm.dm_attn_fwd(p, qh, kh, kh)
    with pytest.raises(dm.DMError) as e:          # the backward of a key block needs the merged delta
        dm.dm_attn_bwd(p, dm.DM_DELTA_MATCHED, qh, kh, kh, qh, lse, None)
    assert e.value.code == dm.DM_ERR_INVALID_ARG
    # causal: query tile 0 sees no key of the block [128, 256)
    assert torch.all(torch.isneginf(lse[:, :, :128])) and float(O[:, :, :128].abs().max()) == 0.0
    assert dm.dm_get_status() == 0


def test_context_parallel_module_one_rank_nccl():
    """fp8_attention_gb300.context_parallel with the library's kernels and NCCL
    collectives in a one-rank group (the whole sequence as the one key block):
    the same results as the unsplit oracle."""
    import socket

    import torch.distributed as dist

    from fp8_attention_gb300 import context_parallel as cp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=DEV)
    try:
        w = custom(1, 4, 2, 384, 128, seed=23)
        q, k, v, do = make_inputs(w)
        p = dm.AttnParams(w.B, w.Hq, w.Hkv, w.N, w.d, kv_offset=0, kv_len=w.N)
        qh, kh, vh = (dm.dm_quantize(t.to(DEV), dm.DM_E4M3) for t in (q, k, v))
        doh = dm.dm_quantize(do.to(DEV), dm.DM_E5M2)
        res = cp.step(p, qh, kh, vh, doh)
        assert dm.dm_get_status() == 0
        r = oracle.pipeline(*[np32(t) for t in (q, k, v, do)])
        for key in ("O", "LSE", "delta", "dQ", "dK", "dV"):
            assert rel_err(np32(res[key]), r[key]) <= TOL, key
    finally:
        dist.destroy_process_group()
