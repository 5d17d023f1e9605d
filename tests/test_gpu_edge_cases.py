"""Edge cases of the method on the GPU, against the oracle on the same inputs.

The per-tile FP32 scales of the method ("Delta-Matching for reliable FP8
attention training", section 01, "What changes in FP8?") give every key tile
(forward) and every query tile (backward) its own scale product, so the
kernels' accumulators change units from tile to tile.  These cases put the
unit bookkeeping at its limits:

* an all-zero K tile, a V tile below the quantiser's 2^-96 flush, an all-zero
  dO tile and a flushed dO tile inside attention (tiles that add exactly
  nothing, or whose scale is zero);
* dO at 1e-25 (far below the workloads' 1e-3 but well above the flush), where
  the backward's scale products fall near 2^-105;
* a row maximum that jumps by ~95 (in score units) at the last key tile,
  whose V tile is scaled by 2^-70: the last tile then dominates those rows
  although its scale product is 2^70 below the running unit (all rows of the
  query tile, or every other row so that the rest keep their earlier unit).

Each result is compared within the 2e-3 relative Frobenius bound over the
whole tensor and, where the effect is confined to some rows, over those rows
alone; FP8 codes and scales of Q, K, V, dO are bit-exact.
"""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
import oracle
from gpu_common import TOL, gpu_pipeline, np32, oracle_pipeline, rel_err
from test_gpu_attention import _codes_match, _compare

pytestmark = pytest.mark.gpu


def _randn(gen, *shape):
    return torch.randn(*shape, generator=gen, dtype=torch.float32)


def _region_errors(g, r, regions):
    """rel_err of each (key, index) region; index selects rows of the tensor."""
    errs = {}
    for key, idx in regions:
        got = np32(g[key]).astype(np.float64)[idx]
        want = r[key][idx]
        errs[(key, str(idx))] = rel_err(got, want)
    bad = {k: v for k, v in errs.items() if not v <= TOL}
    assert not bad, f"region errors above {TOL}: {bad}"
    return errs


@pytest.mark.parametrize("mode", [dm.DM_DELTA_MATCHED, dm.DM_DELTA_STALE_DO])
def test_zero_and_flushed_tiles(mode):
    gen = torch.Generator().manual_seed(31)
    B, Hq, Hkv, N, d = 1, 2, 1, 512, 128
    q = _randn(gen, B, Hq, N, d)
    k = _randn(gen, B, Hkv, N, d)
    v = _randn(gen, B, Hkv, N, d)
    do = 1e-3 * _randn(gen, B, Hq, N, d)
    k[:, :, 128:256] = 0.0                 # key tile 1: all zero (scale 0)
    v[:, :, 256:384] *= 1e-31              # value tile 2: amax below 2^-96, flushed
    do[:, 0, 384:512] = 0.0                # head 0, query tile 3: dO all zero
    do[:, 1, 128:256] *= 1e-28             # head 1, query tile 1: flushed
    omode = {dm.DM_DELTA_MATCHED: oracle.DELTA_MATCHED, dm.DM_DELTA_STALE_DO: oracle.DELTA_STALE_DO}[mode]
    g = gpu_pipeline(q, k, v, do, mode=mode)
    r = oracle_pipeline(q, k, v, do, mode=omode)
    assert float(g["k"].scales[0, 0, 1]) == 0.0 and float(g["v"].scales[0, 0, 2]) == 0.0
    assert float(g["do"].scales[0, 0, 3]) == 0.0 and float(g["do"].scales[0, 1, 1]) == 0.0
    _codes_match(g, r)
    errs = _compare(g, r)
    # the rows whose dO is zero have zero dQ; the others within the bar
    assert float(g["dQ"][0, 0, 384:].abs().max()) == 0.0
    _region_errors(g, r, [("dQ", np.s_[:, 0, :384]), ("dQ", np.s_[:, 1, 256:]), ("O", np.s_[:, :, 256:])])
    print("zero/flushed tiles", errs)


@pytest.mark.parametrize("storage", [torch.float32, torch.bfloat16])
def test_tiny_dO(storage):
    """dO = 1e-25 N(0, 1): every gradient (1e-25 scale) within the bar."""
    gen = torch.Generator().manual_seed(32)
    B, Hq, Hkv, N, d = 1, 4, 2, 384, 128
    q = _randn(gen, B, Hq, N, d)
    k = _randn(gen, B, Hkv, N, d)
    v = _randn(gen, B, Hkv, N, d)
    do = 1e-25 * _randn(gen, B, Hq, N, d)
    q, k, v, do = (t.to(storage) for t in (q, k, v, do))
    g = gpu_pipeline(q, k, v, do)
    r = oracle_pipeline(q, k, v, do)
    _codes_match(g, r)
    errs = _compare(g, r)
    assert np.abs(r["dV"]).max() < 1e-20 and np.abs(r["dV"]).max() > 0
    print("tiny dO", errs)


@pytest.mark.parametrize("every_row", [True, False])
def test_late_row_max_jump_onto_tiny_value_tile(every_row):
    """Key tile 2 carries a key direction that the query rows of tile 2
    align with (scores ~100 against ~5 elsewhere) and a V tile scaled by
    2^-70: for those rows alpha ~ e^-95 and the last tile's contribution,
    2^70 below the running unit, is all there is.  every_row=False: only the
    even rows jump; the odd rows keep their earlier maximum and unit."""
    gen = torch.Generator().manual_seed(33)
    B, Hq, Hkv, N, d = 1, 2, 1, 384, 64
    q = _randn(gen, B, Hq, N, d)
    k = _randn(gen, B, Hkv, N, d)
    v = _randn(gen, B, Hkv, N, d)
    do = 1e-3 * _randn(gen, B, Hq, N, d)
    k[..., 0] = 0.0
    k[:, :, 256:, 0] = 80.0                # sigma * 10 * 80 = 100
    q[..., 0] = 0.0
    jump = np.arange(256, 384) if every_row else np.arange(256, 384, 2)
    q[:, :, jump, 0] = 10.0
    v[:, :, 256:] *= 2.0 ** -70
    g = gpu_pipeline(q, k, v, do)
    r = oracle_pipeline(q, k, v, do)
    _codes_match(g, r)
    errs = _compare(g, r)
    # the rows that jumped: O, delta and dQ at the 2^-70 scale
    rj = np.s_[:, :, jump]
    regions = [("O", rj), ("delta", rj), ("LSE", rj), ("dK", np.s_[:, :, 256:]), ("dV", np.s_[:, :, 256:])]
    if every_row:
        regions.append(("dQ", rj))
    else:
        # the jumping rows' dS (~1e-23) shares its E5M2 tile scale with the odd
        # rows' (~1e-5): it flushes to zero on both sides
        rest = np.s_[:, :, np.arange(257, 384, 2)]
        regions += [("O", rest), ("dQ", rest)]
    assert np.abs(r["O"][rj]).max() < 2.0 ** -60
    rerr = _region_errors(g, r, regions)
    print("late jump", errs, rerr)
