"""GPU forward / delta / backward against the CPU oracle on the same seeded inputs.

Bar (from the method's acceptance criteria): FP8 codes and scales bit-exact;
O, LSE, delta, dQ, dK, dV within relative Frobenius error 2e-3; matched-delta
rows with |sum_j dS_ij| <= 1e-4 * sum_j |dS_ij| before the E5M2 cast.
"""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
import oracle
from fp8_attention_gb300.inputs import WORKLOADS, custom, make_inputs
from gpu_common import DEV, ROWSUM_TOL, TOL, gpu_pipeline, np32, oracle_pipeline, rel_err

pytestmark = pytest.mark.gpu

MODES = {dm.DM_DELTA_MATCHED: oracle.DELTA_MATCHED, dm.DM_DELTA_STALE_DO: oracle.DELTA_STALE_DO,
         dm.DM_DELTA_STALE_DOHAT: oracle.DELTA_STALE_DOHAT}


def _compare(g, r, keys=("O", "LSE", "delta", "dQ", "dK", "dV"), tol=TOL):
    errs = {}
    for key in keys:
        got = np32(g[key]).astype(np.float64)
        want = r[key]
        mask = ~np.isnan(want)
        errs[key] = rel_err(got[mask], want[mask])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"errors above {tol}: {bad} (all: {errs})"
    return errs


def _codes_match(g, r):
    for name in ("q", "k", "v", "do"):
        assert np.array_equal(g[name].codes.cpu().numpy(), r[name + "_codes"]), name
        assert np.array_equal(g[name].scales.cpu().numpy(), r[name + "_scales"]), name


@pytest.mark.parametrize("mode", list(MODES))
def test_tiny_gqa_all_modes(mode):
    w = WORKLOADS["tiny_gqa_n256_d64"]
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, mode=mode, diag=True)
    r = oracle_pipeline(q, k, v, do, mode=MODES[mode], want_diag=True)
    _codes_match(g, r)
    _compare(g, r)


@pytest.mark.parametrize("shape,causal", [
    ((1, 2, 1, 384, 128), True),
    ((1, 4, 2, 256, 128), False),
    ((2, 2, 2, 200, 64), True),       # ragged tail
    ((1, 2, 1, 333, 128), False),     # ragged, non-causal
    ((1, 1, 1, 1, 64), True),         # a single token
    ((1, 3, 1, 130, 128), True),      # 3 query heads per kv head, tail of 2 rows
])
def test_shapes(shape, causal):
    B, Hq, Hkv, N, d = shape
    w = custom(B, Hq, Hkv, N, d, causal=causal, seed=N + d)
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, causal=causal, diag=True)
    r = oracle_pipeline(q, k, v, do, causal=causal, want_diag=True)
    _codes_match(g, r)
    _compare(g, r)


@pytest.mark.parametrize("shape,causal", [
    ((1, 2, 1, 127, 128), True),      # one row short of a tile
    ((1, 2, 1, 129, 128), True),      # one row past a tile
    ((1, 2, 2, 255, 64), False),      # multi-head (G = 1), one short of two tiles
    ((1, 2, 2, 257, 64), True),
    ((3, 8, 1, 96, 64), True),        # G = 8, several batches, a single partial tile
    ((1, 4, 2, 513, 128), True),      # five key tiles, the last one row long
])
def test_tile_boundaries_and_group_sizes(shape, causal):
    """Sequence lengths at tile edges (every kernel's ragged path), group sizes
    1 and 8 and several batches: codes bit-exact, results within the bar."""
    B, Hq, Hkv, N, d = shape
    w = custom(B, Hq, Hkv, N, d, causal=causal, seed=7 * N + d)
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, causal=causal)
    r = oracle_pipeline(q, k, v, do, causal=causal)
    _codes_match(g, r)
    _compare(g, r)


def test_bf16_output_and_explicit_scale():
    w = custom(1, 4, 2, 256, 128, seed=3)
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, o_dtype=torch.bfloat16, sigma=0.07, mode=dm.DM_DELTA_STALE_DO)
    r = oracle_pipeline(q, k, v, do, o_bf16=True, sigma=0.07, mode=oracle.DELTA_STALE_DO)
    _compare(g, r)


def test_delta_computed_inside_backward():
    w = custom(1, 4, 1, 300, 64, seed=5)
    q, k, v, do = make_inputs(w)
    for mode in MODES:
        g = gpu_pipeline(q, k, v, do, mode=mode, delta_in_bwd=True)
        r = oracle_pipeline(q, k, v, do, mode=MODES[mode])
        _compare(g, r, keys=("dQ", "dK", "dV"))


def rowsum_check(rs, ab, delta):
    """Matched delta brings the row sums of dS back to zero within FP32 rounding (project page section 03):
    every row must satisfy |sum_j dS_ij| <= 1e-4 * sum_j |dS_ij| + 2^-20 * |delta_i|.  The second
    term is the FP32 resolution of delta (16 units in its last place): in near-one-hot rows
    sum_j |dS_ij| is only ~1e-3 |delta_i| (one key carries P ~ 1 and dP ~ delta), and the relative
    term alone would ask for less than one ulp of delta.
    Returns (rows, rows that needed the FP32 term)."""
    floor = 2.0 ** -20 * np.abs(delta)
    ok = np.abs(rs) <= ROWSUM_TOL * ab + floor
    needed = np.abs(rs) > ROWSUM_TOL * ab
    if needed.any():
        print("rows needing the FP32 term:", int(needed.sum()), "of", rs.size,
              "max |sum dS|/|delta| there:", float(np.max(np.abs(rs[needed]) / np.abs(delta[needed]))))
    assert ok.all(), float(np.max((np.abs(rs) - floor) / np.maximum(ab, 1e-38)))
    return rs.size, int(needed.sum())


def test_matched_rows_sum_to_zero_and_stale_do_not():
    w = custom(1, 4, 1, 512, 128, seed=7)
    q, k, v, do = make_inputs(w)
    res = {}
    for mode in (dm.DM_DELTA_MATCHED, dm.DM_DELTA_STALE_DO):
        g = gpu_pipeline(q, k, v, do, mode=mode, diag=True)
        res[mode] = tuple(np32(g[n]) for n in ("rowsum_pre", "abssum_pre", "rowsum_post", "abssum_post",
                                                "delta"))
    rs, ab, _, _, delta = res[dm.DM_DELTA_MATCHED]
    rows, needed = rowsum_check(rs, ab, delta)
    assert needed <= 1e-3 * rows + 4   # plus row 0 of each causal head: a single key, dS is pure rounding
    # the stale correction leaves residuals far above both terms
    rs_s, ab_s = res[dm.DM_DELTA_STALE_DO][:2]
    live = ab_s > 0
    assert np.median(np.abs(rs_s[live]) / ab_s[live]) > 10 * ROWSUM_TOL


def test_diagnostics_match_oracle():
    w = WORKLOADS["tiny_gqa_n256_d64"]
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, diag=True)
    r = oracle_pipeline(q, k, v, do, want_diag=True)
    d = r["diag"]
    # absolute sums are well conditioned; compare them with the tensor tolerance
    assert rel_err(np32(g["abssum_pre"]), d[1]) <= TOL
    assert rel_err(np32(g["abssum_post"]), d[3]) <= TOL


def test_empty_inputs_are_noops():
    p = dm.AttnParams(0, 2, 1, 128, 64)
    empty = dm.Fp8(torch.empty(0, dtype=torch.uint8, device=DEV), torch.empty(0, device=DEV))
    O, lse = dm.dm_attn_fwd(p, empty, empty, empty)
    assert O.numel() == 0 and lse.numel() == 0
    p = dm.AttnParams(1, 2, 1, 0, 64)
    O, lse = dm.dm_attn_fwd(p, empty, empty, empty)
    assert O.numel() == 0


def test_argument_errors_do_not_launch():
    w = custom(1, 2, 1, 128, 64)
    q, k, v, do = make_inputs(w)
    qh = dm.dm_quantize(q.to(DEV), dm.DM_E4M3)
    with pytest.raises(dm.DMError) as e:
        dm.dm_attn_fwd(dm.AttnParams(1, 2, 1, 128, 96), qh, qh, qh)
    assert e.value.code == dm.DM_ERR_SHAPE
    with pytest.raises(dm.DMError) as e:
        dm.dm_attn_fwd(dm.AttnParams(1, 3, 2, 128, 64), qh, qh, qh)
    assert e.value.code == dm.DM_ERR_SHAPE
    bad = dm.Fp8(qh.codes.view(-1)[1:], qh.scales)          # misaligned codes pointer
    with pytest.raises(dm.DMError) as e:
        dm.dm_attn_fwd(dm.AttnParams(1, 2, 1, 127, 64), bad, qh, qh)
    assert e.value.code == dm.DM_ERR_ALIGNMENT
    with pytest.raises(dm.DMError) as e:
        dm.dm_quantize(q.to(DEV).half(), dm.DM_E4M3)
    assert e.value.code == dm.DM_ERR_DTYPE
    assert dm.dm_get_status() == 0
