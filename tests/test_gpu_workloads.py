"""Parity on the full-size workloads, in the launch configuration the benchmark times.

The oracle cannot redo the 8K and 64K workloads in seconds, so those are
checked on sampled whole tiles (a P or dS tile's scale depends on all of its
128 rows): query tiles {0, T/3, 2T/3, T-1} of kv group (b=0, g=0) for O, LSE,
delta and dQ, and the last key tiles for dK and dV (they depend only on the
query tiles at or after them).  The 64K workload's dK/dV are in addition
checked through invariants that hold at any size.
"""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
import oracle
from fp8_attention_gb300.inputs import WORKLOADS, make_inputs
from gpu_common import ROWSUM_TOL, TOL, gpu_pipeline, np32, oracle_pipeline, rel_err
from test_gpu_attention import _codes_match, _compare, rowsum_check

pytestmark = pytest.mark.gpu


def _sampled(w):
    T = (w.N + 127) // 128
    q_tiles = sorted({0, T // 3, (2 * T) // 3, T - 1})
    kv_tiles = [T - 2, T - 1]
    return q_tiles, kv_tiles


def _compare_sampled(g, r, w):
    # the oracle leaves unselected rows at NaN; compare the rest
    errs = {}
    for key in ("O", "LSE", "delta", "dQ", "dK", "dV"):
        want = r[key]
        got = np32(g[key]).astype(np.float64)
        mask = ~np.isnan(want)
        assert mask.any(), key
        errs[key] = rel_err(got[mask], want[mask])
    assert all(v <= TOL for v in errs.values()), errs
    return errs


def test_gqa_b4_n2048_full_groups():
    w = WORKLOADS["gqa_b4_n2048_d128"]
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, diag=True)
    r = oracle_pipeline(q, k, v, do, groups=[(0, 0), (3, 3)], q_tiles=list(range(16)),
                        kv_tiles=list(range(16)))
    _codes_match(g, r)
    errs = _compare_sampled(g, r, w)
    print("gqa_b4_n2048 errors", errs)
    rowsum_check(np32(g["rowsum_pre"]), np32(g["abssum_pre"]), np32(g["delta"]))


@pytest.mark.parametrize("name", ["gqa_b1_n8192_d128", "saturation_b2_n4096_d128"])
def test_long_workloads_sampled(name):
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, diag=True)
    q_tiles, kv_tiles = _sampled(w)
    r = oracle_pipeline(q, k, v, do, groups=[(0, 0)], q_tiles=q_tiles, kv_tiles=kv_tiles)
    _codes_match(g, r)
    errs = _compare_sampled(g, r, w)
    rows, needed = rowsum_check(np32(g["rowsum_pre"]), np32(g["abssum_pre"]), np32(g["delta"]))
    assert needed <= 1e-3 * rows + w.B * w.Hq   # plus row 0 of each causal head (a single key)
    print(name, "errors", errs, "row-sum rows", rows, "needing the FP32 term", needed)


@pytest.mark.parametrize("mode,omode", [(dm.DM_DELTA_STALE_DO, oracle.DELTA_STALE_DO),
                                        (dm.DM_DELTA_STALE_DOHAT, oracle.DELTA_STALE_DOHAT)])
def test_saturation_stale_modes_sampled(mode, omode):
    """The stale corrections (diagnostic modes: section 01's saved-output
    shortcut and section 03's dO-matched one) at full size on the saturation
    workload, where they differ most from the matched one: sampled whole tiles
    in the launch configuration the benchmark times."""
    w = WORKLOADS["saturation_b2_n4096_d128"]
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, mode=mode)
    q_tiles, kv_tiles = _sampled(w)
    r = oracle_pipeline(q, k, v, do, mode=omode, groups=[(1, 3)], q_tiles=q_tiles, kv_tiles=kv_tiles)
    _codes_match(g, r)
    errs = _compare_sampled(g, r, w)
    print(w.name, "mode", mode, "errors", errs)


def test_saturation_post_cast_residual_ratio():
    """Section 03 reports post-cast row-sum residuals 5.3-6.3x larger with stale delta than
    with Delta-Matching on the authors' probes (workload unstated); here the ratio of
    mean_i |sum_j dS^_ij| / sum_j |dS^_ij| on the saturation workload is measured and must
    favour the matched correction."""
    w = WORKLOADS["saturation_b2_n4096_d128"]
    q, k, v, do = make_inputs(w)
    ratios = {}
    for mode in (dm.DM_DELTA_MATCHED, dm.DM_DELTA_STALE_DO):
        g = gpu_pipeline(q, k, v, do, mode=mode, diag=True)
        rs, ab = np32(g["rowsum_post"]), np32(g["abssum_post"])
        live = ab > 0
        ratios[mode] = float(np.mean(np.abs(rs[live]) / ab[live]))
    ratio = ratios[dm.DM_DELTA_STALE_DO] / ratios[dm.DM_DELTA_MATCHED]
    print("post-cast normalised row-sum residual stale/matched = %.2f (%s)" % (ratio, ratios))
    assert ratio > 1.0


def test_long_64k_sampled_and_invariants():
    w = WORKLOADS["long_b1_n65536_d128"]
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do)
    q_tiles, kv_tiles = _sampled(w)
    r = oracle_pipeline(q, k, v, do, groups=[(0, 0)], q_tiles=q_tiles, kv_tiles=kv_tiles)
    _codes_match(g, r)
    errs = _compare_sampled(g, r, w)
    print("long_64k errors", errs)
    # invariants over all key rows: sum_j dK_j ~ 0 (zero row sums of dS), and
    # sum_j dV_j ~ sum_i (sum_j P^_ij) dO^_i ~ sum_i dO^_i (rows of P^ sum to 1 within FP8 error)
    dK, dV = g["dK"].double(), g["dV"].double()
    sum_dk = dK.sum(dim=2)
    assert float(sum_dk.norm() / dK.abs().sum(dim=2).norm()) < 1e-2
    G = w.Hq // w.Hkv
    dohat = g["do"].codes.view(torch.float8_e5m2).double() * g["do"].scales.double().repeat_interleave(128, dim=2)[
        :, :, :w.N, None]
    want = dohat.reshape(w.B, w.Hkv, G, w.N, w.d).sum(dim=(2, 3))
    assert float((dV.sum(dim=2) - want).norm() / want.norm()) < 0.05


@pytest.mark.parametrize("mode,omode", [(dm.DM_DELTA_MATCHED, oracle.DELTA_MATCHED),
                                        (dm.DM_DELTA_STALE_DOHAT, oracle.DELTA_STALE_DOHAT)])
def test_non_causal_1k_groups(mode, omode):
    """Non-causal attention at a size where every CTA loops over eight key or
    query tiles, two whole kv groups checked, in the matched and one stale mode."""
    from fp8_attention_gb300.inputs import custom
    w = custom(2, 8, 2, 1024, 128, causal=False, seed=11)
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, causal=False, mode=mode)
    r = oracle_pipeline(q, k, v, do, causal=False, mode=omode, groups=[(0, 0), (1, 1)],
                        q_tiles=list(range(8)), kv_tiles=list(range(8)))
    _codes_match(g, r)
    errs = _compare_sampled(g, r, w)
    print("non-causal 1k errors", errs)
