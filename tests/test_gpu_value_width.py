"""Heads whose value dimension differs from the query/key one (shaped like
multi-head latent attention) on the GPU against the oracle.  They run on the
d = 256 kernels, which read the missing channels as zeros through the tensor
maps and write only the real ones; same bar as every other shape: codes and
scales bit-exact, O, LSE, delta, dQ, dK, dV within relative Frobenius error
2e-3, matched row sums within the FP32 criterion.
"""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
import oracle
from fp8_attention_gb300.inputs import WORKLOADS, custom, make_inputs
from gpu_common import gpu_pipeline, np32, oracle_pipeline
from test_gpu_attention import MODES, _codes_match, _compare, rowsum_check
from test_gpu_workloads import _compare_sampled, _sampled

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,causal", [
    ((1, 2, 2, 256, 192, 128), True),    # MLA-shaped, one kv head per query head
    ((1, 2, 2, 300, 192, 128), False),   # ragged, non-causal
    ((2, 4, 2, 200, 256, 128), True),    # GQA, two batches, ragged
    ((1, 2, 1, 384, 128, 256), True),    # value wider than query/key
    ((1, 2, 1, 257, 192, 192), True),    # d = 192 on both sides
    ((1, 1, 1, 1, 192, 128), True),      # a single token
])
def test_value_width_shapes(shape, causal):
    B, Hq, Hkv, N, d, dv = shape
    w = custom(B, Hq, Hkv, N, d, causal=causal, seed=5 * N + d + dv, dv=dv)
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, causal=causal, diag=True)
    r = oracle_pipeline(q, k, v, do, causal=causal, want_diag=True)
    assert g["O"].shape == (B, Hq, N, dv) and g["dV"].shape == (B, Hkv, N, dv) and g["dK"].shape == (B, Hkv, N, d)
    _codes_match(g, r)
    _compare(g, r)
    rowsum_check(np32(g["rowsum_pre"]), np32(g["abssum_pre"]), np32(g["delta"]))


@pytest.mark.parametrize("mode", list(MODES))
def test_value_width_all_modes(mode):
    w = custom(1, 4, 4, 384, 192, seed=41, dv=128)
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, mode=mode, o_dtype=torch.bfloat16 if mode == dm.DM_DELTA_STALE_DO else torch.float32)
    r = oracle_pipeline(q, k, v, do, mode=MODES[mode], o_bf16=mode == dm.DM_DELTA_STALE_DO)
    _compare(g, r)


def test_value_width_delta_inside_backward():
    w = custom(1, 2, 2, 300, 192, seed=43, dv=128)
    q, k, v, do = make_inputs(w)
    for mode in MODES:
        g = gpu_pipeline(q, k, v, do, mode=mode, delta_in_bwd=True)
        r = oracle_pipeline(q, k, v, do, mode=MODES[mode])
        _compare(g, r, keys=("dQ", "dK", "dV"))


def test_mla_b1_n8192_sampled():
    """The MLA-shaped benchmark workload in the benchmark's launch configuration,
    sampled whole tiles against the oracle, row sums over every row."""
    w = WORKLOADS["mla_b1_n8192_d192_dv128"]
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, diag=True)
    q_tiles, kv_tiles = _sampled(w)
    r = oracle_pipeline(q, k, v, do, groups=[(0, 0)], q_tiles=q_tiles, kv_tiles=kv_tiles)
    _codes_match(g, r)
    errs = _compare_sampled(g, r, w)
    rows, needed = rowsum_check(np32(g["rowsum_pre"]), np32(g["abssum_pre"]), np32(g["delta"]))
    assert needed <= 1e-3 * rows + w.B * w.Hq
    print("mla_b1_n8192_d192_dv128 errors", errs, "row-sum rows", rows, "needing the FP32 term", needed)
