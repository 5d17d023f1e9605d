"""Failure detection without a GPU fault: a forward launch told to wait on a
barrier that nothing signals must return DM_ERR_TIMEOUT through dm_get_status
(after its bounded wait expires), leave the context usable, and the next
normal launch must be correct."""
import numpy as np
import pytest

import fp8_attention_gb300 as dm
from fp8_attention_gb300.inputs import WORKLOADS, make_inputs
from gpu_common import DEV, TOL, gpu_pipeline, np32, oracle_pipeline, rel_err

pytestmark = pytest.mark.gpu


def test_stall_times_out_and_recovers():
    w = WORKLOADS["tiny_gqa_n256_d64"]
    q, k, v, do = make_inputs(w)
    p = dm.AttnParams(w.B, w.Hq, w.Hkv, w.N, w.d)
    qh = dm.dm_quantize(q.to(DEV), dm.DM_E4M3)
    kh = dm.dm_quantize(k.to(DEV), dm.DM_E4M3)
    vh = dm.dm_quantize(v.to(DEV), dm.DM_E4M3)
    assert dm.dm_get_status() == dm.DM_OK
    try:
        dm.dm_set_knob(dm.DM_KNOB_WAIT_LIMIT_NS, 50_000_000)   # 50 ms
        dm.dm_set_knob(dm.DM_KNOB_STALL_TEST, 1)
        dm.dm_attn_fwd(p, qh, kh, vh)
        assert dm.dm_get_status() == dm.DM_ERR_TIMEOUT
        assert dm.dm_last_timeout_site() == 103                 # the forward's never-signalled barrier
        assert dm.dm_get_status() == dm.DM_OK                   # cleared by the previous read
    finally:
        dm.dm_set_knob(dm.DM_KNOB_STALL_TEST, 0)
        dm.dm_set_knob(dm.DM_KNOB_WAIT_LIMIT_NS, 0)
    g = gpu_pipeline(q, k, v, do)
    r = oracle_pipeline(q, k, v, do)
    for key in ("O", "LSE", "dQ", "dK", "dV"):
        assert rel_err(np32(g[key]), r[key]) <= TOL, key
