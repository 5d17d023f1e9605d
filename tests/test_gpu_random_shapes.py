"""Seeded random shapes against the oracle: every supported head-dimension
pair (d = d_v in {64, 128, 192, 256}; d != d_v among {128, 192, 256}), random
sequence lengths (ragged tails, lengths below one tile), group sizes, batch
counts, causal and not, each delta mode and both O dtypes.  Same bar as the
fixed-shape tests: codes and scales bit-exact, O, LSE, delta, dQ, dK, dV
within relative Frobenius error 2e-3, matched row sums within the FP32
criterion.
"""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
from fp8_attention_gb300.inputs import custom, make_inputs
from gpu_common import gpu_pipeline, np32, oracle_pipeline
from test_gpu_attention import MODES, _codes_match, _compare, rowsum_check

pytestmark = pytest.mark.gpu

PAIRS = [(64, 64), (128, 128), (192, 192), (256, 256), (192, 128), (256, 128), (128, 192), (256, 192)]


def _cases(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        d, dv = PAIRS[i % len(PAIRS)]
        Hkv = int(rng.choice([1, 2]))
        G = int(rng.choice([1, 2, 3, 4]))
        B = int(rng.choice([1, 2]))
        N = int(rng.integers(1, 420))
        causal = bool(rng.integers(0, 2))
        mode = list(MODES)[int(rng.integers(0, 3))]
        bf16_o = bool(rng.integers(0, 4) == 0)
        out.append((B, G * Hkv, Hkv, N, d, dv, causal, mode, bf16_o, 100 + i))
    return out


@pytest.mark.parametrize("B,Hq,Hkv,N,d,dv,causal,mode,bf16_o,seed", _cases())
def test_random_shape(B, Hq, Hkv, N, d, dv, causal, mode, bf16_o, seed):
    w = custom(B, Hq, Hkv, N, d, causal=causal, seed=seed, dv=dv)
    q, k, v, do = make_inputs(w)
    g = gpu_pipeline(q, k, v, do, causal=causal, mode=mode, diag=True,
                     o_dtype=torch.bfloat16 if bf16_o else torch.float32)
    r = oracle_pipeline(q, k, v, do, causal=causal, mode=MODES[mode], o_bf16=bf16_o, want_diag=True)
    _codes_match(g, r)
    _compare(g, r)
    if mode == dm.DM_DELTA_MATCHED:
        rowsum_check(np32(g["rowsum_pre"]), np32(g["abssum_pre"]), np32(g["delta"]))
