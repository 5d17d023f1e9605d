"""GPU attention-input prologue (dm_rope_table, dm_qk_prologue_batch) against
the oracle.  The prologue computes RMSNorm, gains and the rotary rotation in
FP32, the oracle in FP64, so a code may legitimately differ where the exact
pre-rounding value y * r lies within FP32 rounding of a code boundary.  The
test therefore accepts, for every element, exactly the codes that the E4M3
encoder gives for some value within a small band around the oracle's
y * r_gpu (relative 2^-16 plus an absolute 2^-12 in code units, far inside
one E4M3 step), and requires the scales within 2^-19 relative and at most
0.1 % of codes (or two) off the oracle's own."""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
import oracle
from fp8_attention_gb300.inputs import WORKLOADS, custom, make_prologue_inputs
from gpu_common import DEV

pytestmark = pytest.mark.gpu

EPS = dm.RMS_EPS


def _ulp_diff32(a, b):
    ia = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    ib = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(ia - ib)


@pytest.mark.parametrize("N,d", [(8192, 128), (1000, 64), (1, 128), (8192, 256)])
def test_rope_table_matches_oracle(N, d):
    """Within one FP32 ulp of the FP64 value, plus 2^-36 absolute: both sides
    form the angle n * base^(-2i/d) in FP64, whose last-bit differences move
    an angle of a few thousand radians by ~1e-12."""
    cos, sin = dm.dm_rope_table(N, d, device=DEV)
    oc, os_ = oracle.rope_table(N, d)
    for got, want in ((cos, oc), (sin, os_)):
        g = got.cpu().numpy().astype(np.float64)
        tol = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64) + 2.0 ** -36
        assert np.all(np.abs(g - want) <= tol)
    # small angles (position 0 and the first positions) agree to the bit
    k = min(N, 4)
    assert _ulp_diff32(cos.cpu().numpy()[:k], oc[:k].astype(np.float32)).max() == 0


def check_codes(got, x, gain, rope):
    """got: Fp8 from the GPU; x: [B][H][N][d] CPU tensor (the prologue input)."""
    codes_g = got.codes.cpu().numpy()
    scales_g = got.scales.cpu().numpy()
    codes_o, scales_o, y = oracle.qk_prologue_quantized(x.float().numpy(), None if gain is None else gain.numpy(),
                                                        EPS, rope)
    np.testing.assert_allclose(scales_g, scales_o, rtol=2.0 ** -19, atol=0)
    B, H, N, d = y.shape
    rows = np.arange(N) // 128
    s_rows = scales_g[:, :, rows][..., None].astype(np.float64)
    amax_g = np.where(s_rows > 0, s_rows * 448.0, 1.0).astype(np.float32)
    r_g = np.where(s_rows > 0, (np.float32(448.0) / amax_g).astype(np.float64), 0.0)
    t = y * r_g
    band = np.abs(t) * 2.0 ** -16 + 2.0 ** -12
    lo = oracle.fp8_encode((t - band).astype(np.float32), oracle.E4M3)
    hi = oracle.fp8_encode((t + band).astype(np.float32), oracle.E4M3)
    lut = oracle.fp8_decode(np.arange(256, dtype=np.uint8), oracle.E4M3)
    vg, vlo, vhi = lut[codes_g], lut[lo], lut[hi]
    ok = (vg >= np.minimum(vlo, vhi)) & (vg <= np.maximum(vlo, vhi))
    # -0 and +0 both encode zero
    ok |= (vg == 0) & (np.minimum(vlo, vhi) <= 0) & (np.maximum(vlo, vhi) >= 0)
    assert ok.all(), f"{(~ok).sum()} codes outside the rounding band, first at {np.argwhere(~ok)[:3]}"
    assert np.sum(codes_g != codes_o) <= max(2, 1e-3 * codes_g.size)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape", [(1, 2, 256, 64), (2, 3, 300, 128), (1, 1, 1, 128), (1, 4, 1000, 64),
                                   (1, 2, 300, 256), (1, 1, 1, 256)])
@pytest.mark.parametrize("rope,gains", [(True, {7: 5.4, 0: 3.0, 1: 3.0, 2: 3.0}), (False, {}), (True, None)])
def test_prologue_matches_oracle(dtype, shape, rope, gains):
    B, H, N, d = shape
    g = torch.Generator().manual_seed(B * 1000 + H * 100 + N + d)
    x = torch.randn(shape, generator=g) * torch.exp(torch.randn(shape[:3] + (1,), generator=g) * 3)
    if N > 128:
        x[0, 0, :128] = 0.0  # an all-zero tile: scale 0, codes 0
    x = x.to(dtype)
    gain = None
    if gains is not None:
        gain = torch.ones(d)
        for ch, val in gains.items():
            gain[ch] = val
    table = dm.dm_rope_table(N, d, device=DEV) if rope else None
    (got,) = dm.dm_qk_prologue_batch([(x.to(DEV), None if gain is None else gain.to(DEV))], rope=table)
    assert dm.dm_get_status() == 0
    check_codes(got, x, gain, rope)
    if N > 128:
        assert np.all(got.scales.cpu().numpy()[0, 0, 0] == 0.0)
        assert not got.codes.cpu().numpy()[0, 0, :128].any()


@pytest.mark.parametrize("name", ["gqa_b1_n8192_d128", "gqa_b1_n8192_d256"])
def test_prologue_batch_q_and_k_of_the_bench_workload(name):
    """Q and K of an 8K workload (pre-normalisation draws, bf16) in one launch
    at the bench's configuration; whole heads checked against the oracle."""
    w = WORKLOADS[name]
    xq, xk, gain = make_prologue_inputs(w)
    table = dm.dm_rope_table(w.N, w.d, device=DEV)
    gq, gk = dm.dm_qk_prologue_batch([(xq.to(DEV), gain.to(DEV)), (xk.to(DEV), gain.to(DEV))], rope=table)
    assert dm.dm_get_status() == 0
    for got, x, heads in ((gq, xq, [0, w.Hq // 2 + 1, w.Hq - 1]), (gk, xk, [0, w.Hkv - 1])):
        for h in heads:
            sub = dm.Fp8(got.codes[:, h:h + 1].contiguous(), got.scales[:, h:h + 1].contiguous())
            check_codes(sub, x[:, h:h + 1], gain, True)


def test_prologue_saturation_gains_and_empty_job():
    w = custom(1, 2, 1, 4096, 128, gains={7: 5.4, 0: 3.0, 1: 3.0, 2: 3.0}, seed=3)
    xq, xk, gain = make_prologue_inputs(w)
    table = dm.dm_rope_table(w.N, w.d, device=DEV)
    empty = torch.empty((0, 2, 4096, 128), dtype=xq.dtype, device=DEV)
    gq, ge, gk = dm.dm_qk_prologue_batch([(xq.to(DEV), gain.to(DEV)), (empty, gain.to(DEV)),
                                          (xk.to(DEV), gain.to(DEV))], rope=table)
    assert dm.dm_get_status() == 0
    check_codes(gq, xq, gain, True)
    check_codes(gk, xk, gain, True)
    assert ge.codes.numel() == 0
