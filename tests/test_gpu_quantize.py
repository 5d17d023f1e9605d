"""GPU tile quantiser (dm_quantize) against the oracle: codes and scales bit-exact.

Includes an exhaustive sweep of the hardware FP8 conversion through the
public call: every fp32 bit pattern of magnitude <= FMAX is placed in a tile
whose largest element is exactly FMAX, so that r = FMAX/amax = 1 and the code
is the plain RNE/satfinite encoding of the value itself.
"""
import numpy as np
import pytest
import torch

import fp8_attention_gb300 as dm
import oracle
from gpu_common import DEV

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("fmt", [dm.DM_E4M3, dm.DM_E5M2])
@pytest.mark.parametrize("shape", [(1, 2, 256, 64), (2, 3, 200, 128), (1, 1, 77, 64), (1, 2, 1, 128),
                                   (3, 4, 1000, 128), (1, 2, 300, 192), (2, 1, 129, 256), (1, 1, 5, 256)])
def test_quantize_bit_exact(dtype, fmt, shape):
    g = torch.Generator().manual_seed(sum(shape) + fmt)
    x = torch.randn(shape, generator=g) * torch.exp(torch.randn(shape[:3] + (1,), generator=g) * 4)
    x[0, 0, :min(shape[2], 128)] = 0.0                       # all-zero tile
    if shape[2] > 128:
        x[0, -1, 128:] *= 2.0 ** -110                         # tile under the flush threshold
    x = x.to(dtype)
    (got, codes_t) = dm.dm_quantize(x.to(DEV), fmt, want_transposed=True)
    codes, scales = oracle.quantize(x.float().numpy(), fmt)
    assert np.array_equal(got.scales.cpu().numpy(), scales)
    assert np.array_equal(got.codes.cpu().numpy(), codes)
    assert np.array_equal(codes_t.cpu().numpy(), codes.transpose(0, 1, 3, 2))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_batch_matches_oracle(dtype):
    """One launch for Q, K, V (E4M3) and dO (E5M2) of different head counts and a ragged N, plus an empty
    tensor: every tensor's codes and scales bit-exact with the oracle."""
    g = torch.Generator().manual_seed(7)
    shapes = [((2, 4, 333, 128), dm.DM_E4M3), ((2, 1, 333, 128), dm.DM_E4M3), ((2, 1, 333, 128), dm.DM_E4M3),
              ((2, 4, 333, 128), dm.DM_E5M2), ((0, 4, 333, 128), dm.DM_E4M3)]
    xs = []
    for shape, fmt in shapes:
        x = torch.randn(shape, generator=g) * torch.exp(torch.randn(shape[:3] + (1,), generator=g) * 3)
        if fmt == dm.DM_E5M2:
            x *= 1e-3
        xs.append((x.to(dtype), fmt))
    outs = dm.dm_quantize_batch([(x.to(DEV), fmt) for x, fmt in xs])
    for (x, fmt), got in zip(xs, outs):
        if x.numel() == 0:
            assert got.codes.numel() == 0
            continue
        codes, scales = oracle.quantize(x.float().numpy(), fmt)
        assert np.array_equal(got.scales.cpu().numpy(), scales)
        assert np.array_equal(got.codes.cpu().numpy(), codes)


def test_quantize_empty_is_noop():
    x = torch.empty((0, 2, 128, 64), device=DEV)
    out = dm.dm_quantize(x, dm.DM_E4M3)
    assert out.codes.numel() == 0
    x = torch.empty((1, 2, 0, 64), device=DEV)
    out = dm.dm_quantize(x, dm.DM_E4M3)
    assert out.codes.numel() == 0


@pytest.mark.parametrize("fmt", [dm.DM_E4M3, dm.DM_E5M2])
def test_hardware_encode_exhaustive(fmt):
    fmax = np.float32(oracle.FMAX[fmt])
    top = int(fmax.view(np.uint32))
    per_tile = 128 * 64 - 1
    chunk_tiles = 1 << 14
    start = 0
    while start <= top:
        n = min(chunk_tiles * per_tile, top + 1 - start)
        bits = np.arange(start, start + n, dtype=np.uint64).astype(np.uint32)
        tiles = (n + per_tile - 1) // per_tile
        padded = np.zeros(tiles * per_tile, dtype=np.uint32)
        padded[:n] = bits
        body = np.empty((tiles, per_tile + 1), dtype=np.uint32)
        body[:, 0] = fmax.view(np.uint32)
        body[:, 1:] = padded.reshape(tiles, per_tile)
        vals = body.reshape(-1).view(np.float32)
        # odd chunks test the negative half-range
        if (start // (chunk_tiles * per_tile)) % 2 == 1:
            vals = -vals
        x = torch.from_numpy(vals.reshape(1, 1, tiles * 128, 64))
        got = dm.dm_quantize(x.to(DEV), fmt)
        assert np.all(got.scales.cpu().numpy() == np.float32(1.0))
        want = oracle.fp8_encode(vals, fmt)
        g = got.codes.cpu().numpy().reshape(-1)
        bad = np.nonzero(g != want)[0]
        assert bad.size == 0, (f"{bad.size} mismatches, first value {vals[bad[0]]!r}: "
                               f"gpu {g[bad[0]]:#x} oracle {want[bad[0]]:#x}")
        start += n
