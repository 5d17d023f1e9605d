"""CPU oracle for Delta-Matching FP8 attention -- TEST INFRASTRUCTURE ONLY.

A plain FP64 restatement of the computation described on the project page
"Delta-Matching for reliable FP8 attention training" (sections 01-03), in
``oracle.cpp``, loaded through ctypes.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it; the
product package never does, and the two share no code.

Every array here is numpy, laid out [B][H][N][d] (d fastest).  FP8 formats:
0 = E4M3, 1 = E5M2.  Flags for the attention calls (combine with ``|``):

* ``QUANT_P_FWD``  quantise the forward P~ per 128x128 tile (one-pass contract)
* ``QUANT_P_BWD``  quantise the backward P per 128x128 tile
* ``QUANT_DS``     quantise dS per 128x128 tile
* ``ROUND32``      round P~, P and dS to FP32 where the GPU holds them in FP32
* ``GPU_CONTRACT`` all four: the exact contract the CUDA path implements
* ``EXACT``        none: plain attention in FP64

Parity status: every function below is pinned by ``tests/test_oracle_*.py``
(see the module docstrings there): the backward's per-tile P^ and dS^
quantisation and the one-pass forward over several key tiles by
``tests/test_oracle_tile_pins.py`` (torch-cast emulations on exact grid
inputs).  Nothing here is "parity unpinned" except the full-size dK/dV of the
65536-token workload, which tests only check through invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

E4M3, E5M2 = 0, 1
QUANT_P_FWD, QUANT_P_BWD, QUANT_DS, ROUND32 = 1, 2, 4, 8
GPU_CONTRACT = QUANT_P_FWD | QUANT_P_BWD | QUANT_DS | ROUND32
EXACT = 0
DELTA_MATCHED, DELTA_STALE_DO, DELTA_STALE_DOHAT = 0, 1, 2
FMAX = {E4M3: 448.0, E5M2: 57344.0}
TILE = 128

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so with the host g++ (OpenMP, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared",
               "-ffp-contract=off", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            lib.or_fp8_decode.restype = D
            lib.or_fp8_decode.argtypes = [ctypes.c_uint8, I]
            lib.or_fp8_encode.restype = ctypes.c_uint8
            lib.or_fp8_encode.argtypes = [ctypes.c_float, I]
            lib.or_fp8_encode_array.argtypes = [P, ctypes.c_int64, I, P]
            lib.or_quantize.restype = I
            lib.or_quantize.argtypes = [P, I, I, I, I, I, P, P]
            lib.or_dequantize.argtypes = [P, P, I, I, I, I, I, P]
            lib.or_attn_fwd.restype = I
            lib.or_attn_fwd.argtypes = [I, I, I, I, I, I, I, D, I, P, P, P, P, I, P, I, P, P, P, I, I]
            lib.or_attn_delta.restype = I
            lib.or_attn_delta.argtypes = [I, I, I, I, I, I, I, D, I, I, P, P, P, P, P, P, P, P, I, P, I, P,
                                          I, I, P]
            lib.or_attn_bwd.restype = I
            lib.or_attn_bwd.argtypes = [I, I, I, I, I, I, I, D, I, P, P, P, P, P, P,
                                        P, I, P, I, P, I, P, P, P, P, P, P, P, I, I]
            lib.or_attn_merge.restype = I
            lib.or_attn_merge.argtypes = [I, ctypes.c_int64, I, P, P, P, P]
            lib.or_rope_table.argtypes = [I, I, D, P, P]
            lib.or_qk_prologue.restype = I
            lib.or_qk_prologue.argtypes = [P, I, I, I, I, P, D, I, D, P]
            lib.or_num_threads.restype = I
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _check(Q, K, V, *rows_v):
    """Shape checks: Q [B][Hq][N][d], K [B][Hkv][N][d], V [B][Hkv][N][dv] (dv may
    differ from d), Hkv | Hq; rows_v arrays (dO, O) [B][Hq][N][dv]."""
    if Q.ndim != 4 or K.ndim != 4 or V.ndim != 4 or K.shape[:3] != V.shape[:3]:
        raise ValueError("Q, K, V must be [B][H][N][d] with K and V of the same B, H, N")
    B, Hq, N, d = Q.shape
    if K.shape[0] != B or K.shape[2:] != (N, d) or Hq % K.shape[1]:
        raise ValueError(f"shape mismatch: Q {Q.shape} K {K.shape}")
    for a in rows_v:
        if a is not None and a.shape != (B, Hq, N, V.shape[3]):
            raise ValueError(f"shape mismatch: {a.shape} vs (B, Hq, N, dv) {(B, Hq, N, V.shape[3])}")


def _sel(tiles):
    if tiles is None:
        return None, 0
    arr = np.ascontiguousarray(np.asarray(tiles, dtype=np.int32))
    return arr, int(arr.size)


def _groups(groups):
    if groups is None:
        return None, 0
    arr = np.ascontiguousarray(np.asarray(groups, dtype=np.int32).reshape(-1, 2))
    return arr, int(arr.shape[0])


def num_threads() -> int:
    return _load().or_num_threads()


# --------------------------------------------------------------------- codec
def fp8_decode(codes, fmt: int) -> np.ndarray:
    """Value of each FP8 code (OCP OFP8), as float64."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.or_fp8_decode(int(v), fmt) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def fp8_encode(x, fmt: int) -> np.ndarray:
    """Round-to-nearest-even, saturating FP8 encoding of fp32 values."""
    lib = _load()
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(xa.shape, dtype=np.uint8)
    lib.or_fp8_encode_array(_p(xa), xa.size, fmt, _p(out))
    return out


def quantize(x, fmt: int):
    """Per 128-row x d tile quantisation of a [B][H][N][d] fp32 tensor -> (codes, scales)."""
    lib = _load()
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    B, H, N, d = xa.shape
    T = (N + TILE - 1) // TILE
    codes = np.empty(xa.shape, dtype=np.uint8)
    scales = np.empty((B, H, T), dtype=np.float32)
    if lib.or_quantize(_p(xa), B, H, N, d, fmt, _p(codes), _p(scales)) != 0:
        raise ValueError("or_quantize: bad arguments")
    return codes, scales


def dequantize(codes, scales, fmt: int) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.float32)
    B, H, N, d = c.shape
    out = np.empty(c.shape, dtype=np.float64)
    lib.or_dequantize(_p(c), _p(s), B, H, N, d, fmt, _p(out))
    return out


# ----------------------------------------------------------------- attention
def _kv_range(kv_range):
    """(begin, end) of a key range for the C calls; None selects every key."""
    if kv_range is None:
        return 0, 0
    b, e = kv_range
    return int(b), int(e)


def attn_fwd(Q, K, V, causal=True, sigma=0.0, flags=GPU_CONTRACT, q_tiles=None, groups=None,
             want_pfwd=False, kv_range=None):
    """Forward on decoded operands.  Returns (O, LSE[, Pfwd]) in FP64.

    Rows outside the selected query tiles / groups are left at NaN.  kv_range
    = (begin, end) restricts attention to those keys (a key block of
    context-parallel attention; rows seeing none get O = 0, LSE = -inf)."""
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    _check(Q, K, V)
    B, Hq, N, d = Q.shape
    Hkv, dv = K.shape[1], V.shape[3]
    O = np.full((B, Hq, N, dv), np.nan)
    LSE = np.full((B, Hq, N), np.nan)
    P = np.zeros((B, Hq, N, N)) if want_pfwd else None
    qs, nq = _sel(q_tiles)
    gs, ng = _groups(groups)
    kb, ke = _kv_range(kv_range)
    rc = lib.or_attn_fwd(B, Hq, Hkv, N, d, dv, int(causal), float(sigma), int(flags), _p(Q), _p(K), _p(V),
                         _p(qs), nq, _p(gs), ng, _p(O), _p(LSE), _p(P), kb, ke)
    if rc != 0:
        raise ValueError("or_attn_fwd: bad arguments")
    return (O, LSE, P) if want_pfwd else (O, LSE)


def attn_delta(Q, K, V, dOhat, LSE, mode=DELTA_MATCHED, dO=None, O=None, causal=True, sigma=0.0,
               flags=GPU_CONTRACT, q_tiles=None, groups=None, kv_range=None, partial=False):
    """Softmax row correction delta [B][Hq][N] for the given mode.  Matched mode
    with kv_range sums over those keys only; partial=True returns the two sums
    (sum_j P dP^, sum_j P) apart instead of their quotient."""
    lib = _load()
    Q, K, V, dOhat, LSE = _f64(Q), _f64(K), _f64(V), _f64(dOhat), _f64(LSE)
    dO, O = _f64(dO), _f64(O)
    _check(Q, K, V, dOhat, dO, O)
    if LSE.shape != Q.shape[:3]:
        raise ValueError("LSE must be [B][Hq][N]")
    if mode == DELTA_STALE_DO and (dO is None or O is None):
        raise ValueError("stale_dO needs dO and O")
    if mode == DELTA_STALE_DOHAT and O is None:
        raise ValueError("stale_dOhat needs O")
    B, Hq, N, d = Q.shape
    Hkv, dv = K.shape[1], V.shape[3]
    delta = np.full((B, Hq, N), np.nan)
    den = np.full((B, Hq, N), np.nan) if partial else None
    qs, nq = _sel(q_tiles)
    gs, ng = _groups(groups)
    kb, ke = _kv_range(kv_range)
    rc = lib.or_attn_delta(B, Hq, Hkv, N, d, dv, int(causal), float(sigma), int(flags), int(mode),
                           _p(Q), _p(K), _p(V), _p(dOhat), _p(dO), _p(O), _p(LSE),
                           _p(qs), nq, _p(gs), ng, _p(delta), kb, ke, _p(den))
    if rc != 0:
        raise ValueError("or_attn_delta: bad arguments")
    return (delta, den) if partial else delta


def attn_bwd(Q, K, V, dOhat, LSE, delta, causal=True, sigma=0.0, flags=GPU_CONTRACT, q_tiles=None,
             kv_tiles=None, groups=None, want_diag=False, want_tiles=False, kv_range=None):
    """Backward on decoded operands.  Returns dict with dQ, dK, dV (+ diag, dS, dShat, Phat).
    With kv_range only those keys take part: dQ is the key block's partial sum."""
    lib = _load()
    Q, K, V, dOhat, LSE, delta = _f64(Q), _f64(K), _f64(V), _f64(dOhat), _f64(LSE), _f64(delta)
    _check(Q, K, V, dOhat)
    if LSE.shape != Q.shape[:3] or delta.shape != Q.shape[:3]:
        raise ValueError("LSE and delta must be [B][Hq][N]")
    B, Hq, N, d = Q.shape
    Hkv, dv = K.shape[1], V.shape[3]
    out = {
        "dQ": np.full(Q.shape, np.nan),
        "dK": np.full(K.shape, np.nan),
        "dV": np.full(V.shape, np.nan),
    }
    diag = np.full((4, B, Hq, N), np.nan) if want_diag else None
    tiles = [np.zeros((B, Hq, N, N)) for _ in range(3)] if want_tiles else [None] * 3
    qs, nq = _sel(q_tiles)
    ks, nk = _sel(kv_tiles)
    gs, ng = _groups(groups)
    rc = lib.or_attn_bwd(B, Hq, Hkv, N, d, dv, int(causal), float(sigma), int(flags),
                         _p(Q), _p(K), _p(V), _p(dOhat), _p(LSE), _p(delta),
                         _p(qs), nq, _p(ks), nk, _p(gs), ng,
                         _p(out["dQ"]), _p(out["dK"]), _p(out["dV"]), _p(diag),
                         _p(tiles[0]), _p(tiles[1]), _p(tiles[2]), *_kv_range(kv_range))
    if rc != 0:
        raise ValueError("or_attn_bwd: bad arguments")
    if want_diag:
        out["diag"] = diag
    if want_tiles:
        out["dS"], out["dShat"], out["Phat"] = tiles
    return out


def attn_merge(O_parts, LSE_parts):
    """Merge of per-key-block attention results: O_parts [S][B][H][N][dv],
    LSE_parts [S][B][H][N] -> (O, LSE) of the union of the blocks."""
    lib = _load()
    Op = np.ascontiguousarray(O_parts, dtype=np.float64)
    Lp = np.ascontiguousarray(LSE_parts, dtype=np.float64)
    S = Op.shape[0]
    rows = int(np.prod(Lp.shape[1:]))
    dv = Op.shape[-1]
    if Op.shape[:-1] != Lp.shape:
        raise ValueError("O_parts must be LSE_parts' shape plus a value dimension")
    O = np.empty(Op.shape[1:])
    LSE = np.empty(Lp.shape[1:])
    if lib.or_attn_merge(S, rows, dv, _p(Op), _p(Lp), _p(O), _p(LSE)) != 0:
        raise ValueError("or_attn_merge: bad arguments")
    return O, LSE


# ------------------------------------------------------------ whole pipeline
def round_bf16(x) -> np.ndarray:
    """Round float values to bfloat16 (nearest even) and return them as float64."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    out = rounded.astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(a)
    out[nan] = np.nan
    return out


def pipeline(q, k, v, do, causal=True, sigma=0.0, mode=DELTA_MATCHED, o_bf16=False,
             q_tiles=None, kv_tiles=None, groups=None, want_diag=False, flags=GPU_CONTRACT):
    """Quantise the fp32 inputs, then forward, delta and backward under the GPU contract.

    Returns a dict with codes/scales of Q, K, V, dO and O, LSE (as stored: O in
    fp32 or bf16, LSE in fp32), delta, dQ, dK, dV (FP64)."""
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    do = np.asarray(do, np.float32)
    res = {}
    dec = {}
    for name, x, fmt in (("q", q, E4M3), ("k", k, E4M3), ("v", v, E4M3), ("do", do, E5M2)):
        c, s = quantize(x, fmt)
        res[name + "_codes"], res[name + "_scales"] = c, s
        dec[name] = dequantize(c, s, fmt)
    rows = _delta_tiles(q_tiles, kv_tiles, q.shape[2], causal)
    O, LSE = attn_fwd(dec["q"], dec["k"], dec["v"], causal, sigma, flags, rows, groups)
    O_st = round_bf16(O) if o_bf16 else O.astype(np.float32).astype(np.float64)
    LSE_st = LSE.astype(np.float32).astype(np.float64)
    res["O"], res["LSE"] = O_st, LSE_st
    res["O_exact"] = O
    delta = attn_delta(dec["q"], dec["k"], dec["v"], dec["do"], LSE_st, mode,
                       dO=do, O=O_st, causal=causal, sigma=sigma, flags=flags,
                       q_tiles=rows, groups=groups)
    res["delta"] = delta
    res.update(attn_bwd(dec["q"], dec["k"], dec["v"], dec["do"], LSE_st, delta, causal, sigma, flags,
                        q_tiles, kv_tiles, groups, want_diag=want_diag))
    return res


def pipeline_key_blocks(q, k, v, do, bounds, causal=True, sigma=0.0, flags=GPU_CONTRACT, o_bf16=False,
                        q_tiles=None, kv_tiles=None, groups=None):
    """The pipeline with the keys split into blocks [bounds[r], bounds[r+1])
    (context parallelism): quantise, forward per block, merge of O and LSE,
    matched delta from the blocks' partial sums (added before the division),
    backward per block with the merged LSE and delta, dQ summed over blocks.
    Returns the same keys as pipeline() plus the per-block O_parts, LSE_parts.
    q_tiles / kv_tiles / groups select outputs as in pipeline() (other rows NaN)."""
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    do = np.asarray(do, np.float32)
    res, dec = {}, {}
    for name, x, fmt in (("q", q, E4M3), ("k", k, E4M3), ("v", v, E4M3), ("do", do, E5M2)):
        c, s = quantize(x, fmt)
        res[name + "_codes"], res[name + "_scales"] = c, s
        dec[name] = dequantize(c, s, fmt)
    rows = _delta_tiles(q_tiles, kv_tiles, q.shape[2], causal)
    blocks = list(zip(bounds[:-1], bounds[1:]))
    parts = [attn_fwd(dec["q"], dec["k"], dec["v"], causal, sigma, flags, rows, groups, kv_range=b) for b in blocks]
    # each block's O as the GPU stores it (fp32), its LSE in fp32
    O_parts = np.stack([p[0].astype(np.float32).astype(np.float64) for p in parts])
    L_parts = np.stack([p[1].astype(np.float32).astype(np.float64) for p in parts])
    with np.errstate(invalid="ignore"):
        O, LSE = attn_merge(O_parts, L_parts)
    unsel = np.isnan(L_parts).any(0)      # rows the selection left out stay NaN
    O[unsel] = np.nan
    LSE[unsel] = np.nan
    O_st = round_bf16(O) if o_bf16 else O.astype(np.float32).astype(np.float64)
    LSE_st = LSE.astype(np.float32).astype(np.float64)
    num = np.zeros(LSE.shape)
    den = np.zeros(LSE.shape)
    for b in blocks:
        n_r, d_r = attn_delta(dec["q"], dec["k"], dec["v"], dec["do"], LSE_st, DELTA_MATCHED, causal=causal,
                              sigma=sigma, flags=flags, q_tiles=rows, groups=groups, kv_range=b, partial=True)
        num += n_r.astype(np.float32)
        den += d_r.astype(np.float32)
    with np.errstate(invalid="ignore", divide="ignore"):
        delta = np.where(den > 0, num / den, 0.0)
    delta[np.isnan(num)] = np.nan
    dQ = np.full(q.shape, np.nan) if q_tiles is not None or groups is not None else np.zeros(q.shape)
    dK = np.full(k.shape, np.nan)
    dV = np.full(v.shape, np.nan)
    T = (q.shape[2] + TILE - 1) // TILE
    for b in blocks:
        block_tiles = range(b[0] // TILE, (b[1] + TILE - 1) // TILE)
        kts = [t for t in block_tiles if kv_tiles is None or t in set(kv_tiles)]
        g = attn_bwd(dec["q"], dec["k"], dec["v"], dec["do"], LSE_st, delta, causal, sigma, flags, q_tiles, kts,
                     groups, kv_range=b)
        dQ = np.where(np.isnan(g["dQ"]), dQ, np.nan_to_num(dQ) + g["dQ"])
        for t in kts:
            rs = slice(t * TILE, min(b[1], t * TILE + TILE))
            dK[:, :, rs] = g["dK"][:, :, rs]
            dV[:, :, rs] = g["dV"][:, :, rs]
    res.update(O_parts=O_parts, LSE_parts=L_parts, O=O_st, LSE=LSE_st, delta=delta, dQ=dQ, dK=dK, dV=dV,
               O_exact=O)
    return res


def _delta_tiles(q_tiles, kv_tiles, N, causal):
    """Query tiles whose delta the selected dQ / dK / dV outputs depend on."""
    if q_tiles is None:
        return None
    T = (N + TILE - 1) // TILE
    need = set(int(t) for t in q_tiles)
    for kt in (kv_tiles if kv_tiles is not None else range(T)):
        need.update(range(int(kt) if causal else 0, T))
    return sorted(need)


# ------------------------------------------------------------------ prologue
ROPE_BASE = 10000.0
RMS_EPS = 1e-6


def rope_table(N: int, d: int, base: float = ROPE_BASE):
    """cos and sin of the rotary angles n * base^(-2i/d), each [N][d/2] float64."""
    lib = _load()
    if d <= 0 or d % 2 or N < 0:
        raise ValueError("rope_table: need N >= 0 and an even d > 0")
    c = np.empty((N, d // 2), dtype=np.float64)
    s = np.empty((N, d // 2), dtype=np.float64)
    lib.or_rope_table(N, d, float(base), _p(c), _p(s))
    return c, s


def qk_prologue(x, gain=None, eps: float = RMS_EPS, rope: bool = True, base: float = ROPE_BASE) -> np.ndarray:
    """rotary(RMSNorm(x) * gain) of a [B][H][N][d] tensor, in FP64 (positions n = row index)."""
    lib = _load()
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if xa.ndim != 4:
        raise ValueError("x must be [B][H][N][d]")
    B, H, N, d = xa.shape
    g = None if gain is None else np.ascontiguousarray(np.asarray(gain, dtype=np.float64).reshape(d))
    y = np.empty(xa.shape, dtype=np.float64)
    if lib.or_qk_prologue(_p(xa), B, H, N, d, _p(g), float(eps), int(bool(rope)), float(base), _p(y)) != 0:
        raise ValueError("or_qk_prologue: bad arguments")
    return y


def qk_prologue_quantized(x, gain=None, eps: float = RMS_EPS, rope: bool = True, base: float = ROPE_BASE):
    """The prologue's E4M3 tile quantisation: (codes, scales, y) with codes and
    scales = quantize(fl32(y), E4M3) and y the FP64 prologue output."""
    y = qk_prologue(x, gain, eps, rope, base)
    codes, scales = quantize(y.astype(np.float32), E4M3)
    return codes, scales, y
