"""Python binding of libdm: FP8 flash attention with the Delta-Matching correction on GB300.

Thin ctypes marshalling over the C ABI in ``include/dm.h`` (same function
names).  PyTorch only provides device memory and streams; every step of the
computation runs in the library's sm_103a kernels.  Importing works without
a GPU, but the first call raises if ``libdm.so`` has not been built
(``python -c "import __graft_entry__ as g; g.build()"``) -- there is no CPU
fallback.

FP8 tensors are passed as ``Fp8(codes, scales)``: codes uint8 [B][H][N][d] and
scales float32 [B][H][ceil(N/128)], both contiguous CUDA tensors.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from dataclasses import dataclass
from typing import NamedTuple, Optional

import torch

__all__ = [
    "AttnParams", "Fp8", "DMError", "lib", "dm_version", "dm_status_string", "dm_set_knob",
    "dm_get_status", "dm_last_timeout_site", "dm_quantize", "dm_quantize_batch", "dm_rope_table",
    "dm_qk_prologue_batch", "ROPE_BASE", "RMS_EPS", "DM_PROLOGUE_MAX_JOBS", "dm_attn_fwd", "dm_attn_delta", "dm_attn_bwd",
    "dm_attn_bwd_workspace_size", "dm_attn_bwd_noalloc", "DM_NOALLOC_MAX_DELTA_ROWS",
    "dm_attn_delta_partial", "dm_attn_merge", "dm_attn_delta_combine",
    "DM_F32", "DM_BF16", "DM_E4M3", "DM_E5M2", "DM_DELTA_MATCHED", "DM_DELTA_STALE_DO",
    "DM_DELTA_STALE_DOHAT", "DM_KNOB_WAIT_LIMIT_NS", "DM_KNOB_STALL_TEST",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdm.so")

DM_OK, DM_ERR_INVALID_ARG, DM_ERR_SHAPE, DM_ERR_DTYPE, DM_ERR_ALIGNMENT = 0, 1, 2, 3, 4
DM_ERR_UNSUPPORTED, DM_ERR_CUDA, DM_ERR_TIMEOUT = 5, 6, 7
DM_F32, DM_BF16 = 0, 1
DM_E4M3, DM_E5M2 = 0, 1
DM_DELTA_MATCHED, DM_DELTA_STALE_DO, DM_DELTA_STALE_DOHAT = 0, 1, 2
DM_KNOB_WAIT_LIMIT_NS, DM_KNOB_STALL_TEST = 0, 1
TILE = 128
DM_NOALLOC_MAX_DELTA_ROWS = 1 << 21


class DMError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {dm_status_string(code)}")


class _Params(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("N", ctypes.c_int),
                ("d", ctypes.c_int), ("causal", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("d_v", ctypes.c_int), ("kv_offset", ctypes.c_int), ("kv_len", ctypes.c_int)]


class _Fp8(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


class _Diag(ctypes.Structure):
    _fields_ = [("rowsum_pre", ctypes.c_void_p), ("abssum_pre", ctypes.c_void_p),
                ("rowsum_post", ctypes.c_void_p), ("abssum_post", ctypes.c_void_p)]


@dataclass(frozen=True)
class AttnParams:
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool = True
    softmax_scale: float = 0.0   # <= 0 selects 1/sqrt(d)
    d_v: int = 0                 # head dimension of V, dO, O, dV; 0 selects d
    kv_offset: int = 0           # key block: keys at [kv_offset, kv_offset + kv_len) only
    kv_len: int = 0              # (both 0: the whole sequence; kv_len 0: up to N)

    def c(self) -> _Params:
        return _Params(self.B, self.Hq, self.Hkv, self.N, self.d, int(bool(self.causal)),
                       float(self.softmax_scale), int(self.d_v), int(self.kv_offset), int(self.kv_len))

    @property
    def dv(self) -> int:
        return self.d_v if self.d_v else self.d

    @property
    def Nk(self) -> int:
        """Rows of K, V, dK and dV (the key block's, else N)."""
        return self.kv_len if self.kv_len > 0 else self.N - self.kv_offset

    @property
    def T(self) -> int:
        return (self.N + TILE - 1) // TILE


class Fp8(NamedTuple):
    codes: torch.Tensor
    scales: torch.Tensor


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded libdm.so; raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -c \"import __graft_entry__ as g; g.build()\"`")
            L = ctypes.CDLL(LIB_PATH)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            PP = ctypes.POINTER(_Params)
            L.dm_version.restype = I
            L.dm_status_string.restype = ctypes.c_char_p
            L.dm_status_string.argtypes = [I]
            L.dm_set_knob.restype = I
            L.dm_set_knob.argtypes = [I, ctypes.c_longlong]
            L.dm_get_status.restype = I
            L.dm_get_status.argtypes = [P]
            L.dm_last_timeout_site.restype = ctypes.c_uint
            L.dm_quantize.restype = I
            L.dm_quantize.argtypes = [P, I, I, I, I, I, I, P, P, P, P]
            L.dm_quantize_batch.restype = I
            L.dm_quantize_batch.argtypes = [P, I, I, P]
            L.dm_rope_table.restype = I
            L.dm_rope_table.argtypes = [I, I, ctypes.c_double, P, P, P]
            L.dm_qk_prologue_batch.restype = I
            L.dm_qk_prologue_batch.argtypes = [P, I, I, ctypes.c_float, P]
            L.dm_attn_fwd.restype = I
            L.dm_attn_fwd.argtypes = [PP, _Fp8, _Fp8, _Fp8, P, I, P, P]
            L.dm_attn_delta.restype = I
            L.dm_attn_delta.argtypes = [PP, I, _Fp8, _Fp8, _Fp8, _Fp8, P, P, I, P, I, P, P]
            L.dm_attn_bwd.restype = I
            L.dm_attn_bwd.argtypes = [PP, I, _Fp8, _Fp8, _Fp8, _Fp8, P, P, P, I, P, I, P, P, P,
                                      ctypes.POINTER(_Diag), P, S, P]
            L.dm_attn_bwd_noalloc.restype = I
            L.dm_attn_bwd_noalloc.argtypes = [PP, I, _Fp8, _Fp8, _Fp8, _Fp8, P, P, I, P, I, P, P, P,
                                              ctypes.POINTER(_Diag), P]
            L.dm_attn_bwd_workspace_size.restype = S
            L.dm_attn_bwd_workspace_size.argtypes = [PP]
            L.dm_attn_delta_partial.restype = I
            L.dm_attn_delta_partial.argtypes = [PP, _Fp8, _Fp8, _Fp8, _Fp8, P, P, P, P]
            L.dm_attn_merge.restype = I
            L.dm_attn_merge.argtypes = [PP, I, P, P, P, I, P, P]
            L.dm_attn_delta_combine.restype = I
            L.dm_attn_delta_combine.argtypes = [PP, I, P, P, P, P]
            _lib = L
    return _lib


# ---------------------------------------------------------------- marshalling
def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdm must be contiguous")
    return t.data_ptr() or None


def _dtype(t: Optional[torch.Tensor]) -> int:
    if t is None:
        return DM_F32
    return {torch.float32: DM_F32, torch.bfloat16: DM_BF16}.get(t.dtype, -1)


def _fp8(x: Optional[Fp8]) -> _Fp8:
    if x is None:
        return _Fp8(None, None)
    return _Fp8(_ptr(x.codes), _ptr(x.scales))


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _on(dev):
    """Makes `dev` the current CUDA device around a library call: the library
    keeps per-device state (the status word, the no-allocation array) and looks
    it up on the current device, so tensors on another GPU must switch to it."""
    dev = torch.device(dev)
    if dev.type != "cuda":
        return contextlib.nullcontext()
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    if idx == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(idx)


def _check(rc: int, where: str):
    if rc != DM_OK:
        raise DMError(rc, where)


def dm_version() -> int:
    return lib().dm_version()


def dm_status_string(code: int) -> str:
    return lib().dm_status_string(int(code)).decode()


def dm_set_knob(knob: int, value: int) -> None:
    _check(lib().dm_set_knob(int(knob), int(value)), "dm_set_knob")


def dm_get_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return lib().dm_get_status(_stream(stream))


def dm_last_timeout_site() -> int:
    """kernel * 100 + wait number of the last expired wait reported by dm_get_status (0: none)."""
    return int(lib().dm_last_timeout_site())


def dm_quantize(x: torch.Tensor, fmt: int, codes=None, scales=None, codes_t=None, want_transposed=False,
                stream=None):
    """Per 128-row x d tile FP8 quantisation of x [B][H][N][d] (fp32 or bf16) -> Fp8 (+ codes^T)."""
    B, H, N, d = x.shape
    T = (N + TILE - 1) // TILE
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((B, H, T), dtype=torch.float32, device=x.device)
    if want_transposed and codes_t is None:
        codes_t = torch.empty((B, H, d, N), dtype=torch.uint8, device=x.device)
    with _on(x.device):
        rc = lib().dm_quantize(_ptr(x), _dtype(x), B, H, N, d, int(fmt), _ptr(codes), _ptr(scales),
                               _ptr(codes_t), _stream(stream))
    _check(rc, "dm_quantize")
    out = Fp8(codes, scales)
    return (out, codes_t) if codes_t is not None else out


class _QuantJob(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("d", ctypes.c_int), ("fmt", ctypes.c_int), ("codes", ctypes.c_void_p),
                ("scales", ctypes.c_void_p), ("codes_t", ctypes.c_void_p)]


def dm_quantize_batch(tensors, stream=None):
    """dm_quantize of several tensors in one launch: tensors is a sequence of (x, fmt) with x [B][H][N][d]
    (all of one dtype and one d); returns one Fp8 per tensor."""
    jobs, outs = [], []
    for x, fmt in tensors:
        B, H, N, d = x.shape
        T = (N + TILE - 1) // TILE
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        scales = torch.empty((B, H, T), dtype=torch.float32, device=x.device)
        jobs.append(_QuantJob(_ptr(x), B, H, N, d, int(fmt), _ptr(codes), _ptr(scales), None))
        outs.append(Fp8(codes, scales))
    if not jobs:
        return []
    dtype = _dtype(tensors[0][0])
    if any(_dtype(x) != dtype for x, _ in tensors):
        raise DMError(DM_ERR_DTYPE, "dm_quantize_batch: tensors of different dtypes")
    arr = (_QuantJob * len(jobs))(*jobs)
    with _on(tensors[0][0].device):
        rc = lib().dm_quantize_batch(arr, len(jobs), dtype, _stream(stream))
    _check(rc, "dm_quantize_batch")
    return outs


ROPE_BASE = 10000.0
RMS_EPS = 1e-6
DM_PROLOGUE_MAX_JOBS = 4


def dm_rope_table(N: int, d: int, base: float = ROPE_BASE, device="cuda", stream=None):
    """cos and sin of the rotary angles n * base^(-2i/d): two float32 tensors [N][d/2] on the device."""
    cos = torch.empty((N, d // 2), dtype=torch.float32, device=device)
    sin = torch.empty((N, d // 2), dtype=torch.float32, device=device)
    with _on(cos.device):
        rc = lib().dm_rope_table(int(N), int(d), float(base), _ptr(cos), _ptr(sin), _stream(stream))
    _check(rc, "dm_rope_table")
    return cos, sin


class _PrologueJob(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("d", ctypes.c_int), ("gain", ctypes.c_void_p), ("rope_cos", ctypes.c_void_p),
                ("rope_sin", ctypes.c_void_p), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


def dm_qk_prologue_batch(tensors, rope=None, eps: float = RMS_EPS, stream=None):
    """RMSNorm with channel gains, rotary embedding and E4M3 tile quantisation of
    several [B][H][N][d] tensors in one launch.  tensors: sequence of (x, gain)
    with gain a float32 [d] device tensor or None; rope: (cos, sin) from
    dm_rope_table (covering every position) or None.  Returns one Fp8 each."""
    jobs, outs = [], []
    cos, sin = rope if rope is not None else (None, None)
    for x, gain in tensors:
        B, H, N, d = x.shape
        T = (N + TILE - 1) // TILE
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
        scales = torch.empty((B, H, T), dtype=torch.float32, device=x.device)
        jobs.append(_PrologueJob(_ptr(x), B, H, N, d, _ptr(gain), _ptr(cos), _ptr(sin), _ptr(codes),
                                 _ptr(scales)))
        outs.append(Fp8(codes, scales))
    if not jobs:
        return []
    dtype = _dtype(tensors[0][0])
    if any(_dtype(x) != dtype for x, _ in tensors):
        raise DMError(DM_ERR_DTYPE, "dm_qk_prologue_batch: tensors of different dtypes")
    arr = (_PrologueJob * len(jobs))(*jobs)
    with _on(tensors[0][0].device):
        rc = lib().dm_qk_prologue_batch(arr, len(jobs), dtype, float(eps), _stream(stream))
    _check(rc, "dm_qk_prologue_batch")
    return outs


def dm_attn_fwd(p: AttnParams, q: Fp8, k: Fp8, v: Fp8, O=None, o_dtype=torch.float32, lse=None, stream=None):
    """Forward: returns (O [B][Hq][N][d_v], LSE [B][Hq][N])."""
    dev = q.codes.device
    if O is None:
        O = torch.empty((p.B, p.Hq, p.N, p.dv), dtype=o_dtype, device=dev)
    if lse is None:
        lse = torch.empty((p.B, p.Hq, p.N), dtype=torch.float32, device=dev)
    cp = p.c()
    with _on(dev):
        rc = lib().dm_attn_fwd(ctypes.byref(cp), _fp8(q), _fp8(k), _fp8(v), _ptr(O), _dtype(O), _ptr(lse),
                               _stream(stream))
    _check(rc, "dm_attn_fwd")
    return O, lse


def dm_attn_delta(p: AttnParams, mode: int, q: Fp8, k: Fp8, v: Fp8, do_hat: Fp8, lse, dO=None, O=None,
                  delta=None, stream=None):
    """Softmax row correction delta [B][Hq][N] for the given mode."""
    ref = lse if lse is not None else O
    if delta is None:
        delta = torch.empty((p.B, p.Hq, p.N), dtype=torch.float32, device=ref.device)
    cp = p.c()
    with _on(delta.device):
        rc = lib().dm_attn_delta(ctypes.byref(cp), int(mode), _fp8(q), _fp8(k), _fp8(v), _fp8(do_hat),
                                 _ptr(lse), _ptr(dO), _dtype(dO), _ptr(O), _dtype(O), _ptr(delta),
                                 _stream(stream))
    _check(rc, "dm_attn_delta")
    return delta


def dm_attn_bwd_workspace_size(p: AttnParams) -> int:
    cp = p.c()
    return int(lib().dm_attn_bwd_workspace_size(ctypes.byref(cp)))


def _diag(p: AttnParams, diag, dev, out: dict):
    """The dm_diag struct for `diag` (False: none; True: four new row-sum
    buffers; a dict: the caller's buffers by name), recording them in `out`."""
    if not diag:
        return None
    names = ("rowsum_pre", "abssum_pre", "rowsum_post", "abssum_post")
    if isinstance(diag, dict):
        bufs = {n: diag.get(n) for n in names}
    else:
        bufs = {n: torch.empty((p.B, p.Hq, p.N), dtype=torch.float32, device=dev) for n in names}
    out.update({n: t for n, t in bufs.items() if t is not None})
    return _Diag(*[_ptr(bufs[n]) for n in names])


def dm_attn_bwd(p: AttnParams, mode: int, q: Fp8, k: Fp8, v: Fp8, do_hat: Fp8, lse, delta=None, dO=None,
                O=None, dQ=None, dK=None, dV=None, diag=False, workspace=None, stream=None):
    """Backward: returns dict with dQ, dK, dV (and the four diagnostic row sums if diag)."""
    dev = lse.device
    if dQ is None:
        dQ = torch.empty((p.B, p.Hq, p.N, p.d), dtype=torch.float32, device=dev)
    if dK is None:
        dK = torch.empty((p.B, p.Hkv, p.Nk, p.d), dtype=torch.float32, device=dev)
    if dV is None:
        dV = torch.empty((p.B, p.Hkv, p.Nk, p.dv), dtype=torch.float32, device=dev)
    out = {"dQ": dQ, "dK": dK, "dV": dV}
    cdiag = _diag(p, diag, dev, out)
    ws_bytes = 0
    own_ws = delta is None and workspace is None
    if delta is None:
        ws_bytes = dm_attn_bwd_workspace_size(p)
        if workspace is None:
            workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        ws_bytes = workspace.numel() * workspace.element_size()
    cp = p.c()
    with _on(dev):
        rc = lib().dm_attn_bwd(ctypes.byref(cp), int(mode), _fp8(q), _fp8(k), _fp8(v), _fp8(do_hat), _ptr(lse),
                               _ptr(delta), _ptr(dO), _dtype(dO), _ptr(O), _dtype(O), _ptr(dQ), _ptr(dK),
                               _ptr(dV), ctypes.byref(cdiag) if cdiag is not None else None, _ptr(workspace),
                               ws_bytes, _stream(stream))
    _check(rc, "dm_attn_bwd")
    if own_ws and stream is not None:
        # the workspace was allocated on the current stream but is used on
        # `stream`: keep the allocator from handing it out again before the
        # work queued there has finished
        s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(int(stream), device=dev)
        workspace.record_stream(s)
    return out


def dm_attn_bwd_noalloc(p: AttnParams, mode: int, q: Fp8, k: Fp8, v: Fp8, do_hat: Fp8, lse, dO=None, O=None,
                        dQ=None, dK=None, dV=None, diag=False, stream=None):
    """Backward with delta computed for `mode` in the library's fixed device array (no
    workspace, no allocation inside the call; the outputs and diagnostic buffers here are
    allocated by torch only when the caller passes none)."""
    dev = lse.device
    if dQ is None:
        dQ = torch.empty((p.B, p.Hq, p.N, p.d), dtype=torch.float32, device=dev)
    if dK is None:
        dK = torch.empty((p.B, p.Hkv, p.N, p.d), dtype=torch.float32, device=dev)
    if dV is None:
        dV = torch.empty((p.B, p.Hkv, p.N, p.dv), dtype=torch.float32, device=dev)
    out = {"dQ": dQ, "dK": dK, "dV": dV}
    cdiag = _diag(p, diag, dev, out)
    cp = p.c()
    with _on(dev):
        rc = lib().dm_attn_bwd_noalloc(ctypes.byref(cp), int(mode), _fp8(q), _fp8(k), _fp8(v), _fp8(do_hat),
                                       _ptr(lse), _ptr(dO), _dtype(dO), _ptr(O), _dtype(O), _ptr(dQ), _ptr(dK),
                                       _ptr(dV), ctypes.byref(cdiag) if cdiag is not None else None,
                                       _stream(stream))
    _check(rc, "dm_attn_bwd_noalloc")
    return out


def dm_attn_delta_partial(p: AttnParams, q: Fp8, k: Fp8, v: Fp8, do_hat: Fp8, lse, num=None, den=None,
                          stream=None):
    """The matched correction's two sums over the key block of p: returns
    (num, den), each float32 [B][Hq][N] (sum_j P dP^ and sum_j P over the block)."""
    dev = lse.device
    if num is None:
        num = torch.empty((p.B, p.Hq, p.N), dtype=torch.float32, device=dev)
    if den is None:
        den = torch.empty((p.B, p.Hq, p.N), dtype=torch.float32, device=dev)
    cp = p.c()
    with _on(dev):
        rc = lib().dm_attn_delta_partial(ctypes.byref(cp), _fp8(q), _fp8(k), _fp8(v), _fp8(do_hat), _ptr(lse),
                                         _ptr(num), _ptr(den), _stream(stream))
    _check(rc, "dm_attn_delta_partial")
    return num, den


def dm_attn_merge(p: AttnParams, O_parts, lse_parts, O=None, o_dtype=torch.float32, lse=None, stream=None):
    """(O, LSE) of the union of key blocks from their stacked results:
    O_parts float32 [S][B][Hq][N][d_v], lse_parts float32 [S][B][Hq][N]."""
    dev = lse_parts.device
    if O is None:
        O = torch.empty((p.B, p.Hq, p.N, p.dv), dtype=o_dtype, device=dev)
    if lse is None:
        lse = torch.empty((p.B, p.Hq, p.N), dtype=torch.float32, device=dev)
    cp = p.c()
    with _on(dev):
        rc = lib().dm_attn_merge(ctypes.byref(cp), int(lse_parts.shape[0]), _ptr(O_parts), _ptr(lse_parts),
                                 _ptr(O), _dtype(O), _ptr(lse), _stream(stream))
    _check(rc, "dm_attn_merge")
    return O, lse


def dm_attn_delta_combine(p: AttnParams, num_parts, den_parts, delta=None, stream=None):
    """delta = sum of the stacked num parts / sum of the den parts ([S][B][Hq][N] each)."""
    dev = num_parts.device
    if delta is None:
        delta = torch.empty((p.B, p.Hq, p.N), dtype=torch.float32, device=dev)
    cp = p.c()
    with _on(dev):
        rc = lib().dm_attn_delta_combine(ctypes.byref(cp), int(num_parts.shape[0]), _ptr(num_parts),
                                         _ptr(den_parts), _ptr(delta), _stream(stream))
    _check(rc, "dm_attn_delta_combine")
    return delta
