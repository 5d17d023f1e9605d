"""Seeded synthetic inputs for the attention workloads.

This module only draws and lays out inputs; it holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle are fed from it.

Recipe (the same for every workload): a fresh ``torch.Generator`` on the CPU
seeded with ``seed``; draws in the order Q, K, V, dO, each ``randn`` in fp32
of shape [B][H][N][d] (V and dO [B][H][N][dv] where the value head dimension
differs); Q, K, V ~ N(0, 1) and dO = 1e-3 * N(0, 1).  Where the
workload asks for it, Q and K are RMS-normalised per (b, h, n) row,
``x / sqrt(mean_k x_k^2 + 1e-6) * g`` with per-channel gains g.  Storage is
bf16 (round to nearest even) except for the tiny workload, which stays fp32.

The saturation workload uses the gain profile the project page reports for a
failing run ("Delta-Matching for reliable FP8 attention training", section 02:
a key-norm gain near 5.4 on channel 7), with channels 0-2 at 3.0 and the rest
at 1.0, which makes most softmax rows nearly one-hot.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool = True
    storage: str = "bf16"          # "bf16" or "fp32"
    rms_norm: bool = True
    gains: dict = field(default_factory=dict)   # channel -> gain (others 1.0)
    seed: int = 0
    dv: int = 0                    # value head dimension (V, dO, O, dV); 0 = d

    @property
    def d_v(self) -> int:
        return self.dv if self.dv else self.d

    @property
    def units(self) -> int:
        """U = B * Hq * N^2 * d; issued causal-halved FLOPs are fwd 2U, delta 2U, bwd 5U."""
        return self.B * self.Hq * self.N * self.N * self.d

    def flops(self, causal_halved: bool = True) -> dict:
        """Issued FLOPs per pass.  Each matmul contracts or produces over d (S,
        dQ, dK) or over d_v (O, dP, dV): fwd S + O, delta S + dP, bwd S + dP +
        dV + dQ + dK, 2 B Hq N^2 x width each (halved when causal)."""
        f = 0.5 if (self.causal and causal_halved) else 1.0
        base = 2.0 * self.B * self.Hq * self.N * self.N * f
        d, dv = self.d, self.d_v
        return {"fwd": base * (d + dv), "delta": base * (d + dv), "bwd": base * (3 * d + 2 * dv)}


WORKLOADS = {
    "tiny_gqa_n256_d64": Workload("tiny_gqa_n256_d64", 1, 2, 1, 256, 64, storage="fp32", rms_norm=False),
    "gqa_b4_n2048_d128": Workload("gqa_b4_n2048_d128", 4, 16, 4, 2048, 128),
    "gqa_b1_n8192_d128": Workload("gqa_b1_n8192_d128", 1, 16, 4, 8192, 128),
    "saturation_b2_n4096_d128": Workload("saturation_b2_n4096_d128", 2, 16, 4, 4096, 128,
                                         gains={7: 5.4, 0: 3.0, 1: 3.0, 2: 3.0}),
    "long_b1_n65536_d128": Workload("long_b1_n65536_d128", 1, 16, 4, 65536, 128),
    # head dimension 256 (the width of the gqa_b1_n8192_d128 heads, Hq * d =
    # 2048, in half as many heads; the same U)
    "gqa_b1_n8192_d256": Workload("gqa_b1_n8192_d256", 1, 8, 2, 8192, 256),
    # heads shaped like multi-head latent attention: query/key dimension 192
    # (128 + 64 rotary channels), value dimension 128, one kv head per query head
    "mla_b1_n8192_d192_dv128": Workload("mla_b1_n8192_d192_dv128", 1, 16, 16, 8192, 192, dv=128),
}


def custom(B, Hq, Hkv, N, d, causal=True, storage="bf16", rms_norm=True, gains=None, seed=0,
           name="custom", dv=0) -> Workload:
    return Workload(name, B, Hq, Hkv, N, d, causal, storage, rms_norm, dict(gains or {}), seed, dv)


def _rms_norm(x: torch.Tensor, gains: dict) -> torch.Tensor:
    g = torch.ones(x.shape[-1], dtype=torch.float32)
    for ch, val in gains.items():
        if ch < x.shape[-1]:
            g[ch] = float(val)
    return x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + 1e-6) * g


def make_inputs(w: Workload):
    """Return (q, k, v, do) as CPU tensors in the workload's storage dtype."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    q = torch.randn(w.B, w.Hq, w.N, w.d, generator=gen, dtype=torch.float32)
    k = torch.randn(w.B, w.Hkv, w.N, w.d, generator=gen, dtype=torch.float32)
    v = torch.randn(w.B, w.Hkv, w.N, w.d_v, generator=gen, dtype=torch.float32)
    do = 1e-3 * torch.randn(w.B, w.Hq, w.N, w.d_v, generator=gen, dtype=torch.float32)
    if w.rms_norm:
        q = _rms_norm(q, w.gains)
        k = _rms_norm(k, w.gains)
    dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
    return tuple(t.to(dt).contiguous() for t in (q, k, v, do))


def gain_vector(w: Workload) -> torch.Tensor:
    """The workload's per-channel gains as a float32 [d] vector (1.0 where unset)."""
    g = torch.ones(w.d, dtype=torch.float32)
    for ch, val in w.gains.items():
        if ch < w.d:
            g[ch] = float(val)
    return g


def make_prologue_inputs(w: Workload):
    """Return (xq, xk, gain): the workload's Q and K draws before any
    normalisation (same generator order as make_inputs), in its storage dtype,
    and its gain vector, as inputs for the attention-input prologue."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    xq = torch.randn(w.B, w.Hq, w.N, w.d, generator=gen, dtype=torch.float32)
    xk = torch.randn(w.B, w.Hkv, w.N, w.d, generator=gen, dtype=torch.float32)
    dt = torch.bfloat16 if w.storage == "bf16" else torch.float32
    return xq.to(dt).contiguous(), xk.to(dt).contiguous(), gain_vector(w)
