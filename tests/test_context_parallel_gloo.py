"""The exchange logic of context-parallel attention on two CPU ranks (gloo).

fp8_attention_gb300.context_parallel splits the keys of a sequence over the
ranks of a process group (project page "Delta-Matching for reliable FP8
attention training", section 06, extends the context to 64K tokens): each rank
computes its key block's forward, partial delta sums and backward, and the
ranks exchange the blocks' O/LSE (all-gather, then the log-sum-exp merge), the
delta sums (one all-reduce) and dQ (one all-reduce).  Here the per-rank steps
are the oracle's, on CPU, so that two gloo ranks run the module's exchange
exactly as GPU ranks would run it over NCCL; the gathered results must equal
the single-process split pipeline of the oracle (and, but for O, the unsplit
one).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The per-rank steps on CPU through the oracle (FP64; stored values rounded
    as the GPU stores them: O, LSE and the delta sums in FP32)."""

    @staticmethod
    def _full(p, x):
        """The key block x ([B][Hkv][Nk][.]) placed in a whole-sequence array."""
        out = np.zeros(x.shape[:2] + (p.N,) + x.shape[3:])
        out[:, :, p.kv_offset:p.kv_offset + x.shape[2]] = x
        return out

    @staticmethod
    def _range(p):
        return (p.kv_offset, p.kv_offset + p.Nk)

    @classmethod
    def fwd(cls, p, q, k, v):
        import oracle
        O, L = oracle.attn_fwd(q, cls._full(p, k), cls._full(p, v), p.causal, 0.0, oracle.GPU_CONTRACT,
                               kv_range=cls._range(p))
        return (torch.from_numpy(O.astype(np.float32).astype(np.float64)),
                torch.from_numpy(L.astype(np.float32).astype(np.float64)))

    @staticmethod
    def merge(p, O_parts, lse_parts):
        import oracle
        O, L = oracle.attn_merge(O_parts.numpy(), lse_parts.numpy())
        return torch.from_numpy(O), torch.from_numpy(L)

    @classmethod
    def delta_partial(cls, p, q, k, v, do_hat, lse, nd):
        import oracle
        num, den = oracle.attn_delta(q, cls._full(p, k), cls._full(p, v), do_hat,
                                     lse.numpy().astype(np.float32).astype(np.float64), oracle.DELTA_MATCHED,
                                     causal=p.causal, kv_range=cls._range(p), partial=True)
        nd[0] = torch.from_numpy(num.astype(np.float32).astype(np.float64))
        nd[1] = torch.from_numpy(den.astype(np.float32).astype(np.float64))

    @staticmethod
    def delta_combine(p, nd):
        num, den = nd[0].numpy(), nd[1].numpy()
        return torch.from_numpy(np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0))

    @classmethod
    def bwd(cls, p, q, k, v, do_hat, lse, delta):
        import oracle
        g = oracle.attn_bwd(q, cls._full(p, k), cls._full(p, v), do_hat,
                            lse.numpy().astype(np.float32).astype(np.float64), delta.numpy(), p.causal, 0.0,
                            oracle.GPU_CONTRACT, kv_range=cls._range(p))
        blk = slice(p.kv_offset, p.kv_offset + p.Nk)
        return {"dQ": torch.from_numpy(g["dQ"]), "dK": torch.from_numpy(g["dK"][:, :, blk].copy()),
                "dV": torch.from_numpy(g["dV"][:, :, blk].copy())}


def _rank(rank, world, port, path, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist

    import fp8_attention_gb300 as dm
    from fp8_attention_gb300 import context_parallel as cp
    from test_context_parallel_gloo import OracleOps
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        z = np.load(path)
        bounds = z["bounds"]
        B, Hq, N, d = z["q"].shape
        Hkv = z["k"].shape[1]
        kb, ke = int(bounds[rank]), int(bounds[rank + 1])
        p = dm.AttnParams(B, Hq, Hkv, N, d, causal=bool(z["causal"]), kv_offset=kb, kv_len=ke - kb)
        # the default LibraryOps would run the same exchange on GPU tensors over NCCL
        res = cp.step(p, z["q"], z["k"][:, :, kb:ke], z["v"][:, :, kb:ke], z["do"], ops=OracleOps)
        out.put((rank, {key: t.numpy() for key, t in res.items()}))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("causal", [True, False])
def test_two_ranks_match_the_split_oracle(tmp_path, causal):
    import oracle
    from fp8_attention_gb300.inputs import custom, make_inputs
    w = custom(1, 4, 2, 300, 32, causal=causal, seed=41)
    q, k, v, do = (t.float().numpy() for t in make_inputs(w))
    bounds = [0, 128, 300]
    ref = oracle.pipeline_key_blocks(q, k, v, do, bounds, causal=causal)
    full = oracle.pipeline(q, k, v, do, causal=causal)
    dec = {n: oracle.dequantize(ref[n + "_codes"], ref[n + "_scales"], f)
           for n, f in (("q", oracle.E4M3), ("k", oracle.E4M3), ("v", oracle.E4M3), ("do", oracle.E5M2))}
    path = str(tmp_path / "inputs.npz")
    np.savez(path, bounds=np.array(bounds), causal=np.array(causal), **dec)
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, path, out)) for r in range(2)]
    for pr in procs:
        pr.start()
    got = dict(out.get(timeout=300) for _ in range(2))
    for pr in procs:
        pr.join(120)
        assert pr.exitcode == 0
    for r in range(2):      # every rank holds the whole sequence's O, LSE, delta and dQ
        for key in ("O", "LSE", "delta", "dQ"):
            want = ref[key] if key != "O" else ref["O_exact"]
            val = got[r][key].astype(np.float32).astype(np.float64) if key == "LSE" else got[r][key]  # stored fp32
            np.testing.assert_allclose(val, want, rtol=1e-12, atol=1e-14, err_msg=f"rank {r} {key}")
    dK = np.concatenate([got[0]["dK"], got[1]["dK"]], axis=2)
    dV = np.concatenate([got[0]["dV"], got[1]["dV"]], axis=2)
    np.testing.assert_allclose(dK, ref["dK"], rtol=1e-12, atol=1e-14 * np.abs(ref["dK"]).max())
    np.testing.assert_allclose(dV, ref["dV"], rtol=1e-12, atol=1e-14 * np.abs(ref["dV"]).max())
    # against the unsplit pipeline: everything but O (see the module docstring of the oracle pins)
    for key, val in (("LSE", got[0]["LSE"]), ("delta", got[0]["delta"]), ("dQ", got[0]["dQ"]), ("dK", dK),
                     ("dV", dV)):
        err = np.linalg.norm(val - full[key]) / np.linalg.norm(full[key])
        assert err < 2e-3, (key, err)
