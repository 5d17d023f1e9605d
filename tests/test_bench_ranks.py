"""The multi-process side of bench.py on CPU with the gloo backend (two
ranks): the job time is the slowest rank's, and under a launcher only rank 0
of the reference arm runs and prints."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        import bench
        out.put((rank, bench.max_over_ranks(1.5 + rank, dist, "cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(out.get(timeout=10) for _ in range(2))
    assert got == {0: 2.5, 1: 2.5}


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_under_two_ranks(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_gqa_n256_d64",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    if rank == 0:
        assert len(lines) == 1
        line = json.loads(lines[0])
        assert line["impl"] == "reference" and line["n_gpus"] == 2
        assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True and line["value"] > 0
        assert line["config"]["workload"] == "tiny_gqa_n256_d64" and line["warmup"] == 0 and line["steps"] == 1
        cb = line["cpu_baseline"]
        assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
        assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                               "d2h_bytes_per_step": 0}
    else:
        assert lines == []
