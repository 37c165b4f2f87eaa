"""Host-side logic of bench.py, on CPU.

- The reference arm (the float64 oracle on the host cores) prints one JSON
  line with the contract's keys.
- Under torchrun with two gloo ranks, rank 0 alone prints it and both ranks
  exit 0.
- The replica timing helpers (barrier, max over ranks) agree across two
  gloo ranks; with one rank they are the identity.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(out: str):
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def _run(cmd, timeout=600):
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, (r.returncode, r.stdout[-2000:], r.stderr[-4000:])
    return _json_lines(r.stdout)


def test_reference_arm_line():
    lines = _run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3"])
    assert len(lines) == 1
    d = lines[0]
    for k in KEYS:
        assert k in d, k
    assert d["impl"] == "reference"
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 3)
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_warmup_is_at_least_three():
    lines = _run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"])
    assert len(lines) == 1 and lines[0]["warmup"] == 3


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    lines = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                  "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                  "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert len(lines) == 1, lines
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def _replica_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(dist)
    m = bench.max_over_ranks(dist, 1.5 + rank)
    bench.barrier(dist)
    q.put((rank, m))
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_replica_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert got == {0: 2.5, 1: 2.5}
    assert all(p.exitcode == 0 for p in procs)


def test_single_rank_helpers_are_the_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(None, 3.25) == 3.25
    bench.barrier(None)
