"""The bench's multi-rank logic on CPU: gloo process groups of world size 2
(barrier, max over ranks), and the reference arm under torchrun, where rank 0
alone prints the JSON line and every rank exits 0."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.dist_init(world, "gloo")
    bench.dist_barrier(world)
    v = bench.dist_max(1.5 * (rank + 1), world)
    bench.dist_barrier(world)
    out.put((rank, v, bench.dist_info()))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.0, 3.0]
    assert [r[2] for r in res] == [(2, 0, 0), (2, 1, 1)]


def test_reference_arm_under_torchrun_rank0_only():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "1", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--budget-s", "5"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_does_not_load_the_library():
    """The reference arm times the oracle alone: the CUDA package is never
    imported and libsinkattn.so is never mapped; its `config` names the
    workload with the same keys as the native arm's line."""
    code = (
        "import io, json, os, sys, contextlib\n"
        "sys.path.insert(0, %r)\n"
        "import bench\n"
        "buf = io.StringIO()\n"
        "with contextlib.redirect_stdout(buf):\n"
        "    bench.main(['--impl', 'reference', '--config', '1', '--steps', '2', '--warmup', '3', '--budget-s', '3'])\n"
        "maps = open('/proc/self/maps').read()\n"
        "print(json.dumps({'line': json.loads(buf.getvalue().strip().splitlines()[-1]),\n"
        "                  'pkg': 'gqa_attention_sinks_head_gb300' in sys.modules,\n"
        "                  'so': 'libsinkattn.so' in maps}))\n" % ROOT)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert not d["pkg"] and not d["so"]
    assert d["line"]["impl"] == "reference"
    assert sorted(d["line"]["config"]) == ["global_batch", "parallelism", "seq_len_max", "workload"]
