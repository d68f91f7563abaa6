"""The multi-GPU path is replicas only: each rank runs the whole layer on its own
batch, and the ranks exchange nothing but the timing.  These CPU tests run that
host logic as world-size-2 gloo process groups: the MAX reduction of the timed
regions and the whole-job rate, and the reference arm under torch.distributed.run
(rank 0 alone measures and prints; the other rank exits 0 without work)."""
import importlib.util
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def _bench():
    spec = importlib.util.spec_from_file_location("k3moe_bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rank(rank, ws, port, local_ms, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    b = _bench()
    slowest = b.slowest_rank_ms(local_ms[rank], ws, "cpu")
    q.put((rank, slowest, b.whole_job_rate(1000, slowest, ws)))
    dist.barrier()
    dist.destroy_process_group()


def test_timing_reduces_to_the_slowest_rank():
    ws, port = 2, _free_port()
    local_ms = [12.5, 40.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, local_ms, q)) for r in range(ws)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate in got:
        assert slowest == 40.0
        assert rate == 2 * 1000 / 0.040  # every rank's units over the slowest rank's time


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.slowest_rank_ms(7.0, 1, "cpu") == 7.0
    assert b.whole_job_rate(10, 5.0, 1) == 2000.0


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["steps"] == 2 and rec["value"] > 0
