"""N > 1 host logic of bench.py on the CPU: the rank helpers over gloo with two
processes, and the reference arm under torchrun with two ranks (rank 0 alone
prints its line).  The op itself has no exchange step; with N GPUs bench.py runs
N independent replicas and reports the maximum time over ranks."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["RANK"] = str(rank)
    os.environ["WORLD_SIZE"] = str(world)
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks(rank, world, backend="gloo")
    r.barrier()
    got = r.max_over_ranks(3.0 * rank + 1.0)  # per-rank "times" 1.0 and 4.0
    r.barrier()
    r.close()
    q.put((rank, got))


def test_ranks_gloo_two_processes_take_the_maximum():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 4.0), (1, 4.0)]


def test_ranks_single_process_is_local():
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks(0, 1)
    assert r.max_over_ranks(2.5) == 2.5
    r.barrier()
    r.close()


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--workload", "tiny_varlen",
           "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    # the workload keys the GPU arm reports for the same workload
    assert d["config"]["workload"] == "tiny_varlen" and d["config"]["total_tokens"] == 96
    assert d["config"]["lower_bound"] == -5.0
    assert d["config"]["state_pool"] == "float32 [8,2,128,128]"
    assert d["higher_is_better"] is True and d["unit"] == "tokens/s"
