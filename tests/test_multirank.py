"""The N > 1 path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The library runs one process per GPU with no exchange inside the matmul
(replicas only), so what the ranks share is the timing: every time is the
maximum over ranks, and the job's rate is the replicas' sum at that time.
The reference arm runs on rank 0 alone; the other ranks exit without work."""
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (r + 1) ms on the first call and (10 - r) ms on the second
        times = bench.max_over_ranks([rank + 1.0, 10.0 - rank, 0.25 * rank], world, "cpu")
        rate = bench.replicas_rate(100.0, world)
        dist.barrier()
        queue.put((rank, times, rate))
    finally:
        dist.destroy_process_group()


def test_timing_is_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, _, _ in results) == [0, 1]
    for _, times, rate in results:
        assert times == [2.0, 10.0, 0.25]
        assert rate == 200.0


def _reference_arm(rank, world):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
               MASTER_ADDR="127.0.0.1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus",
                           str(world), "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                          env=env, timeout=300)


def test_reference_arm_runs_on_rank_zero_only():
    import json
    other = _reference_arm(1, 2)
    assert other.returncode == 0 and other.stdout.strip() == ""
    zero = _reference_arm(0, 2)
    assert zero.returncode == 0, zero.stderr[-2000:]
    lines = [l for l in zero.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
