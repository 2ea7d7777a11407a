"""The multi-process plumbing of bench.py on the CPU: two `gloo` ranks.

bench.py runs one process per GPU.  Each rank does the whole workload
(replicas: the path has no exchange step), the timed region is bracketed by
barriers, the time is the maximum over ranks, and only rank 0 prints.  These
tests run that plumbing as two local processes with the gloo backend."""
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


def _run_ranks(args, world=2, timeout=300):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable] + args, cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=timeout)
            outs.append((p.returncode, out, err))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    return outs


def test_barrier_and_max_over_ranks():
    code = ("import bench; d = bench.Dist(); d.barrier(); "
            "v = d.max(float(d.rank + 1) * 1.5); d.barrier(); "
            "print(d.world, d.rank, v); d.close()")
    outs = _run_ranks(["-c", code])
    seen = set()
    for rc, out, err in outs:
        assert rc == 0, err
        world, rank, v = out.split()
        assert int(world) == 2 and float(v) == 3.0
        seen.add(int(rank))
    assert seen == {0, 1}


def test_reference_arm_prints_on_rank_zero_only():
    outs = _run_ranks(["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "2",
                       "--warmup", "3", "--ref-budget", "2"], timeout=600)
    (rc0, out0, err0), (rc1, out1, err1) = outs
    assert rc0 == 0, err0
    assert rc1 == 0, err1
    lines = [json.loads(l) for l in out0.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and not out1.strip()
    line = lines[0]
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    # the oracle runs on all host cores (a bit-identical row split over threads)
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["cores"] == len(os.sched_getaffinity(0))
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["n_gpus"] == 2
