"""The N > 1 path of bench.py on CPU: two ranks over gloo.

The method has no data-path exchange (sequences and decode streams are
independent), so `bench.py --gpus N` runs N replicas; what crosses ranks is
the barrier around the timed region and the maximum of the step times.
These tests run that plumbing in two real processes, and check that the
reference arm leaves all work to rank 0.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import bench
d = bench.Dist()
d.init("gloo")
x = float(os.environ["X"])
d.barrier()
m = d.max(x)
d.barrier()
d.close()
print(json.dumps({"rank": d.rank, "world": d.world, "max": m}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port, **extra):
    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    env.update({k: str(v) for k, v in extra.items()})
    return env


def test_two_ranks_barrier_and_max():
    port = _free_port()
    xs = (3.25, 7.5)
    procs = [subprocess.Popen([sys.executable, "-c", WORKER, ROOT], env=_env(r, 2, port, X=xs[r]),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["world"] == 2 for o in outs)
    # every rank times with the slowest rank's step (the max over ranks)
    assert all(o["max"] == max(xs) for o in outs)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    saved = {k: os.environ.pop(k, None) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    try:
        d = bench.Dist()
        d.init("gloo")
        assert d.world == 1 and d.pg is None
        assert d.max(2.5) == 2.5
        d.barrier()
        d.close()
    finally:
        for k, v in saved.items():
            if v is not None:
                os.environ[k] = v


def test_reference_arm_other_ranks_exit_without_work():
    """Under torchrun only rank 0 runs the oracle and prints; rank 1 exits 0
    at once and prints nothing (no process group is even formed)."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=_env(1, 2, _free_port()), capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
