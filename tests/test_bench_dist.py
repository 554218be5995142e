"""Multi-rank harness of bench.py on CPU: two gloo ranks on 127.0.0.1.

Checks that the timed region is bracketed by barriers and reports the
maximum over ranks, that sums / maxima reduce across ranks, and that the
reference arm prints from rank 0 only.
"""

import json
import os
import socket
import subprocess
import sys
import time

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench

    dist_mod = bench.init_dist("gloo")
    naps = {0: 0.001, 1: 0.02}

    def step(i):
        time.sleep(naps[rank])

    ms = bench.timed_steps(step, 5, 1, dist_mod)
    mx = bench.max_over_ranks(float(rank + 1), dist_mod)
    sm = bench.sum_over_ranks(float(rank + 1), dist_mod)
    q.put((rank, ms, mx, sm))
    dist_mod.destroy_process_group()


def test_timed_steps_takes_the_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    ms0, ms1 = res[0][1], res[1][1]
    assert ms0 == ms1 >= 5 * 20.0  # both ranks report the slower rank's time
    assert all(r[2] == 2.0 and r[3] == 3.0 for r in res)


@pytest.mark.timeout(600)
def test_reference_arm_prints_on_rank0_only():
    port = _free_port()
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2")
    outs = []
    procs = []
    for r in range(2):
        e = dict(env, RANK=str(r), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
                                       "reference", "--steps", "2", "--warmup", "1"],
                                      env=e, stdout=subprocess.PIPE, text=True, cwd=ROOT))
    for p in procs:
        out, _ = p.communicate(timeout=600)
        assert p.returncode == 0
        outs.append(out.strip())
    assert outs[1] == ""
    line = json.loads(outs[0].splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
