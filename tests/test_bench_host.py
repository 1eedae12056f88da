"""Host-side logic of bench.py, without a GPU: the max-over-ranks timing
reduction on a world-size-2 gloo group, and the oracle reference arm's
launch contract (rank 0 prints one JSON line, other ranks exit quietly)."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    got = bench.max_over_ranks(1.5 + rank, dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, got))


def test_max_over_ranks_gloo_world2():
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 2.5, 1: 2.5}


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25


def _bench(args, env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True,
                          text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_arm_other_ranks_exit_quietly():
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "0"], {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.slow
def test_reference_arm_prints_one_json_line():
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "0"], {"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_beta_sweep_mean_and_standard_error():
    import numpy as np
    from precision_flash_attention_attn_gb300.beta_sweep import _mean_se
    m, se = _mean_se(np.array([1.0, 2.0, 3.0, 6.0]))
    assert m == 3.0 and abs(se - np.std([1.0, 2.0, 3.0, 6.0], ddof=1) / 2.0) < 1e-15
    assert _mean_se(np.array([])) == (None, None)
    assert _mean_se(np.array([4.0])) == (4.0, None)


def test_recorded_traffic_only_for_its_workload():
    # the committed DRAM figures belong to one workload; another workload's
    # roofline must not borrow them
    sys.path.insert(0, ROOT)
    import bench
    assert bench.recorded_traffic("bwd_main", "long") is None
    assert bench.recorded_traffic("fwd", "ties") is None
    assert bench.recorded_traffic("no_such_kernel") is None
