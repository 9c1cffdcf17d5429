"""The benchmark's multi-rank logic on CPU: two gloo ranks, max over ranks
of the timed region, whole-job weak-scaling throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        assert (r, lr, w) == (rank, rank, world)
        t = 1.5 + rank  # rank 1 is the slower one
        m = bench.max_over_ranks(t, world)
        out[rank] = m
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_weak_scaling_value():
    # 2 ranks, 10 steps of 1e12 FLOPs each, slowest rank 4 s -> 5 TFLOP/s
    assert bench.weak_scaling_value(1e12, 10, 2, 4.0) == pytest.approx(5.0)
    assert bench.max_over_ranks(3.0, 1) == 3.0


def _bench(args, env_extra=None, timeout=240):
    import json
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, bench.__file__, *args], capture_output=True, text=True,
                       env=env, timeout=timeout)
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return r.returncode, [json.loads(ln) for ln in lines], r.stderr


def test_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` outside a launcher starts two ranks itself (gloo
    here); rank 0 alone prints, and it saw both."""
    rc, lines, err = _bench(["--gpus", "2", "--launch-selftest"])
    assert rc == 0, err[-2000:]
    assert lines == [{"launch_selftest": True, "n_gpus": 2, "max_over_ranks": 2.0}]


def test_gpus_flag_must_match_the_launchers_world():
    rc, lines, err = _bench(["--gpus", "2", "--launch-selftest"],
                            {"WORLD_SIZE": "3", "RANK": "0", "LOCAL_RANK": "0"})
    assert rc != 0 and not lines
    assert "WORLD_SIZE=3 but --gpus 2" in err


def test_check_world():
    env = dict(os.environ)
    try:
        os.environ.pop("WORLD_SIZE", None)
        assert bench.check_world(1) is None
        assert bench.check_world(4) == 4
        os.environ["WORLD_SIZE"] = "4"
        assert bench.check_world(4) is None
        with pytest.raises(ValueError):
            bench.check_world(2)
    finally:
        os.environ.clear()
        os.environ.update(env)
    cmd = bench.launch_command(8, ["--gpus", "8"], 29511)
    assert cmd[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=8" in cmd and "127.0.0.1" in cmd and cmd[-2:] == ["--gpus", "8"]


def test_clock_summary_counts_only_the_timed_region():
    """The bench's clock record: samples outside the timed region (the idle
    lead-in) do not count; a power-capped sample inside it does."""
    import datetime

    def ts(sec):
        return datetime.datetime.fromtimestamp(sec).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]

    t0 = 1_800_000_000.0
    rows = [f"{ts(t0 + 0.02 * i)}, 0, 2070, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, "
            "Not Active" for i in range(10)]
    rows += [f"{ts(t0 + 0.3 + 0.02 * i)}, 0, {1950 if i > 2 else 2070}, 2070, 700.0, 0x4, "
             f"Not Active, Not Active, Not Active, {'Active' if i > 2 else 'Not Active'}"
             for i in range(7)]
    s = bench.ClockSampler.summarise(rows, t0 + 0.29, t0 + 0.45)
    assert s["samples"] == 7 and s["samples_total"] == 17 and s["window"] == "timed region"
    assert s["reasons"] == ["sw_power_cap"] and s["sm_mhz"] == 1950.0
    assert s["power_w_max"] == 700.0
    whole = bench.ClockSampler.summarise(rows)
    assert whole["samples"] == 17 and whole["sm_mhz"] == 2070.0
    none_inside = bench.ClockSampler.summarise(rows, t0 + 5.0, t0 + 6.0)
    assert none_inside["samples"] == 17 and none_inside["window"].startswith("whole run")
