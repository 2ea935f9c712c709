"""Host-side logic of bench.py, on the CPU.

* the multi-rank helpers (barrier, max over ranks, whole-job throughput) with
  two gloo ranks, the layout a torchrun launch has on the GPU machine;
* parsing of the nvidia-smi clock samples, restricted to the timed region;
* the reference arm (the fp64 oracle on the host cores), which must print one
  JSON line with the contract's keys on rank 0 only.
"""
import datetime
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.dist_init(world, use_cuda=False)
    r, w, lr = bench.dist_env()
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + r, w)
    q.put((r, w, lr, t, bench.aggregate_throughput(10.0, w, t)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[0] for x in res] == [0, 1]
    for r, w, lr, t, thr in res:
        assert w == 2 and lr == r
        assert t == 2.5                      # the slowest rank's time, seen by every rank
        assert thr == pytest.approx(10.0 * 2 / 2.5)


def test_clock_summary_parsing():
    ts = "2026/12/02 19:00:0{}.000"
    csv = "\n".join([
        ts.format(1) + ", GPU-abc, 0, 1800, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        ts.format(2) + ", GPU-abc, 0, 1500, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        ts.format(3) + ", GPU-abc, 0, 1600, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active",
        ts.format(4) + ", GPU-other, 1, 300, 2070, 100.0, 0x0, Active, Not Active, Not Active, Not Active",
        ts.format(8) + ", GPU-abc, 0, 300, 2070, 100.0, 0x0, Active, Not Active, Not Active, Not Active",
    ])
    s = bench.summarize_clocks(csv, "abc")
    assert s["samples"] == 4 and "hw_slowdown" in s["reasons"]
    t0 = datetime.datetime(2026, 12, 2, 19, 0, 1).timestamp()
    t1 = datetime.datetime(2026, 12, 2, 19, 0, 5).timestamp()
    s = bench.summarize_clocks(csv, "abc", t0, t1)   # the sample at :08 is outside the region
    assert s["sm_mhz"] == 1600 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.summarize_clocks("", None) is None


def test_layer_subset_argument():
    a = bench.parse_args(["--layers", "deep,tiny"])
    assert a.layers == ("tiny", "deep")
    with pytest.raises(SystemExit):
        bench.parse_args(["--layers", "nope"])


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "1", "--reference-budget-seconds", "3"],
                         capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_nonzero_rank_is_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, env=env,
                         timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == ""
