"""Host-side logic of bench.py without a GPU: the max-over-ranks timing
reduction on two gloo ranks, and the CPU reference arm on a tiny sample, alone
and under a two-rank torchrun launch."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, _ = bench.dist_env()
    got = bench.max_over_ranks(10.0 + 5.0 * r, ws)
    q.put((r, got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def test_reference_arm_prints_one_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--n", "512", "--steps", "1", "--warmup", "1", "--cpu-pairs", "2"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT, check=True)
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cpu_model"] and d["cpu_baseline"]["host_cpus"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_under_torchrun_prints_from_rank_0_only():
    # the launch a multi-GPU run uses; ranks other than 0 exit 0 without work
    port = 29000 + os.getpid() % 1000
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                          "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                          "--master-port", str(port), "bench.py", "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "1", "--cpu-pairs", "2"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT, check=True)
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["config"]["parallelism"] == "dp2"


def test_method_roofline_counts_and_fractions():
    sys.path.insert(0, ROOT)
    import bench
    # b4 h32 n32768 d=e=128 bf16: 4.29 GB of tokens + 8.4 MB of final states forward,
    # 7.52 GB backward; 0.412 / 1.10 TFLOP in the 64-token chunk accounting
    w = bench.method_work(4, 32768, 32, 128, 128)
    th = 4 * 32768 * 32
    assert w["fwd_bytes"] == th * 2 * 512 + 4 * 32 * 128 * 128 * 4
    assert w["bwd_bytes"] == th * 2 * 896
    assert abs(w["fwd_flops"] / 1e12 - 0.4123) < 1e-3
    assert abs(w["bwd_flops"] / 1e12 - 1.0995) < 1e-3
    # at 1 TB/s and 1000 TFLOP/s the bytes bound both; a run at exactly the
    # roofline time has fraction 1
    r = bench.method_roofline(w, w["fwd_bytes"] / 1e9, w["bwd_bytes"] / 1e9, 1000.0, 1000.0)
    for k in ("fwd", "bwd"):
        assert r[k]["bound"] == "hbm" and abs(r[k]["frac"] - 1.0) < 1e-12
        assert abs(r[k]["gbs"] - 1000.0) < 1e-9
    # with a tiny tensor peak the FLOPs bound instead
    r = bench.method_roofline(w, 1.0, 1.0, 1e6, 1.0)
    assert r["fwd"]["bound"] == "tensor"
    assert abs(r["fwd"]["frac"] - w["fwd_flops"] / 1e12 / 1e-3) < 1e-6


def test_clock_summary_keeps_the_timed_region():
    sys.path.insert(0, ROOT)
    import datetime
    import bench
    base = datetime.datetime(2026, 1, 2, 3, 4, 5)

    def line(dt_s, sm, power_cap="Not Active", thermal="Not Active"):
        ts = (base + datetime.timedelta(seconds=dt_s)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return ", ".join([ts, str(sm), "2070", "900.0", "0x0", "Not Active", "Not Active",
                          thermal, power_cap])

    out = "\n".join([line(0.0, 2070), line(0.05, 2070), line(0.40, 1900, "Active"),
                     line(0.45, 1950), line(0.50, 1800, "Active"), line(0.90, 2070,
                                                                        thermal="Active")])
    t0 = base.timestamp() + 0.30
    t1 = base.timestamp() + 0.60
    c = bench.ClockSampler.summarize(out, t0, t1)
    assert c["samples_in_timed_region"] == 3 and c["samples"] == 3
    assert c["sm_mhz"] == 1900 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]          # the thermal flag came after the region
    # no sample inside the region: every sample is summarised, and the count says so
    c = bench.ClockSampler.summarize(out, t1 + 10, t1 + 11)
    assert c["samples_in_timed_region"] == 0 and c["samples"] == 6
    assert "sw_thermal_slowdown" in c["reasons"]
    assert bench.ClockSampler.summarize("", t0, t1) is None
    assert bench.ClockSampler.summarize("garbage\n1,2,3", t0, t1) is None
