"""Benchmark: forward + backward of decayed causal linear attention on the
Lightning-2 benchmark shape (batch 4, 32 heads, d = e = 128, bf16, ALiBi-style
decay slopes, scale 1) at n = 32768 tokens per sequence.

One step = la_fwd (o, final_state) + la_bwd (dq, dk, dv) over one batch.
`value` is whole-job tokens/s (B*n per step per rank) with inputs resident in
HBM (each 1.07 GB tensor is larger than the 129 MB L2, so no flush is
needed); `e2e` is the same metric through the public Python API with pinned
host buffers copied in and results copied out inside the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--n 32768] [--impl reference]

`--impl reference` times the fp64 CPU oracle (the reference arm: there is no
runnable reference implementation) on the host cores, on a bounded sample of
the same workload.  Under torchrun (N > 1) every rank runs its own batch
(weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fwd+bwd tokens/s & % roofline at b4 h32 d=e=128 bf16, n=512..32768"
# Lightning-Attention-2 README, Benchmark tables (hardware unstated): fwd 17.661427 ms and
# bwd 74.594788 ms at n = 32768 -> 4*32768 / 92.256215 ms.
PAGES_TOKENS_PER_S = {512: 4 * 512 / ((0.351540 + 1.169621) * 1e-3),
                      1024: 4 * 1024 / ((0.585876 + 2.334296) * 1e-3),
                      2048: 4 * 2048 / ((1.134238 + 4.657026) * 1e-3),
                      4096: 4 * 4096 / ((2.240815 + 9.307817) * 1e-3),
                      8192: 4 * 8192 / ((4.414397 + 18.617611) * 1e-3),
                      16384: 4 * 16384 / ((8.832678 + 37.212578) * 1e-3),
                      32768: 4 * 32768 / ((17.661427 + 74.594788) * 1e-3)}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def bench_config(B, H, n, d, e, ws):
    """The `config` object of the bench line, shared by both arms."""
    unit = B * n * H * d * 2
    l2 = ("inputs larger than L2 (%.2f GB per token tensor), no flush" % (unit / 1e9)
          if unit > 2 * 129e6 else "inputs within twice the L2 (%.3f GB per token tensor)"
          % (unit / 1e9))
    return {"workload": "fwd+bwd b%d h%d n%d d=e=%d bf16, ALiBi slopes, scale 1" % (B, H, n, d),
            "B": B, "H": H, "n": n, "d": d, "e": e, "l2": l2, "parallelism": "dp%d" % ws}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, world_size, device=None):
    """Max of a float over ranks (identity when world_size == 1)."""
    if world_size == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor peak in TFLOP/s: the measured burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


# The method's own roofline.  Per (token, head) of B*T*H token-heads:
#   bytes   fwd 2(2d + 2e) (q, k, v read, o written, bf16) + the fp32 final states;
#           bwd 2(4d + 3e) (q, k, v, do read; dq, dk, dv written)
#   FLOPs   chunked accounting with 64-token chunks and full 64 x 64 tiles:
#           fwd 2C(d + e) + 4de, bwd 6C(d + e) + 10de
# Roofline time = max(FLOPs / tensor peak, bytes / HBM peak); the fraction is
# roofline time / measured time.  (The kernels run 128-token chunks, so they
# execute more than these FLOPs; the count is the fixed convention.)
ACCOUNT_CHUNK = 64
NOMINAL_HBM_GBS = 8000.0
NOMINAL_BF16_TFLOPS = 2250.0


def method_work(B, T, H, d, e, token_bytes=2):
    th = B * T * H
    C = ACCOUNT_CHUNK
    return {"fwd_bytes": th * token_bytes * (2 * d + 2 * e) + B * H * d * e * 4,
            "bwd_bytes": th * token_bytes * (4 * d + 3 * e),
            "fwd_flops": th * (2 * C * (d + e) + 4 * d * e),
            "bwd_flops": th * (6 * C * (d + e) + 10 * d * e)}


def method_roofline(work, fwd_ms, bwd_ms, hbm_gbs, tflops):
    """TFLOP/s, GB/s and the roofline fraction of the forward and the backward."""
    out = {}
    for name, ms in (("fwd", fwd_ms), ("bwd", bwd_ms)):
        t_mem = work[name + "_bytes"] / (hbm_gbs * 1e9)
        t_math = work[name + "_flops"] / (tflops * 1e12)
        roof = max(t_mem, t_math)
        out[name] = {"tflops": work[name + "_flops"] / (ms * 1e-3) / 1e12,
                     "gbs": work[name + "_bytes"] / (ms * 1e-3) / 1e9,
                     "roofline_ms": roof * 1e3,
                     "bound": "hbm" if t_mem >= t_math else "tensor",
                     "frac": roof / (ms * 1e-3)}
    return out


class ClockSampler:
    """nvidia-smi clock / throttle sampling around the timed region.  Each sample
    carries nvidia-smi's timestamp; the summary uses the samples that fall inside
    the timed region (wall clock) and falls back to all of them when none does."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, t0=None, t1=None):
        """t0, t1: the timed region in time.time() seconds."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarize(out, t0, t1)

    @staticmethod
    def _stamp(text):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text, fmt).timestamp()
            except ValueError:
                pass
        return None

    @classmethod
    def summarize(cls, out, t0=None, t1=None):
        rows = []
        for line in (out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            flags = {name for name, flag in zip(cls.REASONS, parts[5:9])
                     if flag.lower().startswith("active")}
            rows.append((cls._stamp(parts[0]), sm, mx, flags))
        if not rows:
            return None
        inside = [r for r in rows
                  if t0 is not None and r[0] is not None and t0 <= r[0] <= t1]
        use = inside or rows
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(set().union(*(r[3] for r in use))),
                "samples": len(use), "samples_in_timed_region": len(inside)}


def gpu_bench(args):
    import torch
    import linear_attention_head_gb300 as la
    from linear_attention_head_gb300 import _native
    import workloads as W

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = W.sweep_bf16(args.n)
    B, T, H, D, E = w.B, w.T, w.H, w.d, w.e
    gen = torch.Generator(device=dev).manual_seed(1234 + rank)
    q = torch.randn((B, T, H, D), generator=gen, device=dev).to(torch.bfloat16)
    k = torch.randn((B, T, H, D), generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn((B, T, H, E), generator=gen, device=dev).to(torch.bfloat16)
    do = torch.randn((B, T, H, E), generator=gen, device=dev).to(torch.bfloat16)
    g = w.g_gamma.to(dev)
    scale = w.scale
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        o, fin = la.la_fwd(q, k, v, g, scale)
        if ev is not None:
            ev[1].record(stream)
        dq = la.la_bwd_dq(q, k, v, do, g, scale)
        if ev is not None:
            ev[2].record(stream)
        dk, dv, _ = la.la_bwd_dkdv(q, k, v, do, g, scale, want_d_initial_state=False)
        if ev is not None:
            ev[3].record(stream)
        return o, dq, dk, dv

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    la.get_device_error(dev)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    launches0 = _native.lib().la_launch_count()
    t_wall0 = time.perf_counter()
    t_region0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    t_region1 = time.time()
    launches = _native.lib().la_launch_count() - launches0
    clocks = sampler.stop(t_region0, t_region1)
    la.get_device_error(dev)
    ms = start.elapsed_time(end)
    ms = max_over_ranks(ms, ws, dev)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    dq_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    dkdv_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)

    tokens_step = B * T
    value = ws * tokens_step * args.steps / (ms * 1e-3)

    # Algorithmic bytes of each call, by the method's steps (bf16 tokens, fp32
    # states; one unit = one token tensor of B*T*H*128 bf16):
    #   la_fwd      (a1-a8)  q, k, v read, o written: 4 units + the fp32 final state
    #   la_bwd_dq   (b1)     k, v, do read, dq written: 4 units
    #   la_bwd_dkdv (b2)     q, k, v, do read, dk, dv written: 6 units
    # and the bytes its launches stream (what each kernel moves): a sweep
    # launch reads 3 token tensors and writes 1, so la_bwd_dkdv streams 4 units
    # per launch (2 launches when dv and dk run as separate sweeps).
    unit = B * T * H * D * 2
    state_bytes = B * H * D * E * 4
    n_launch = call_launches(la, q, k, v, do, g, scale)
    calls = {
        "la_fwd": dict(ms=fwd_ms, launches=n_launch["la_fwd"],
                       method=4 * unit + state_bytes,
                       stream=4 * unit * n_launch["la_fwd"] + state_bytes),
        "la_bwd_dq": dict(ms=dq_ms, launches=n_launch["la_bwd_dq"], method=4 * unit,
                          stream=4 * unit * n_launch["la_bwd_dq"]),
        "la_bwd_dkdv": dict(ms=dkdv_ms, launches=n_launch["la_bwd_dkdv"], method=6 * unit,
                            stream=4 * unit * n_launch["la_bwd_dkdv"]),
    }
    fused = n_launch["la_bwd_dkdv"] == 1
    groups = {
        "tc_sweep_kernel forward-type (la_fwd, la_bwd_dq)": ("la_fwd", "la_bwd_dq"),
        ("tc_dkdv_kernel (la_bwd_dkdv: dk and dv in one sweep)" if fused else
         "tc_sweep_kernel backward-type (la_bwd_dkdv: dv, dk)"): ("la_bwd_dkdv",),
    }
    gsum = {name: {f: sum(calls[c][f] for c in members)
                   for f in ("ms", "launches", "method", "stream")}
            for name, members in groups.items()}
    dom = max(gsum, key=lambda n: gsum[n]["ms"])
    gd = gsum[dom]
    peak, peak_src = peaks()
    tpeak, tpeak_src = tensor_peak()
    work = method_work(B, T, H, D, E)
    measured_rf = method_roofline(work, fwd_ms, dq_ms + dkdv_ms, peak, tpeak)
    method = {
        "definition": "per (token, head): bytes fwd 2(2d+2e) + final states, bwd 2(4d+3e); "
                      "FLOPs with 64-token chunks fwd 2C(d+e)+4de, bwd 6C(d+e)+10de; frac = "
                      "max(FLOPs / tensor peak, bytes / HBM peak) / measured; fwd = la_fwd, "
                      "bwd = la_bwd_dq + la_bwd_dkdv",
        "work": work,
        "step_tflops": (work["fwd_flops"] + work["bwd_flops"]) / (ms / args.steps * 1e-3) / 1e12,
        "measured_peaks": dict(measured_rf, hbm_gbs=peak, bf16_tflops=tpeak,
                               source=peak_src + "/" + tpeak_src),
        "nominal_peaks": dict(method_roofline(work, fwd_ms, dq_ms + dkdv_ms, NOMINAL_HBM_GBS,
                                              NOMINAL_BF16_TFLOPS),
                              hbm_gbs=NOMINAL_HBM_GBS, bf16_tflops=NOMINAL_BF16_TFLOPS),
    }
    ms_launch = gd["ms"] / gd["launches"]
    achieved = (gd["method"] / gd["launches"]) / (ms_launch * 1e-3) / 1e9
    streamed = (gd["stream"] / gd["launches"]) / (ms_launch * 1e-3) / 1e9
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "traffic_tc_sweep_kernel.json")
    if os.path.exists(tr_path):
        try:
            with open(tr_path) as f:
                tr = json.load(f)
            key = ("forward-type" if "forward-type" in dom else
                   "dkdv" if fused else "backward-type")
            entry = tr.get(key)
            if entry and entry.get("source_sha") == source_sha():
                traffic = entry["bytes_per_launch_scaled"] * T / entry["n_full"]
        except Exception:
            traffic = None
    # compulsory step traffic (forward and backward as separate passes, nothing saved in
    # between): forward reads q, k, v and writes o (4 units) plus the final state;
    # backward reads q, k, v, do and writes dq, dk, dv (7 units)
    roof_ms = (11 * unit + state_bytes) / (peak * 1e9) * 1e3

    # end to end: pinned host buffers -> device -> fwd+bwd -> host, every step
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (t.to("cpu").pin_memory() for t in (q, k, v, do))
        houts = [torch.empty((B, T, H, E), dtype=torch.bfloat16).pin_memory(),
                 torch.empty((B, T, H, D), dtype=torch.bfloat16).pin_memory(),
                 torch.empty((B, T, H, D), dtype=torch.bfloat16).pin_memory(),
                 torch.empty((B, T, H, E), dtype=torch.bfloat16).pin_memory(),
                 torch.empty((B, H, D, E), dtype=torch.float32).pin_memory()]

        # One batch row at a time on three streams, so that the copies of
        # neighbouring rows overlap the compute of this one: host-to-device
        # (q, k, v, do of row b), compute (la_fwd, la_bwd of row b), and
        # device-to-host (o, dq, dk, dv, final_state of row b).
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))

        def e2e_step():
            for b in range(B):
                with torch.cuda.stream(s_in):
                    xb = [t[b:b + 1].to(dev, non_blocking=True) for t in (hq, hk, hv, hdo)]
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(ev_in)
                    for t in xb:
                        t.record_stream(s_cmp)
                    o, fin = la.la_fwd(xb[0], xb[1], xb[2], g, scale)
                    gq, gk, gv, _ = la.la_bwd(xb[0], xb[1], xb[2], xb[3], g, scale,
                                              want_d_initial_state=False)
                    ev_cmp = torch.cuda.Event()
                    ev_cmp.record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp)
                    for h, d_ in zip(houts, (o, gq, gk, gv, fin)):
                        d_.record_stream(s_out)
                        h[b:b + 1].copy_(d_, non_blocking=True)

        for _ in range(max(1, min(args.warmup, 2))):
            e2e_step()
        torch.cuda.synchronize()
        ke = max(1, min(args.steps, 10))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        s_in.wait_stream(stream)
        for _ in range(ke):
            e2e_step()
        stream.wait_stream(s_out)
        t1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(t0.elapsed_time(t1), ws, dev)
        bi = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
        bo = sum(t.numel() * t.element_size() for t in houts)
        e2e = {"value": ws * tokens_step * ke / (e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": ke,
               "schedule": "per batch row: copy in, la_fwd + la_bwd, copy out, on three "
                           "streams (rows overlap)"}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGES_TOKENS_PER_S[T] if T in PAGES_TOKENS_PER_S else None,
        "dtype": "bf16", "data": "synthetic",
        "config": bench_config(B, H, T, D, E, ws),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "bytes_per_launch": gd["method"] / gd["launches"],
                     "bytes_definition": "the method's algorithmic bytes of the kernel's "
                                         "calls (la_fwd 4 units + final state, la_bwd_dq 4, "
                                         "la_bwd_dkdv 6; unit = one bf16 token tensor) per "
                                         "launch",
                     "ms_per_launch": ms_launch,
                     "stream_bytes_per_launch": gd["stream"] / gd["launches"],
                     "stream_frac": streamed / peak,
                     "method_fwd_frac": measured_rf["fwd"]["frac"],
                     "method_bwd_frac": measured_rf["bwd"]["frac"],
                     "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else peak_src,
                     "step_compulsory_frac": roof_ms / (ms / args.steps)},
        "method_roofline": method,
        "calls_ms": {"la_fwd": fwd_ms, "la_bwd_dq": dq_ms, "la_bwd_dkdv": dkdv_ms},
        "calls_ms_median": {
            "la_fwd": statistics.median(e[0].elapsed_time(e[1]) for e in evs),
            "la_bwd_dq": statistics.median(e[1].elapsed_time(e[2]) for e in evs),
            "la_bwd_dkdv": statistics.median(e[2].elapsed_time(e[3]) for e in evs)},
        "bytes_per_call": {c: calls[c]["method"] for c in calls},
        "launches_per_call": {c: calls[c]["launches"] for c in calls},
        "kernel_family": la.kernel_family(B, T, H, D, E),
        "gpu_launches": int(launches),
        "clocks": clocks,
        "e2e": e2e,
        "wall_s_timed": t_wall,
    }
    if not args.no_sweep:
        line["sweep"] = length_sweep(la, torch, dev, stream, T)
        line["configs"] = configs_bench(la, torch, dev, stream, peak, tpeak)
        line["decode"] = decode_bench(la, torch, dev, stream, peak)
        line["long_sequence"] = split_bench(la, torch, dev, stream, peak)
        line["grouped_kv"] = gqa_bench(la, torch, dev, stream, peak)
        line["gated"] = gla_bench(la, torch, dev, stream, peak)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.n, args.cpu_pairs)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def call_launches(la, q, k, v, do, g, scale):
    """Kernel launches of one call of each entry point of the step, by the
    library's own launch counter."""
    from linear_attention_head_gb300 import _native
    lib = _native.lib()
    out = {}
    for name, fn in (("la_fwd", lambda: la.la_fwd(q, k, v, g, scale)),
                     ("la_bwd_dq", lambda: la.la_bwd_dq(q, k, v, do, g, scale)),
                     ("la_bwd_dkdv", lambda: la.la_bwd_dkdv(q, k, v, do, g, scale,
                                                            want_d_initial_state=False))):
        n0 = lib.la_launch_count()
        fn()
        out[name] = max(1, int(lib.la_launch_count() - n0))
    return out


def length_sweep(la, torch, dev, stream, skip_n):
    """fwd and bwd times at every length of the Lightning-2 benchmark table (b4 h32
    d=e=128 bf16), each the median of 20 calls after 5 warm-up calls.  The GPU is first
    held busy (torch.cuda._sleep) so that all 5 calls are queued before the first
    runs and host-side call overhead stays out of the events.  Lengths up to 4096
    tokens are timed with a 512 MB L2 flush before each call (`fwd_ms`, `bwd_ms`)
    and also back to back without one (`*_unflushed`); longer ones stream more
    than the 129 MB L2 holds per call and are timed back to back."""
    import workloads as W
    out = {}
    hbm, tfl = peaks()[0], tensor_peak()[0]
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for n in W.SWEEP_LENGTHS:
        if n == skip_n:
            continue
        w = W.sweep_bf16(n)
        gen = torch.Generator(device=dev).manual_seed(7)
        q, k, v, do = (torch.randn((w.B, n, w.H, w.d), generator=gen, device=dev).bfloat16()
                       for _ in range(4))
        g = w.g_gamma.to(dev)
        small = n <= 4096

        def timed(fn, flush_first):
            return _timed_calls(torch, stream, fn, flush if flush_first else None)

        fwd = lambda: la.la_fwd(q, k, v, g, w.scale)
        bwd = lambda: la.la_bwd(q, k, v, do, g, w.scale, want_d_initial_state=False)
        f_ms, b_ms = timed(fwd, small), timed(bwd, small)
        tps = w.B * n / ((f_ms + b_ms) * 1e-3)
        rf = method_roofline(method_work(w.B, n, w.H, w.d, w.e), f_ms, b_ms, hbm, tfl)
        out[str(n)] = {"fwd_ms": f_ms, "bwd_ms": b_ms, "tokens_per_s": tps,
                       "vs_pages": tps / PAGES_TOKENS_PER_S[n], "l2_flushed": small,
                       "tflops_fwd": rf["fwd"]["tflops"], "tflops_bwd": rf["bwd"]["tflops"],
                       "roofline_frac_fwd": rf["fwd"]["frac"],
                       "roofline_frac_bwd": rf["bwd"]["frac"]}
        if small:
            out[str(n)]["fwd_ms_unflushed"] = timed(fwd, False)
            out[str(n)]["bwd_ms_unflushed"] = timed(bwd, False)
        del q, k, v, do
    return out


def _timed_calls(torch, stream, fn, flush=None, calls=20, warm=5):
    """Median event time of `calls` calls of fn queued behind torch.cuda._sleep (no host
    gap enters the events), after `warm` untimed calls; with `flush`, that buffer is
    overwritten before each call (an L2 flush, inside the stream but outside the events)."""
    import statistics
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    evs = []
    torch.cuda._sleep(20_000_000)
    for _ in range(calls):
        if flush is not None:
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)


def packed_work(T, H, d, e, n_seqs, token_bytes=2):
    """The method's work for packed sequences with states in and out (same accounting as
    method_work): forward adds the initial state read and the final state written,
    backward the initial state (dq sweep) and d_final_state read and d_initial_state
    written."""
    w = method_work(1, T, H, d, e, token_bytes)
    st = n_seqs * H * d * e * 4
    w["fwd_bytes"] = T * H * token_bytes * (2 * d + 2 * e) + 2 * st
    w["bwd_bytes"] = T * H * token_bytes * (4 * d + 3 * e) + 3 * st
    return w


def configs_bench(la, torch, dev, stream, hbm, tfl):
    """The other workload shapes, fwd and bwd timed separately (median of 20 queued
    calls after 5 warm-up calls):
      * b1 h2 n256 d=e=32 fp32, forward only (L2 flushed before each call);
      * b2 h8 n2048 d=e=64 and b2 h12 n2048 d=e=192 (bf16): their token tensors fit
        in L2, so each call follows a 512 MB L2 flush (`*_ms`); back to back without
        one in `*_ms_unflushed`;
      * 16 packed sequences of U[64, 8192] tokens (seed 0), h16 d=e=128 bf16, initial
        state and d_final_state in, final state and d_initial_state out, reverse off
        and on; each with the longest-first schedule (the library's workspace) and
        without it (no workspace: index order).  Its tensors exceed L2; no flush.
    Fractions are the method's roofline against the measured peaks."""
    import workloads as W
    out = {}
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for w in (W.small_bf16(), W.d192_bf16()):
        gen = torch.Generator(device=dev).manual_seed(23)
        q, k = (torch.randn((w.B, w.T, w.H, w.d), generator=gen, device=dev).bfloat16()
                for _ in range(2))
        v, do = (torch.randn((w.B, w.T, w.H, w.e), generator=gen, device=dev).bfloat16()
                 for _ in range(2))
        g = w.g_gamma.to(dev)
        fwd = lambda: la.la_fwd(q, k, v, g, w.scale)
        bwd = lambda: la.la_bwd(q, k, v, do, g, w.scale, want_d_initial_state=False)
        f_ms, b_ms = _timed_calls(torch, stream, fwd, flush), _timed_calls(torch, stream, bwd, flush)
        rf = method_roofline(method_work(w.B, w.T, w.H, w.d, w.e), f_ms, b_ms, hbm, tfl)
        out[w.name] = {
            "kernel_family": la.kernel_family(w.B, w.T, w.H, w.d, w.e),
            "fwd_ms": f_ms, "bwd_ms": b_ms, "tokens_per_s": w.B * w.T / ((f_ms + b_ms) * 1e-3),
            "roofline_frac_fwd": rf["fwd"]["frac"], "roofline_frac_bwd": rf["bwd"]["frac"],
            "tflops_fwd": rf["fwd"]["tflops"], "tflops_bwd": rf["bwd"]["tflops"],
            "fwd_ms_unflushed": _timed_calls(torch, stream, fwd),
            "bwd_ms_unflushed": _timed_calls(torch, stream, bwd),
            "l2": "flushed before each call (512 MB write)"}
        del q, k, v, do
    # config 1: b1 h2 n256 d=e=32 fp32, forward only (the CUDA-core chunked
    # kernels; fp32 tokens, 4-byte method bytes)
    w = W.tiny_fp32()
    gen = torch.Generator(device=dev).manual_seed(31)
    q, k, v = (torch.randn((w.B, w.T, w.H, w.d), generator=gen, device=dev) for _ in range(3))
    g = w.g_gamma.to(dev)
    fwd = lambda: la.la_fwd(q, k, v, g, w.scale)
    f_ms = _timed_calls(torch, stream, fwd, flush)
    rf = method_roofline(method_work(w.B, w.T, w.H, w.d, w.e, token_bytes=4), f_ms, f_ms, hbm,
                         tfl)
    out[w.name] = {"kernel_family": la.kernel_family(w.B, w.T, w.H, w.d, w.e, dtype=torch.float32),
                   "fwd_ms": f_ms, "tokens_per_s": w.B * w.T / (f_ms * 1e-3),
                   "roofline_frac_fwd": rf["fwd"]["frac"],
                   "fwd_ms_unflushed": _timed_calls(torch, stream, fwd),
                   "l2": "flushed before each call (512 MB write)"}
    del q, k, v
    w = W.varlen_bf16(seed=0)
    gen = torch.Generator(device=dev).manual_seed(29)
    q, k = (torch.randn((1, w.T, w.H, w.d), generator=gen, device=dev).bfloat16()
            for _ in range(2))
    v, do = (torch.randn((1, w.T, w.H, w.e), generator=gen, device=dev).bfloat16()
             for _ in range(2))
    S = (w.num_seqs, w.H, w.d, w.e)
    init = torch.randn(S, generator=gen, device=dev) * 0.02
    dfin = torch.randn(S, generator=gen, device=dev) * 0.02
    g = w.g_gamma.to(dev)
    cu = w.cu_seqlens
    work = packed_work(w.T, w.H, w.d, w.e, w.num_seqs)
    pk = {"workload": "16 packed sequences, lengths U[64, 8192] (seed 0, %d tokens, longest %d),"
                      " h16 d=e=128 bf16, states in and out" % (w.T, max(w.seqlens)),
          "tokens": w.T}
    for rev in (False, True):
        for sched in (True, False):
            fwd = lambda: la.la_fwd(q, k, v, g, w.scale, init, rev, cu, workspace=sched)
            bwd = lambda: la.la_bwd(q, k, v, do, g, w.scale, init, dfin, rev, cu,
                                    workspace=sched)
            f_ms, b_ms = _timed_calls(torch, stream, fwd), _timed_calls(torch, stream, bwd)
            rf = method_roofline(work, f_ms, b_ms, hbm, tfl)
            pk["%s_%s" % ("reverse" if rev else "forward",
                          "longest_first" if sched else "index_order")] = {
                "fwd_ms": f_ms, "bwd_ms": b_ms, "tokens_per_s": w.T / ((f_ms + b_ms) * 1e-3),
                "roofline_frac_fwd": rf["fwd"]["frac"], "roofline_frac_bwd": rf["bwd"]["frac"]}
    out["varlen16_h16_d128_bf16"] = pk
    la.get_device_error(dev)
    del q, k, v, do, flush
    return out


def decode_bench(la, torch, dev, stream, peak):
    """Decoding against a carried state (the token-by-token kernels): la_fwd on
    a batch of 64 sequences x 32 heads, d = e = 128 bf16, with a fp32 initial
    state in and the final state out, for 1 and 16 new tokens per sequence.
    Each point is the mean of 20 calls queued behind torch.cuda._sleep, so no
    host gap enters the events.  Bound: HBM; algorithmic bytes per call = the
    state read and written (2 x B*H*d*e*4) + q, k, v read and o written."""
    import workloads as W
    B, H, D, E = 64, 32, 128, 128
    g = W.alibi_g_gamma(H).to(dev)
    gen = torch.Generator(device=dev).manual_seed(11)
    s0 = torch.randn((B, H, D, E), generator=gen, device=dev) * 0.1
    fin = torch.empty_like(s0)
    out = {}
    for T in (1, 16):
        q, k, v = (torch.randn((B, T, H, D), generator=gen, device=dev).bfloat16()
                   for _ in range(3))
        o = torch.empty_like(v)
        fn = lambda: la.la_fwd(q, k, v, g, D ** -0.5, s0, out=o, final_state=fin)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        torch.cuda._sleep(20_000_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(20):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 20
        nbytes = 2 * B * H * D * E * 4 + 4 * B * T * H * D * 2
        out["b%d_h%d_t%d" % (B, H, T)] = {
            "kernel_family": la.kernel_family(B, T, H, D, E), "us_per_call": ms * 1e3,
            "tokens_per_s": B * T / (ms * 1e-3), "bytes_per_call": nbytes,
            "achieved_gbs": nbytes / (ms * 1e-3) / 1e9, "frac_of_peak": nbytes / (ms * 1e-3) / 1e9 / peak}
        del q, k, v, o
    la.get_device_error(dev)
    return out


def split_bench(la, torch, dev, stream, peak):
    """One long sequence with few heads (b1 h8 n262144 d=e=128 bf16): 8
    (sequence, head) pairs for 152 SMs.  la_fwd + la_bwd with the sequence
    split (the library's default) and without it (la_set_sequence_split(0)),
    each the mean of 5 queued steps after 2 warm-up steps.  Algorithmic bytes
    per step are the unsplit sweeps' compulsory traffic (11 token tensors)."""
    import workloads as W
    from linear_attention_head_gb300 import _native
    B, T, H, D = 1, 262144, 8, 128
    g = W.alibi_g_gamma(H).to(dev)
    gen = torch.Generator(device=dev).manual_seed(13)
    q, k, v, do = (torch.randn((B, T, H, D), generator=gen, device=dev).bfloat16()
                   for _ in range(4))

    def step():
        la.la_fwd(q, k, v, g, 1.0)
        la.la_bwd(q, k, v, do, g, 1.0, want_d_initial_state=False)

    out = {"workload": "fwd+bwd b1 h8 n262144 d=e=128 bf16, ALiBi slopes, scale 1"}
    nbytes = 11 * B * T * H * D * 2
    for name, mode in (("split", 1), ("unsplit", 0)):
        _native.check(_native.lib().la_set_sequence_split(mode, 0))
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        torch.cuda._sleep(20_000_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 5
        out[name] = {"ms_per_step": ms, "tokens_per_s": B * T / (ms * 1e-3),
                     "compulsory_frac_of_peak": nbytes / (ms * 1e-3) / 1e9 / peak}
    _native.check(_native.lib().la_set_sequence_split(1, 0))
    la.get_device_error(dev)
    del q, k, v, do
    return out


def gqa_bench(la, torch, dev, stream, peak):
    """Grouped key/value heads: b4 h32 with 8 key/value heads, n32768 d=e=128 bf16.
    la_fwd and la_bwd timed separately (mean of 5 queued calls after 2 warm-up
    calls).  Algorithmic bytes: forward reads q and the shared k, v and writes o;
    backward reads q, k, v, do and writes dq, dk, dv (k, v, dk, dv at 8 heads)."""
    import workloads as W
    B, T, H, Hkv, D = 4, 32768, 32, 8, 128
    g = W.alibi_g_gamma(H).to(dev)
    gen = torch.Generator(device=dev).manual_seed(17)
    q, do = (torch.randn((B, T, H, D), generator=gen, device=dev).bfloat16() for _ in range(2))
    k, v = (torch.randn((B, T, Hkv, D), generator=gen, device=dev).bfloat16() for _ in range(2))

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        torch.cuda._sleep(20_000_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 5

    f_ms = timed(lambda: la.la_fwd(q, k, v, g, 1.0))
    b_ms = timed(lambda: la.la_bwd(q, k, v, do, g, 1.0, want_d_initial_state=False))
    full, kvu = B * T * H * D * 2, B * T * Hkv * D * 2
    fb, bb = 2 * full + 2 * kvu, 3 * full + 4 * kvu + 2 * kvu
    la.get_device_error(dev)
    del q, k, v, do
    return {"workload": "fwd+bwd b4 h32 kv_heads8 n32768 d=e=128 bf16, ALiBi slopes, scale 1",
            "fwd_ms": f_ms, "bwd_ms": b_ms, "tokens_per_s": B * T / ((f_ms + b_ms) * 1e-3),
            "fwd_frac_of_peak": fb / (f_ms * 1e-3) / 1e9 / peak,
            "bwd_compulsory_frac_of_peak": bb / (b_ms * 1e-3) / 1e9 / peak}


def gla_bench(la, torch, dev, stream, peak):
    """Gated form (GLA, per-key gate): b4 h32 n8192 d=e=128 bf16, gate fp32.
    gla_fwd alone, then a step (gla_fwd keeping its rescaled operands, gla_bwd
    reusing them); bwd_ms = step - fwd.  The chunked tensor-core form: operand
    pre-pass, tcgen05 sweeps, and for the backward the in-place rescaling of
    dq, dk with dg.  Each figure is the mean of 3 queued calls after 1 warm-up
    call; bwd_alone_ms is gla_bwd computing the operands itself.  Algorithmic bytes: forward reads q, k, v, g
    and writes o; backward reads q, k, v, do, g and writes dq, dk, dv, dg."""
    import workloads as W
    B, T, H, D = 4, 8192, 32, 128
    gg = W.alibi_g_gamma(H).to(dev)
    gen = torch.Generator(device=dev).manual_seed(19)
    q, k, v, do = (torch.randn((B, T, H, D), generator=gen, device=dev).bfloat16()
                   for _ in range(4))
    g = -0.3 * torch.rand((B, T, H, D), generator=gen, device=dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        torch.cuda._sleep(20_000_000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 3

    def step():
        # a training step: the backward reuses the forward's rescaled q, k
        o, fin, ops = la.gla_fwd(q, k, v, g, gg, 1.0, keep_operands=True)
        la.gla_bwd(q, k, v, do, g, gg, 1.0, want_d_initial_state=False, operands=ops)

    f_ms = timed(lambda: la.gla_fwd(q, k, v, g, gg, 1.0))
    b_alone_ms = timed(lambda: la.gla_bwd(q, k, v, do, g, gg, 1.0, want_d_initial_state=False))
    s_ms = timed(step)
    b_ms = s_ms - f_ms
    unit = B * T * H * D * 2
    la.get_device_error(dev)
    del q, k, v, do, g
    out = {"workload": "fwd+bwd b4 h32 n8192 d=e=128 bf16 tokens, fp32 per-key gate",
           "kernels": "chunked tensor-core form (operand pre-pass + tcgen05 sweeps)",
           "fwd_ms": f_ms, "bwd_ms": b_ms, "step_ms": s_ms, "bwd_alone_ms": b_alone_ms,
           "tokens_per_s": B * T / (s_ms * 1e-3),
           "fwd_frac_of_peak": (4 * unit + 2 * unit) / (f_ms * 1e-3) / 1e9 / peak,
           "bwd_frac_of_peak": (7 * unit + 4 * unit) / (b_ms * 1e-3) / 1e9 / peak}
    out["long_sequence"] = gla_long_bench(la, torch, dev, timed, peak)
    return out


def gla_long_bench(la, torch, dev, timed, peak):
    """The gated form on one long sequence with few heads (b1 h8 n262144
    d=e=128 bf16, fp32 gate): 8 (sequence, head) pairs for 152 SMs, with the
    sequence split (segment decays, pre-pass, passes around scans with
    per-channel decays, dg offsets per segment) and without it.  gla_fwd alone,
    and a training step: gla_fwd then gla_bwd (unsplit, the backward reuses
    the forward's operands; split, it computes its own).  Algorithmic bytes:
    forward q, k, v, g read (the gate fp32), o written; backward q, k, v, do,
    g read, dq, dk, dv, dg written."""
    import workloads as W
    from linear_attention_head_gb300 import _native
    B, T, H, D = 1, 262144, 8, 128
    gg = W.alibi_g_gamma(H).to(dev)
    gen = torch.Generator(device=dev).manual_seed(23)
    q, k, v, do = (torch.randn((B, T, H, D), generator=gen, device=dev).bfloat16()
                   for _ in range(4))
    g = -0.3 * torch.rand((B, T, H, D), generator=gen, device=dev)

    def step():
        o, fin, ops = la.gla_fwd(q, k, v, g, gg, 1.0, keep_operands=True)
        la.gla_bwd(q, k, v, do, g, gg, 1.0, want_d_initial_state=False, operands=ops)

    out = {"workload": "gla_fwd + gla_bwd b1 h8 n262144 d=e=128 bf16 tokens, fp32 per-key gate"}
    unit = B * T * H * D * 2
    for name, mode in (("split", 1), ("unsplit", 0)):
        _native.check(_native.lib().la_set_sequence_split(mode, 0))
        f_ms = timed(lambda: la.gla_fwd(q, k, v, g, gg, 1.0))
        s_ms = timed(step)
        out[name] = {"fwd_ms": f_ms, "step_ms": s_ms, "tokens_per_s": B * T / (s_ms * 1e-3),
                     "fwd_frac_of_peak": 6 * unit / (f_ms * 1e-3) / 1e9 / peak,
                     "bwd_frac_of_peak": 11 * unit / ((s_ms - f_ms) * 1e-3) / 1e9 / peak}
    _native.check(_native.lib().la_set_sequence_split(1, 0))
    la.get_device_error(dev)
    del q, k, v, do, g
    return out


def source_sha():
    """Hash of the device code the tensor-core kernels of the step are built
    from (the sweep kernel and the fused dk/dv kernel, whose ncu traffic
    profiles/traffic_tc_sweep_kernel.json records; the shared declarations of
    la_internal.h, which every kernel file includes, are left out)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_head_gb300", "csrc")
    for f in ("la_sm100.cuh", "la_tc_common.cuh", "la_tc_sweep.cu", "la_tc_dkdv.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _oracle_sample(n, pairs, n_sample, seed=0):
    """A bounded sample of the workload for the CPU oracle: `pairs` (batch, head)
    streams (heads spread over the decay slopes) of the first n_sample tokens.  The
    oracle's cost is linear in the tokens of each stream, so tokens/s of the sample
    scales to the full job by the ratio of streams."""
    import torch
    import workloads as W
    w = W.sweep_bf16(n)
    H = w.H
    heads = [int(round(i * (H - 1) / max(pairs - 1, 1))) for i in range(pairs)]
    gen = torch.Generator().manual_seed(seed)
    shp = (1, min(n, n_sample), pairs, w.d)
    q, k, v, do = (torch.randn(shp, generator=gen).bfloat16() for _ in range(4))
    g = w.g_gamma[heads].clone()
    return w, q, k, v, do, g


def _oracle_step(w, q, k, v, do, g, cores):
    import oracle
    oracle.forward(q, k, v, g, w.scale, threads=cores)
    oracle.backward(q, k, v, g, w.scale, do, threads=cores)


def cpu_model():
    """The host CPU's name from /proc/cpuinfo (x86 `model name`; Arm implementer and
    part numbers), else the machine type."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                fields.setdefault(key.strip().lower(), val.strip())
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    if fields.get("cpu part"):
        return "%s implementer %s part %s" % (platform.machine(),
                                              fields.get("cpu implementer", "?"),
                                              fields["cpu part"])
    return platform.machine() or "unknown"


def cpu_baseline(n, pairs=None, n_sample=32768):
    """The fp64 oracle as it stands, fwd+bwd, timed on the host cores on a bounded sample;
    reported as the full workload's tokens/s."""
    import oracle
    cores = os.cpu_count() or 1
    pairs = pairs or min(cores, 16)
    w, q, k, v, do, g = _oracle_sample(n, pairs, n_sample)
    oracle._load()
    t0 = time.perf_counter()
    _oracle_step(w, q, k, v, do, g, cores)
    dt = time.perf_counter() - t0
    ns = q.shape[1]
    value = pairs * ns / dt / w.H          # tokens of one (all-heads) sequence per second
    return {"value": value, "unit": "tokens/s", "cores": min(cores, pairs), "kind": "oracle",
            "host_cpus": cores, "cpu_model": cpu_model(),
            "sample": "fwd+bwd of %d (batch, head) streams x %d tokens of the %d x %d-token "
                      "workload in %.2f s on %d threads; tokens/s = streams*tokens/time/H"
                      % (pairs, ns, w.B * w.H, n, dt, min(cores, pairs))}


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    cores = os.cpu_count() or 1
    pairs = args.cpu_pairs or min(cores, 16)
    w, q, k, v, do, g = _oracle_sample(args.n, pairs, 4096)
    oracle._load()
    for _ in range(max(0, min(args.warmup, 1))):
        _oracle_step(w, q[:, :128], k[:, :128], v[:, :128], do[:, :128], g, cores)
    dt = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_step(w, q, k, v, do, g, cores)
        dt += time.perf_counter() - t0
    ns = q.shape[1]
    value = pairs * ns * args.steps / dt / w.H
    sample = ("per step: fwd+bwd of %d (batch, head) streams x %d tokens of the %d x %d-token "
              "workload on %d host threads; tokens/s = streams*tokens/time/H"
              % (pairs, ns, w.B * w.H, args.n, min(cores, pairs)))
    # ms_per_step is the time of one timed step as run (the bounded sample);
    # the full workload's step time at the same rate is reported beside it
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3,
            "projected_full_workload_ms_per_step": w.B * args.n / value * 1e3,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w.B, w.H, args.n, w.d, w.e, ws),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, pairs),
                             "kind": "oracle", "host_cpus": cores, "cpu_model": cpu_model(),
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--n", type=int, default=32768)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--cpu-pairs", type=int, default=None)
    ap.add_argument("--only", default=None,
                    choices=["sweep", "configs", "decode", "long_sequence", "grouped_kv",
                             "gated"],
                    help="run one of the secondary measurements alone (one GPU) and print "
                         "its JSON object")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl != "reference":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.only:
        section_only(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        gpu_bench(args)


def section_only(args):
    """One secondary measurement of the bench line on cuda:0, e.g. for a profiler."""
    import torch
    import linear_attention_head_gb300 as la
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peak, _ = peaks()
    tpeak, _ = tensor_peak()
    fn = {"sweep": lambda: length_sweep(la, torch, dev, stream, args.n),
          "configs": lambda: configs_bench(la, torch, dev, stream, peak, tpeak),
          "decode": lambda: decode_bench(la, torch, dev, stream, peak),
          "long_sequence": lambda: split_bench(la, torch, dev, stream, peak),
          "grouped_kv": lambda: gqa_bench(la, torch, dev, stream, peak),
          "gated": lambda: gla_bench(la, torch, dev, stream, peak)}[args.only]
    print(json.dumps({args.only: fn()}), flush=True)


if __name__ == "__main__":
    main()
