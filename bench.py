"""Benchmark of the renderer bank-attention hot path on one GB300.

A step is one ff_render_attn call of the Wan2.1-1.3B 480p workload at steady
state: RoPE of the chunk's Q/K, publish of (K, V) into the stage bank, and
attention of 4680 queries x 12 heads x d 128 over 2 anchor + 15 history + 3 own
latent frames (31200 keys), which the attention kernel gathers by reading the
bank slots in place.  Steps rotate over the 4 stage banks (and over layers when
more steps are asked for), always at chunks with full history.  Inputs are
seeded synthetic tensors (AR(1) unit-RMS Q/K, N(0,1) V) already resident in
HBM; each call touches ~300 MB, more than L2, so no extra flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gb300,reference}]

Prints one JSON line.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Renderer bank-attention TFLOP/s (% BF16 peak) and chunk-steps/s on 1 GB300"
WORKLOAD = "wan13b_480p"   # 12 heads, d 128, 30x52 tokens/frame, chunk 3 frames, H 5, 2 anchors
LAYERS_PER_CHUNK_STEP = 30  # Wan2.1-1.3B transformer blocks: a chunk-step runs every layer once
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture of the
# steady 1.3B call issued as a batch of 4 calls (profiles/*_wan13b_480p.md), with the
# source digest the counters belong to and the calls the captured launch covered: a
# kernel edited since then, or a launch of another size, reports null.
NCU_TRAFFIC = {
    "bank_attn_kernel": (838.6e6, "ff_attn.cu", "961f0ca6a71ba0a2", 4),
    "rope_publish_kernel": (288.6e6, "ff_publish.cu", "f39c3097d7c98795", 4),
}


def ncu_traffic(kernel, calls_per_launch):
    import hashlib
    nbytes, src, digest, calls = NCU_TRAFFIC[kernel]
    path = os.path.join(ROOT, "kv_cache_attention_ff_gb300", "csrc", src)
    try:
        with open(path, "rb") as f:
            now = hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None
    return nbytes if now == digest and calls == calls_per_launch else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            out = {}
            for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(k)
                if isinstance(v, dict):
                    v = v.get("value")
                if isinstance(v, (int, float)):
                    out[k] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


# nominal dense bf16 tensor rate of one GB300 (HGX B300 datasheet: 36 PFLOP/s with
# 2:4 sparsity per 8 GPUs = 2.25 PFLOP/s dense per GPU); context beside the measured peaks
DATASHEET_BF16_TFLOPS = 2250.0


def bench_config(world=1, stage_streams=1, batch=1):
    """The `config` of the JSON line: the same dict for the GPU arm and the
    reference (oracle) arm."""
    return {"workload": WORKLOAD, "heads": 12, "head_dim": 128, "tokens_per_frame": 1560, "queries": 4680,
            "keys": 31200, "anchors": 2, "history_chunks": 5, "chunk_frames": 3, "stages": 4,
            "parallelism": "replicas" if world > 1 else "single GPU", "stage_streams": stage_streams,
            "calls_per_launch": batch,
            "l2": "inputs larger than L2 (~300 MB touched per call)"}


def workload_numbers(T=1560, heads=12, d=128, nq_frames=3, key_frames=20):
    nq, nk = nq_frames * T, key_frames * T
    flops = 4.0 * nq * nk * d * heads
    F = T * heads * d * 2
    # RoPE/publish algorithmic bytes per steady call: read q, k, v (9F); write
    # Q_rot (3F) and the slot's K, V (6F).  The context is not copied.
    g1_bytes = 18.0 * F
    return nq, nk, flops, g1_bytes


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every `interval_ms` while running;
    the summary keeps the samples taken inside the timed window when there are any."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 200):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def mark(self, t0, t1):
        """Host wall-clock bounds (time.time()) of the timed region."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        import datetime
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = rows
        where = "all samples (none inside the timed window)"
        if self.window is not None:
            t0, t1 = self.window
            sel = [r for r in rows if t0 - 0.025 <= r[0] <= t1 + 0.025]
            if sel:
                inside, where = sel, "timed window"
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        sm = [r[1] for r in inside]
        smax = [r[2] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": where}


def gate(stream, us=1000.0):
    """Hold `stream` for about `us` microseconds before a timed region starts, so
    that the host has queued the first calls of the region when its start event
    fires: the region then measures the GPU's work, not the host's first
    enqueue.  Every call of the region is still inside it."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2000))  # cycles at about 2 GHz


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(ms_local, work_per_rank, world, pg=None, device=None):
    """Whole-job throughput of N replicas: the timed interval is the maximum over
    ranks, the work is the sum (every rank does the same work).  Returns
    (max interval in ms, work units per second / 1e12)."""
    import torch
    ms = float(ms_local)
    if pg is not None and world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t.item())
    return ms, work_per_rank * world / (ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import torch

    from kv_cache_attention_ff_gb300 import build, ff, synth

    world, rank, local = dist_setup()
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device(f"cuda:{local}")
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    T, H, D = 1560, 12, 128
    nq, nk, flops, g1_bytes = workload_numbers()
    steady_per_layer = 4 * (27 - 5)  # chunks 5..26 of each stage have full history
    total_calls = args.warmup + args.steps
    n_layers = max(1, math.ceil(total_calls / steady_per_layer))
    bank = ff.Bank(n_layers=n_layers, n_stages=4, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=9,
                   total_frames=81, heads=H, head_dim=D, frame_h=30, frame_w=52, device=local)
    stream = torch.cuda.Stream(device=dev)
    cfg_id = 2
    # anchors of every layer (3 planner blocks of 3)
    with torch.cuda.stream(stream):
        ka = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, list(range(0, 81, 10)), T, H, D, "ar",
                                 device=dev)
        va = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, list(range(0, 81, 10)), T, H, D, "normal",
                                 device=dev)
        for layer in range(n_layers):
            for b in range(3):
                sl = slice(3 * b * T, 3 * (b + 1) * T)
                bank.anchor_publish(layer, 30 * b, 3, ka[sl].contiguous(), va[sl].contiguous(), stream)
    # pool of 4 input sets (q, k, v) per stage, AR(1) over consecutive frames
    pool = []
    for st in range(4):
        qs = synth.DeviceARStream(cfg_id, 0, st, synth.Q, T, H, D, "ar", device=dev)
        ks = synth.DeviceARStream(cfg_id, 0, st, synth.K, T, H, D, "ar", device=dev)
        vs = synth.DeviceARStream(cfg_id, 0, st, synth.V, T, H, D, "normal", device=dev)
        pool.append([(qs.frames(3), ks.frames(3), vs.frames(3)) for _ in range(4)])
    out = torch.empty((nq, H, D), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()

    # ramp-up chunks 0..4 of every (layer, stage): untimed
    for layer in range(n_layers):
        for st in range(4):
            for i in range(5):
                q, k, v = pool[st][i % 4]
                bank.render_attn(layer, st, i, q, k, v, out, stream)
    next_chunk = {(l, s): 5 for l in range(n_layers) for s in range(4)}
    order = [(l, s) for l in range(n_layers) for s in range(4)]
    seq = []
    while len(seq) < total_calls:
        for key in order:
            if next_chunk[key] < 27 and len(seq) < total_calls:
                seq.append((key[0], key[1], next_chunk[key]))
                next_chunk[key] += 1
    assert all(c >= 5 for _, _, c in seq)

    # one CUDA stream per denoising stage: calls of different stages are independent
    # (anti-diagonal chunks of the stage wavefront), so one stage's HBM-bound
    # publish/gather and combine can run under another stage's attention
    n_streams = max(1, min(4, args.stage_streams))
    sstreams = [torch.cuda.Stream(device=dev) for _ in range(n_streams)] if n_streams > 1 else [stream]
    souts = [torch.empty((nq, H, D), dtype=torch.bfloat16, device=dev) for _ in range(4)]

    def call(j):
        layer, st, c = seq[j]
        q, k, v = pool[st][j % 4]
        rc = bank.render_attn_raw(layer, st, c, q.data_ptr(), k.data_ptr(), v.data_ptr(), souts[st].data_ptr(),
                                  sstreams[st % n_streams].cuda_stream)
        if rc != 0:
            raise RuntimeError(f"ff_render_attn failed with status {rc}")

    def call_batch(j0, j1):
        # consecutive calls rotate over the 4 stages: every batch has distinct stages
        calls = []
        for j in range(j0, j1):
            layer, st, c = seq[j]
            q, k, v = pool[st][j % 4]
            calls.append((layer, st, c, q.data_ptr(), k.data_ptr(), v.data_ptr(), souts[st].data_ptr()))
        rc = bank.render_attn_batch_raw(calls, stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"ff_render_attn_batch failed with status {rc}")

    def run_calls(j0, j1):
        if args.batch <= 1:
            for j in range(j0, j1):
                call(j)
        else:
            for jb in range(j0, j1, args.batch):
                call_batch(jb, min(j1, jb + args.batch))

    run_calls(0, args.warmup)
    torch.cuda.synchronize()
    bank.set_timing(True)
    sampler = ClockSampler(local, args.clock_ms)
    sampler.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    gate(stream)
    e0.record(stream)
    for ss in sstreams:
        ss.wait_event(e0)
    run_calls(args.warmup, total_calls)
    for ss in sstreams:
        done = torch.cuda.Event()
        done.record(ss)
        stream.wait_event(done)
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(wall0, time.time())
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    ms_total = e0.elapsed_time(e1)
    kt = bank.read_timing()
    bank.set_timing(False)
    assert bank.error_poll() == 0, "device-side wait timed out"
    ms_total, value = aggregate(ms_total, flops * args.steps, world, pg, dev)
    ms_step = ms_total / args.steps

    peaks, peak_src = load_peaks()
    # a kernel timed while the power cap governs the clocks is compared with the
    # sustained bf16 figure, one timed at full clocks with the burst figure
    sustained = "sw_power_cap" in (clocks.get("reasons") or []) and "bf16_tflops_sustained" in peaks
    bf16_key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    bf16_label = "sustained (sw_power_cap active in the timed window)" if sustained else "burst"
    attn_ms = kt.attn_ms / max(kt.calls, 1)      # per call
    pub_ms = kt.publish_ms / max(kt.calls, 1)
    comb_ms = kt.combine_ms / max(kt.calls, 1)
    n_launch = math.ceil(args.steps / max(1, args.batch))  # attention (and publish) launches in the timed region
    per_launch = kt.calls / max(n_launch, 1)                # calls one launch covers
    attn_tflops = flops / (attn_ms * 1e-3) / 1e12
    pub_gbs = g1_bytes / (pub_ms * 1e-3) / 1e9
    roofline = {"kernel": "bank_attn_kernel", "bound": "tensor", "achieved": round(attn_tflops, 1),
                "peak": peaks[bf16_key], "unit": "TFLOP/s", "frac": round(attn_tflops / peaks[bf16_key], 4),
                "traffic": ncu_traffic("bank_attn_kernel", per_launch), "traffic_unit": "bytes/launch",
                "peak_source": f"{peak_src} {bf16_key} ({bf16_label})",
                # the same launch against every denominator, side by side
                "frac_of_burst": round(attn_tflops / peaks["bf16_tflops"], 4),
                "frac_of_sustained": (round(attn_tflops / peaks["bf16_tflops_sustained"], 4)
                                      if "bf16_tflops_sustained" in peaks else None),
                "frac_of_datasheet": round(attn_tflops / DATASHEET_BF16_TFLOPS, 4),
                "datasheet_peak": DATASHEET_BF16_TFLOPS,
                "algorithmic_per_launch": f"{per_launch * flops / 1e9:.1f} GFLOP ({per_launch:g} calls x 4*Nq*Nk*d*h)",
                "avg_launch_ms": round(attn_ms * per_launch, 4)}
    pub_traffic = ncu_traffic("rope_publish_kernel", per_launch)
    roofline_publish = {"kernel": "rope_publish_kernel", "bound": "hbm", "achieved": round(pub_gbs, 1),
                        "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(pub_gbs / peaks["hbm_gbs"], 4),
                        "achieved_is": "effective bandwidth: algorithmic bytes / launch time (its writes stay in L2)",
                        "traffic": pub_traffic, "traffic_unit": "bytes/launch",
                        "dram_gbs": round(pub_traffic / (pub_ms * per_launch * 1e-3) / 1e9, 1) if pub_traffic else None,
                        "peak_source": f"{peak_src} hbm_gbs",
                        "algorithmic_per_launch": f"{per_launch * g1_bytes / 1e6:.1f} MB ({per_launch:g} calls x "
                                                  f"18 frames x 4.79 MB)",
                        "avg_launch_ms": round(pub_ms * per_launch, 4)}

    # end to end: pinned host inputs -> device, call, output -> pinned host, every step
    e2e = None if args.no_e2e else run_e2e(bank, n_layers, seq, pool, out, stream, args, flops, dev)

    single = None if (args.no_e2e or args.batch <= 1) else run_single_calls(pool, stream, args, dev, flops)
    sustained = None if (args.no_e2e or args.steps >= 1000) else run_sustained(pool, stream, args, dev, flops, local)
    planner = None if args.no_e2e else run_planner(stream, args, dev)
    packed = None if args.no_e2e else run_packed(stream, args, dev)
    schedule = None if args.no_e2e else run_schedule(pool, stream, args, dev)
    configs = None
    if not args.no_e2e:
        try:
            configs = run_configs(stream, args, dev)
        except Exception as exc:  # an extra measurement must not lose the line
            configs = {"error": f"{type(exc).__name__}: {exc}"}
    baselines = None if args.no_e2e else run_baselines(pool, stream, args, dev, flops)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(budget_s=args.cpu_budget)
    bank.close()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded AR(1) unit-RMS Q/K, N(0,1) V)",
            "config": bench_config(world, n_streams, args.batch),
            "pct_bf16_peak": round(100 * value / peaks[bf16_key], 2),
            "pct_bf16_datasheet": round(100 * value / DATASHEET_BF16_TFLOPS, 2),
            "chunk_steps_per_s": round(1000.0 / (ms_step * LAYERS_PER_CHUNK_STEP) * world, 3),
            "kernel_ms_per_call": {"rope_publish": round(pub_ms, 4), "attention": round(attn_ms, 4),
                          "combine": round(comb_ms, 4)},
            "roofline": roofline, "roofline_publish": roofline_publish,
            "e2e": e2e, "sustained": sustained, "single_call": single, "planner": planner, "packed": packed, "schedule": schedule, "configs_14b": configs, "cache_update_baselines": baselines, "gpu_launches": kt.launches, "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def run_single_calls(pool, stream, args, dev, flops):
    """The headline's steady calls issued one ff_render_attn at a time (no
    wavefront batching): each call splits its query blocks' key ranges to fill
    the SMs and merges them with the combine kernel."""
    import torch

    from kv_cache_attention_ff_gb300 import ff
    T, H, D = 1560, 12, 128
    n = max(8, min(args.steps, 400))
    warm = 4
    layers = max(1, math.ceil((n + warm) / 88))
    sb = ff.Bank(n_layers=layers, n_stages=4, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=9,
                 total_frames=81, heads=H, head_dim=D, frame_h=30, frame_w=52, device=dev.index)
    z = torch.zeros((3 * T, H, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(z)
    for layer in range(layers):
        for b in range(3):
            sb.anchor_publish(layer, 30 * b, 3, z, z, stream)
        for st in range(4):
            for i in range(5):
                sb.render_attn(layer, st, i, *pool[st][i % 4], out, stream)
    calls = [(l, st, i) for i in range(5, 27) for l in range(layers) for st in range(4)][:n + warm]
    for l, st, i in calls[:warm]:
        sb.render_attn(l, st, i, *pool[st][i % 4], out, stream)
    torch.cuda.synchronize()
    sb.set_timing(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gate(stream)
    e0.record(stream)
    for l, st, i in calls[warm:]:
        q, k, v = pool[st][i % 4]
        rc = sb.render_attn_raw(l, st, i, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"ff_render_attn failed with status {rc}")
    e1.record(stream)
    torch.cuda.synchronize()
    kt = sb.read_timing()
    sb.set_timing(False)
    assert sb.error_poll() == 0
    sb.close()
    ms = e0.elapsed_time(e1) / n
    c = max(kt.calls, 1)
    return {"workload": "the headline's steady calls, one ff_render_attn each", "calls": n,
            "ms_per_call": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
            "kernel_ms": {"rope_publish": round(kt.publish_ms / c, 4), "attention": round(kt.attn_ms / c, 4),
                          "combine": round(kt.combine_ms / c, 4)}, "launches": kt.launches}


def run_sustained(pool, stream, args, dev, flops, local):
    """The headline's calls for about a second (1760 calls in batches of
    --batch, 20 layers x 4 stages x 22 steady chunks), long enough for the 1.4 kW
    power cap to settle the clocks, with the clocks sampled inside the window:
    reported beside a short headline run, whose window sees full clocks."""
    import torch

    from kv_cache_attention_ff_gb300 import ff
    T, H, D = 1560, 12, 128
    layers = 20
    sb = ff.Bank(n_layers=layers, n_stages=4, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=9,
                 total_frames=81, heads=H, head_dim=D, frame_h=30, frame_w=52, planner_history=0, device=dev.index)
    z = torch.zeros((3 * T, H, D), dtype=torch.bfloat16, device=dev)
    outs = [torch.empty_like(z) for _ in range(4)]
    for layer in range(layers):
        for b in range(3):
            sb.anchor_publish(layer, 30 * b, 3, z, z, stream)
        for st in range(4):
            for i in range(5):
                sb.render_attn(layer, st, i, *pool[st][i % 4], outs[st], stream)
    calls = [(l, st, i) for i in range(5, 27) for l in range(layers) for st in range(4)]
    B = max(1, args.batch)
    torch.cuda.synchronize()
    sampler = ClockSampler(local, args.clock_ms)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    gate(stream)
    e0.record(stream)
    for j0 in range(0, len(calls), B):
        group = []
        for l, st, i in calls[j0:j0 + B]:
            q, k, v = pool[st][i % 4]
            group.append((l, st, i, q.data_ptr(), k.data_ptr(), v.data_ptr(), outs[st].data_ptr()))
        rc = (sb.render_attn_batch_raw(group, stream.cuda_stream) if B > 1 else
              sb.render_attn_raw(*group[0], stream.cuda_stream))
        if rc != 0:
            raise RuntimeError(f"renderer call failed with status {rc}")
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(wall0, time.time())
    clocks = sampler.stop()
    assert sb.error_poll() == 0
    sb.close()
    ms = e0.elapsed_time(e1) / len(calls)
    return {"workload": "the headline's steady calls for about a second (power-capped clocks)", "calls": len(calls),
            "calls_per_launch": B, "ms_per_step": round(ms, 4), "value": round(flops / (ms * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "clocks": clocks}


def run_planner(stream, args, dev):
    """Planner-role attention at the W_ctx-wide block: 261 latents of the 1.3B 480p
    shape, block 8 over the clean KV of blocks 2..7 plus itself (21 frames)."""
    import torch

    from kv_cache_attention_ff_gb300 import ff, synth
    T, H, D = 1560, 12, 128
    pb = ff.Bank(n_layers=1, n_stages=1, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=27,
                 total_frames=261, heads=H, head_dim=D, frame_h=30, frame_w=52, planner_block=3, planner_history=6,
                 device=dev.index)
    with torch.cuda.stream(stream):
        ka = synth.device_frames(6, 0, synth.ANCHOR_STREAM, synth.K, list(range(60, 240, 10)), T, H, D, "ar",
                                 device=dev)
        va = synth.device_frames(6, 0, synth.ANCHOR_STREAM, synth.V, list(range(60, 240, 10)), T, H, D, "normal",
                                 device=dev)
        q, k, v = (synth.device_frames(6, 0, 51, t, [240, 250, 260], T, H, D, "ar" if t < 2 else "normal",
                                       device=dev) for t in range(3))
    torch.cuda.synchronize()
    pb.anchor_publish(0, 60, 18, ka, va, stream)
    out = torch.empty_like(q)
    for _ in range(args.warmup):
        pb.planner_attn(0, 8, q, k, v, out, stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        pb.planner_attn(0, 8, q, k, v, out, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    assert pb.error_poll() == 0
    pb.close()
    flops = 4.0 * 4680 * 21 * T * D * H
    return {"workload": "planner block, 1.3B 480p shape, 21 context frames (W_ctx)", "queries": 4680,
            "keys": 21 * T, "ms_per_call": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}


def run_baselines(pool, stream, args, dev, flops):
    """Attention cost of one chunk-step (one layer) under FlashForward's schedule and
    the cache-update-only schedules of Self-Forcing and HiAR, every call a steady
    1.3B 480p ff_render_attn.  One GPU, attention only: context for the pages'
    end-to-end multi-GPU speed-ups, not a reproduction of them."""
    import torch

    from kv_cache_attention_ff_gb300 import ff, schedules
    T, H, D = 1560, 12, 128
    S = 4
    bb = ff.Bank(n_layers=1, n_stages=2 * S, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=9,
                 total_frames=81, heads=H, head_dim=D, frame_h=30, frame_w=52, planner_history=0, device=dev.index)
    z = torch.zeros((3 * T, H, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(z)
    for b in range(3):
        bb.anchor_publish(0, 30 * b, 3, z, z, stream)
    # bank slot of a call: denoise stage k -> bank k, re-encode k -> bank S + k
    nxt = [0] * (2 * S)

    def call(kind, k):
        bank_stage = k if kind == "denoise" else S + (k % S)
        i = nxt[bank_stage]
        q, kk, v = pool[k % S][i % 4]
        rc = bb.render_attn_raw(0, bank_stage, i, q.data_ptr(), kk.data_ptr(), v.data_ptr(), out.data_ptr(),
                                stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"ff_render_attn failed with status {rc}")
        nxt[bank_stage] += 1

    # ramp every bank to steady state (5 chunks of history)
    for st in range(2 * S):
        for _ in range(5):
            call("denoise" if st < S else "reencode", st)
    res = {}
    chunks = 4
    for name, fn in schedules.SCHEDULES.items():
        sched = fn(S)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(chunks):
            for kind, k in sched:
                call(kind, k)
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = {"calls_per_chunk_step": len(sched),
                     "cache_update_only_calls": schedules.cache_update_only_calls(sched),
                     "ms_per_chunk_step_per_layer": round(e0.elapsed_time(e1) / chunks, 4)}
    assert bb.error_poll() == 0
    bb.close()
    base = res["flashforward"]["ms_per_chunk_step_per_layer"]
    for name in ("self_forcing", "hiar"):
        res[name]["time_vs_flashforward"] = round(res[name]["ms_per_chunk_step_per_layer"] / base, 3)
    res["note"] = ("attention calls only, one layer, one GPU, S=4 stages; the pages report 1.42-2.92x vs "
                   "Self-Forcing and 1.16-1.69x vs HiAR end to end with up to 4 GPUs")
    return res


def run_schedule(pool, stream, args, dev):
    """The full 81-latent schedule of the 1.3B 480p shape on one GPU: anchors
    published first (3 planner blocks of 3 per layer), then 27 chunks x 4 stages
    x 30 layers of renderer calls in stage-wavefront order: at step w, every
    layer renders chunk w - k at stage k (the pages' wavefront on one GPU),
    ramp-up and drain steps included; with --batch > 1 the calls of one layer
    at one step go out as one ff_render_attn_batch.  Inputs cycle the pool
    (time does not depend on values)."""
    import torch

    from kv_cache_attention_ff_gb300 import ff, synth
    T, H, D, L, N = 1560, 12, 128, 30, 81
    sb = ff.Bank(n_layers=L, n_stages=4, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=9,
                 total_frames=N, heads=H, head_dim=D, frame_h=30, frame_w=52, device=dev.index)
    with torch.cuda.stream(stream):
        ka = synth.device_frames(2, 0, synth.ANCHOR_STREAM, synth.K, list(range(0, N, 10)), T, H, D, "ar", device=dev)
        va = synth.device_frames(2, 0, synth.ANCHOR_STREAM, synth.V, list(range(0, N, 10)), T, H, D, "normal",
                                 device=dev)
        blocks = [(ka[3 * b * T:3 * (b + 1) * T].contiguous(), va[3 * b * T:3 * (b + 1) * T].contiguous())
                  for b in range(3)]
        out = torch.empty((3 * T, H, D), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    e0.record(stream)
    for layer in range(L):
        for b in range(3):
            sb.anchor_publish(layer, 30 * b, 3, blocks[b][0], blocks[b][1], stream)
    e1.record(stream)
    outs = [torch.empty((3 * T, H, D), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    for w in range(27 + 3):
        step = [(st, w - st) for st in range(4) if 0 <= w - st < 27]
        for layer in range(L):
            calls = [(layer, st, i, *pool[st][i % 4], outs[st]) for st, i in step]
            if args.batch > 1:
                sb.render_attn_batch(calls, stream)
            else:
                for c in calls:
                    sb.render_attn(*c, stream)
    e2.record(stream)
    torch.cuda.synchronize()
    assert sb.error_poll() == 0
    key_frames = 0
    for i in range(27):
        key_frames += len(sb.gamma(i)) + 3 * min(i, 5) + 3
    sb.close()
    render_s = e1.elapsed_time(e2) / 1e3
    flops = 4.0 * (3 * T) * (key_frames * T) * D * H * 4 * L
    return {"workload": "1.3B 480p full schedule: 27 chunks x 4 stages x 30 layers in stage-wavefront order, "
                        "anchors published first", "calls_per_launch": args.batch,
            "renderer_calls": 27 * 4 * L, "key_frames_per_layer_stage": key_frames,
            "anchor_publish_ms": round(e0.elapsed_time(e1), 3), "render_ms": round(1e3 * render_s, 2),
            "chunk_steps_per_s": round(27 * 4 / render_s, 2), "tflops": round(flops / render_s / 1e12, 1)}


def run_configs(stream, args, dev):
    """Steady renderer calls of the 14B shapes (40 heads, d 128): 480p (4680 queries
    over 31200 keys) and the 720p long rollout (10800 queries over 72000 keys, 261
    latents, 6 anchor slots filled on demand).  One layer and one stage: a call's
    work does not depend on them.  The timed chunks are steady chunks whose anchors
    all stay resident (720p: chunks 8..16, anchor blocks 0 and 1 in the 6-slot
    ring)."""
    import torch

    from kv_cache_attention_ff_gb300 import ff, synth
    res = {}
    for name, cfg_id, fh, fw, N, cap, reps in (("wan14b_480p", 4, 30, 52, 81, 9, 18),
                                               ("wan14b_720p", 5, 45, 80, 261, 6, 9)):
        T, H, D = fh * fw, 40, 128
        cb = ff.Bank(n_layers=1, n_stages=1, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=cap,
                     total_frames=N, heads=H, head_dim=D, frame_h=fh, frame_w=fw, device=dev.index)
        with torch.cuda.stream(stream):
            q, k = (synth.device_frames(cfg_id, 0, 0, t, [0, 1, 2], T, H, D, "ar", device=dev) for t in (0, 1))
            v = synth.device_frames(cfg_id, 0, 0, 2, [0, 1, 2], T, H, D, "normal", device=dev)
            out = torch.empty_like(q)
        published = set()

        def publish_for(i):
            for a in cb.gamma(i):
                blk = a // 30
                if blk in published:
                    continue
                frames = [f for f in (30 * blk, 30 * blk + 10, 30 * blk + 20) if f < N]
                with torch.cuda.stream(stream):
                    ak = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.K, frames, T, H, D, "ar", device=dev)
                    av = synth.device_frames(cfg_id, 0, synth.ANCHOR_STREAM, synth.V, frames, T, H, D, "normal",
                                             device=dev)
                cb.anchor_publish(0, 30 * blk, len(frames), ak, av, stream)
                published.add(blk)

        first = 5 + 3  # ramp-up chunks 0..4 and 3 warm-up calls untimed
        for i in range(first):
            publish_for(i)
            cb.render_attn(0, 0, i, q, k, v, out, stream)
        for i in range(first, first + reps):  # anchors of the timed chunks, before timing
            publish_for(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(first, first + reps):
            cb.render_attn(0, 0, i, q, k, v, out, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        assert cb.error_poll() == 0
        key_frames = [len(cb.gamma(i)) + 15 + 3 for i in range(first, first + reps)]
        cb.close()
        ms = e0.elapsed_time(e1) / reps
        flops = sum(4.0 * (3 * T) * (kf * T) * D * H for kf in key_frames) / reps
        res[name] = {"queries": 3 * T, "keys": key_frames[0] * T, "heads": H, "calls": reps,
                     "tflop_per_call": round(flops / 1e12, 3), "ms_per_call": round(ms, 3),
                     "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
    return res


def run_packed(stream, args, dev):
    """Packed block-causal renderer forward of one stage of the 81-latent 1.3B 480p
    clip: 27 chunks of 4680 queries over 5..20 key frames each, one call."""
    import torch

    from kv_cache_attention_ff_gb300 import ff, synth
    T, H, D, N = 1560, 12, 128, 81
    pb = ff.Bank(n_layers=1, n_stages=1, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=9,
                 total_frames=N, heads=H, head_dim=D, frame_h=30, frame_w=52, planner_history=0, device=dev.index)
    with torch.cuda.stream(stream):
        q, k = (synth.device_frames(2, 0, 0, t, list(range(N)), T, H, D, "ar", device=dev) for t in (0, 1))
        v = synth.device_frames(2, 0, 0, 2, list(range(N)), T, H, D, "normal", device=dev)
        ak = synth.device_frames(2, 0, synth.ANCHOR_STREAM, synth.K, list(range(0, 81, 10)), T, H, D, "ar", device=dev)
        av = synth.device_frames(2, 0, synth.ANCHOR_STREAM, synth.V, list(range(0, 81, 10)), T, H, D, "normal",
                                 device=dev)
        ws = torch.empty(pb.packed_workspace_bytes(), dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
    torch.cuda.synchronize()
    reps = max(3, min(50, args.steps // 4))
    for _ in range(2):
        pb.packed_render_attn(q, k, v, ak, av, out, ws, stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        pb.packed_render_attn(q, k, v, ak, av, out, ws, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    assert pb.error_poll() == 0
    pb.close()
    key_frames = sum(min(20, 5 + 3 * i) for i in range(27))  # 495
    flops = 4.0 * (3 * T) * (key_frames * T) * D * H
    return {"workload": "packed block-causal forward, one stage of the 81-latent 1.3B 480p clip",
            "chunks": 27, "key_frames_total": key_frames, "ms_per_call": round(ms, 3),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}


def run_e2e(bank, n_layers, seq, pool, out, stream, args, flops, dev):
    """Same calls through the public API with host buffers.  Every step copies
    its q, k, v from pinned host memory to the device and its output back to
    pinned host memory inside the timed region.  Calls are issued like the
    device-timed region (one ff_render_attn per call, or stage-wavefront
    batches of --batch calls); copies run on their own streams with
    double-buffered device staging per group of calls, so the next group's
    upload and the previous group's download overlap a group's kernels."""
    import torch

    from kv_cache_attention_ff_gb300 import ff
    T, H, D = 1560, 12, 128
    nq = 3 * T
    B = max(1, args.batch)
    host_in = [[t.cpu().pin_memory() for t in pool[s][0]] for s in range(4)]
    host_out = [[torch.empty((nq, H, D), dtype=torch.bfloat16).pin_memory() for _ in range(B)] for _ in range(2)]
    dbuf = [[[torch.empty((nq, H, D), dtype=torch.bfloat16, device=dev) for _ in range(3)] for _ in range(B)]
            for _ in range(2)]
    dout = [[torch.empty((nq, H, D), dtype=torch.bfloat16, device=dev) for _ in range(B)] for _ in range(2)]
    steps, warm = args.steps, args.warmup
    layers = max(1, math.ceil((steps + warm) / 88))
    eb = ff.Bank(n_layers=layers, n_stages=4, history=5, chunk_frames=3, anchor_stride=10, anchor_capacity=9,
                 total_frames=81, heads=H, head_dim=D, frame_h=30, frame_w=52, device=dev.index)
    z = torch.zeros((3 * T, H, D), dtype=torch.bfloat16, device=dev)
    for layer in range(layers):
        for b in range(3):
            eb.anchor_publish(layer, 30 * b, 3, z, z, stream)
        for st in range(4):
            for i in range(5):
                q, k, v = pool[st][i % 4]
                eb.render_attn(layer, st, i, q, k, v, out, stream)
    nxt = {(l, s): 5 for l in range(layers) for s in range(4)}
    order = [(l, s) for l in range(layers) for s in range(4)]
    calls = []
    while len(calls) < steps + warm:
        for key in order:
            if nxt[key] < 27 and len(calls) < steps + warm:
                calls.append((key[0], key[1], nxt[key]))
                nxt[key] += 1
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    uploaded = [ev(), ev()]
    computed = [ev(), ev()]
    downloaded = [ev(), ev()]
    started = [False, False]
    groups = [(j, min(warm, j + B)) for j in range(0, warm, B)]
    groups += [(j, min(warm + steps, j + B)) for j in range(warm, warm + steps, B)]

    def group(g, j0, j1):
        b = g & 1
        if started[b]:
            up.wait_event(computed[b])          # staging set b is free once group g-2 ran
        with torch.cuda.stream(up):
            for slot, j in enumerate(range(j0, j1)):
                for dst, src in zip(dbuf[b][slot], host_in[calls[j][1]]):
                    dst.copy_(src, non_blocking=True)
            uploaded[b].record(up)
        stream.wait_event(uploaded[b])
        if started[b]:
            stream.wait_event(downloaded[b])    # output set b was read back
        args_list = []
        for slot, j in enumerate(range(j0, j1)):
            layer, st, c = calls[j]
            dq, dk, dv = dbuf[b][slot]
            args_list.append((layer, st, c, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dout[b][slot].data_ptr()))
        if B == 1:
            rc = eb.render_attn_raw(*args_list[0], stream.cuda_stream)
        else:
            rc = eb.render_attn_batch_raw(args_list, stream.cuda_stream)
        if rc != 0:
            raise RuntimeError(f"renderer call failed with status {rc}")
        computed[b].record(stream)
        down.wait_event(computed[b])
        with torch.cuda.stream(down):
            for slot in range(j1 - j0):
                host_out[b][slot].copy_(dout[b][slot], non_blocking=True)
            downloaded[b].record(down)
        started[b] = True

    n_warm_groups = len([1 for j0, _ in groups if j0 < warm])
    for g in range(n_warm_groups):
        group(g, *groups[g])
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    gate(up)
    e0.record(up)
    for g in range(n_warm_groups, len(groups)):
        group(g, *groups[g])
    e1.record(down)  # every upload precedes its kernels, which precede the download on `down`
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    eb.close()
    bytes_in = 3 * nq * H * D * 2
    return {"value": round(flops * steps / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": bytes_in,
            "d2h_bytes_per_step": nq * H * D * 2, "ms_per_step": round(ms / steps, 4),
            "copies": "pinned host <-> device every step, double-buffered on two copy streams",
            "calls_per_launch": B}


# ----------------------------------------------------------------------------- CPU oracle

def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(rows: int, heads: int, seed: int = 0):
    """Time the fp64 oracle's attention on `rows` query rows x `heads` heads of the
    steady 1.3B call (31200 keys, d 128).  Returns (seconds, flops)."""
    import numpy as np

    from oracle import ff_oracle as fo
    rng = np.random.default_rng(seed)
    nk = 20 * 1560
    q = rng.standard_normal((rows, heads, 128))
    k = rng.standard_normal((nk, heads, 128))
    v = rng.standard_normal((nk, heads, 128))
    t0 = time.perf_counter()
    fo.attention_f64(q, k, v)
    dt = time.perf_counter() - t0
    return dt, 4.0 * rows * nk * 128 * heads


def cpu_baseline(budget_s: float = 15.0):
    # calibrate on a small sample, then size the timed sample (rows x heads) to about budget_s
    dt0, f0 = oracle_sample(512, 1)
    rate = f0 / max(dt0, 1e-6)
    per_head = 4.0 * 4680 * 31200 * 128
    heads = int(min(12, max(1, budget_s * rate // per_head)))
    rows = 4680 if heads > 1 else int(min(4680, max(128, budget_s * rate / (4.0 * 31200 * 128))))
    dt, fl = oracle_sample(rows, heads, seed=1)
    rate = fl / dt
    tiny_s, tiny_fl = oracle_tiny_bruteforce()
    return {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": _host_cores(), "kind": "oracle",
            "sample": f"fp64 numpy oracle attention of {rows} query rows x {heads} heads over the 31200 keys of "
                      f"the steady 1.3B call ({fl / 1e9:.1f} GFLOP, {dt:.1f} s); rope/publish/gather not included",
            "cpu_count": os.cpu_count(), "affinity": _host_cores(), "blas_threads": _blas_threads(),
            "chunk_steps_per_s": round(rate / (30 * 4.0 * 4680 * 31200 * 128 * 12), 6),
            "tiny_bruteforce": {"seconds": round(tiny_s, 3), "gflops": round(tiny_fl / tiny_s / 1e9, 6), "cores": 1,
                                "sample": "pure-Python attention of the tiny schedule's chunk 2 "
                                          "(48 queries x 176 keys x 2 heads, d 64)"}}


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return f"{var}={os.environ[var]}"
    return "library default (threadpoolctl unavailable)"


def oracle_tiny_bruteforce():
    """Time the oracle's pure-Python attention on one call of the tiny schedule
    (chunk 2: 48 queries over 176 keys, 2 heads, d 64) on one core."""
    import numpy as np

    from oracle import ff_oracle as fo
    rng = np.random.default_rng(3)
    q = rng.standard_normal((48, 2, 64)).tolist()
    k = rng.standard_normal((176, 2, 64)).tolist()
    v = rng.standard_normal((176, 2, 64)).tolist()
    t0 = time.perf_counter()
    fo.attention_bruteforce(q, k, v)
    return time.perf_counter() - t0, 4.0 * 48 * 176 * 64 * 2


def run_reference(args):
    """The oracle arm: fp64 numpy attention of the steady 1.3B call on the host
    cores.  Every step is a bounded sample of that call (all 12 heads, the
    first R query rows over all 31200 keys), R sized so that the warm-up and
    timed steps take about three minutes together."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    dt0, f0 = oracle_sample(64, 12)
    rate = f0 / max(dt0, 1e-6)
    per_step_s = max(0.05, 180.0 / max(args.steps + args.warmup, 1))
    per_row = 4.0 * 31200 * 128 * 12
    rows = int(min(4680, max(16, per_step_s * rate / per_row)))
    times, fl = [], 0.0
    for j in range(args.warmup + args.steps):
        dt, fl = oracle_sample(rows, 12, seed=j)
        if j >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = fl * len(times) / total / 1e12
    cores = _host_cores()
    sample = (f"fp64 numpy oracle attention per step: {rows} of the 4680 query rows x 12 heads x 31200 keys "
              f"({fl / 1e9:.2f} GFLOP/step) of the steady 1.3B call; rope/publish not included")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * total / len(times), 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(world, max(1, min(4, args.stage_streams)), args.batch),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample, "blas_threads": _blas_threads()},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-ms", type=int, default=50, help="nvidia-smi sampling interval during the timed region")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass (profiling runs)")
    ap.add_argument("--stage-streams", type=int, default=1,
                    help="CUDA streams the 4 stages are issued on (1..4); per-kernel event times need 1")
    ap.add_argument("--batch", type=int, default=4,
                    help="calls per ff_render_attn_batch (1 = one ff_render_attn per step; 2..4 = stage wavefront "
                         "batches of consecutive calls, which have distinct stages)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if not 1 <= args.batch <= 4 or (args.batch > 1 and args.stage_streams > 1):
        ap.error("--batch must be 1..4 (and with one stream)")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
