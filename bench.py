"""Benchmark: fused attention forward on GB300 (prefill + split-K decode).

One step = one pass of the whole path over one batch of synthetic input:
  * dense non-causal prefill, B=1, H=16, d=128, bf16 in/out, fp32 accumulate,
    scale = 1/sqrt(128), at N = 4096, 8192 and 16384 (one launch each);
  * ragged split-K decode, B=32, H=14, d=64, fp16, KV caches [32,14,4096,64],
    seq_lens uniform on [1, 4096], scale = 1/8 (split kernel + merge kernel).
`value` is prefill TFLOP/s (4*B*H*N^2*d FLOPs per launch) over the device time
of the prefill launches; decode GB/s (K+V bytes of the visible cache rows)
is reported beside it.  L2 is flushed (a 2 x L2 buffer is written) before
every timed kernel, outside its CUDA-event pair.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs the same step on its own GPU with its
own seed (no data-path collective: weak scaling); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "prefill TFLOP/s (% BF16 TC peak) d=128 N=4K–16K; decode HBM GB/s (% peak)"
PREFILL_B, PREFILL_H, PREFILL_D = 1, 16, 128
PREFILL_NS = (4096, 8192, 16384)
DECODE_B, DECODE_H, DECODE_L, DECODE_D = 32, 14, 4096, 64
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture, valid only for the kernel source it was taken on: the first 16 hex
# digits of the sha256 of the listed source files, in order.
NCU_TRAFFIC = {
    # one prefill_kernel<128> launch of each of the step's problems (B=1, H=16,
    # d=128, bf16): --set full at N=8192, the two DRAM counters alone at 4096 and
    # 16384 (one pass each, on the full-size problem).
    "prefill": {"src": ["fa_prefill_sm103.cu", "fa_tiles.cuh", "sm103_ptx.cuh"],
                "src_sha": "e952fd9eb477dd27",
                "bytes_per_launch": {"4096": 50.46e6, "8192": 114.69e6, "16384": 253.71e6}},
    # one decode_split_kernel<64> launch of the step's decode problem (B=32, H=14)
    "decode": {"src": ["fa_decode_sm103.cu", "sm103_ptx.cuh"], "src_sha": "9066595177c6f87f",
               "bytes_per_launch": 263.58e6},
}


def prefill_flops(B, H, N, d, causal=False):
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def decode_bytes(lens, H, d):
    return 2.0 * H * float(sum(int(x) for x in lens)) * d * 2  # K and V rows, 16-bit


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def src_sha(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "attention_forward_prefill_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ ranks
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_seconds: float, local_units: float, world: int, device=None):
    """Max elapsed time and summed work over ranks (both via all_reduce)."""
    if world == 1:
        return local_seconds, local_units
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    u = torch.tensor([local_units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ our path
# configuration ids of the seeded generator (seed = 0xFA000000 + 16 * config + tensor)
CFG_TINY, CFG_GPT2, CFG_LONG, CFG_DECODE, CFG_STRESS = 0, 1, 2, 3, 4
GEN_THREADS = max(1, min(32, os.cpu_count() or 1))


def gen_tensor(torch, device, shape, cfg, tensor, dtype, rank=0, extra=0):
    """The repository's seeded N(0,1) generator (SplitMix64, Box-Muller, RNE to
    16 bits), drawn on the host threads and copied to the device.  Ranks and
    extra problems of a config get their own streams."""
    from attention_forward_prefill_gb300 import inputs as fin
    seed = fin.seed_for(cfg, tensor) + (rank << 40) + (extra << 48)
    bits = fin.normal_bits(shape, seed, "bf16" if dtype == torch.bfloat16 else "f16",
                           threads=GEN_THREADS)
    import numpy as np
    return torch.from_numpy(bits.view(np.int16)).view(dtype).to(device)


def make_inputs(torch, device, rank):
    """Seeded synthetic inputs of the timed step (per rank), on the device."""
    from attention_forward_prefill_gb300 import inputs as fin
    pre = {}
    for N in PREFILL_NS:
        shape = (PREFILL_B, PREFILL_H, N, PREFILL_D)
        pre[N] = [gen_tensor(torch, device, shape, CFG_LONG, t, torch.bfloat16, rank, N)
                  for t in (fin.TENSOR_Q, fin.TENSOR_K, fin.TENSOR_V)]
    shp = (DECODE_B, DECODE_H, DECODE_L, DECODE_D)
    dq = gen_tensor(torch, device, (DECODE_B, DECODE_H, 1, DECODE_D), CFG_DECODE, fin.TENSOR_Q,
                    torch.float16, rank)
    dk = gen_tensor(torch, device, shp, CFG_DECODE, fin.TENSOR_K, torch.float16, rank)
    dv = gen_tensor(torch, device, shp, CFG_DECODE, fin.TENSOR_V, torch.float16, rank)
    lens_np = fin.seq_lens(fin.seed_for(CFG_DECODE, fin.TENSOR_SEQLEN) + rank, DECODE_B, DECODE_L)
    lens = torch.from_numpy(lens_np).to(device)
    return pre, (dq, dk, dv, lens, lens_np)


def run_ours(args):
    import torch

    from attention_forward_prefill_gb300 import binding
    from attention_forward_prefill_gb300 import build as fa_build
    from attention_forward_prefill_gb300 import inputs as fin

    world, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    if rank == 0 or not os.path.exists(fa_build.LIB_PATH):
        fa_build.build()
    if world > 1:
        dist.barrier()
    binding.load()
    scale_p = float(1.0 / math.sqrt(PREFILL_D))
    scale_d = 0.125
    pre, (dq, dk, dv, lens, lens_np) = make_inputs(torch, device, rank)
    outs = {N: torch.empty_like(pre[N][0]) for N in PREFILL_NS}
    dout = torch.empty_like(dq)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    splits = binding.fa_decode_choose_splits(DECODE_B, DECODE_H, DECODE_L, -1)
    ws = torch.empty(binding.fa_decode_workspace_bytes(DECODE_B, DECODE_H, DECODE_L, DECODE_D,
                                                       splits), dtype=torch.uint8, device=device)
    cases = args.case.split(",") if args.case else None
    do_pre = [N for N in PREFILL_NS if cases is None or f"prefill:{N}" in cases]
    do_dec = cases is None or "decode" in cases
    # Extra problems, only when asked for (profiling and diagnostics; not part of
    # the headline): "shape:BxHxNxD[:causal]" is a forward prefill, "backward" the
    # backward of (1, 16, 4096, 128) and "backward:BxHxNxD[:causal]" any other;
    # fp16 at d = 64, bf16 at d = 128.  "decode:BxHqxHkv" is a decode over caches
    # of 4096 rows, d = 64, fp16, with the decode configs' ragged lengths for B
    # (grouped when Hkv < Hq), reported in GB/s of K/V rows read.
    extras = []
    for c in cases or []:
        kind, _, spec = c.partition(":")
        if kind == "backward" and not spec:
            spec = "1x16x4096x128"
        if kind == "decode" and spec:
            B, Hq, Hkv = (int(x) for x in spec.split("x"))
            xq = gen_tensor(torch, device, (B, Hq, 1, DECODE_D), CFG_DECODE, fin.TENSOR_Q, torch.float16,
                            rank, 1000 + len(extras))
            xk, xv = (gen_tensor(torch, device, (B, Hkv, DECODE_L, DECODE_D), CFG_DECODE, t, torch.float16,
                                 rank, 1000 + len(extras)) for t in (fin.TENSOR_K, fin.TENSOR_V))
            x_lens_np = fin.seq_lens(fin.seed_for(CFG_DECODE, fin.TENSOR_SEQLEN) + B, B, DECODE_L)
            x_lens = torch.from_numpy(x_lens_np).to(device)
            xo = torch.empty_like(xq)
            fn = (lambda xq=xq, xk=xk, xv=xv, x_lens=x_lens, xo=xo:
                  binding.decode(xq, xk, xv, x_lens, scale=0.125, out=xo))
            extras.append((c, fn, decode_bytes(x_lens_np, Hkv, DECODE_D), "GB/s"))
            continue
        if kind not in ("shape", "backward") or not spec:
            continue
        dims, _, flag = spec.partition(":")
        B, H, N, d = (int(x) for x in dims.split("x"))
        dt = torch.float16 if d == 64 else torch.bfloat16
        t = [gen_tensor(torch, device, (B, H, N, d), CFG_LONG, i, dt, rank, 1000 + len(extras))
             for i in range(4 if kind == "backward" else 3)]
        causal = flag == "causal"
        sc = 1.0 / math.sqrt(d)
        if kind == "backward":
            o, lse = binding.prefill_with_lse(t[0], t[1], t[2], causal=causal, scale=sc)
            fn = (lambda t=t, o=o, lse=lse, causal=causal, sc=sc:
                  binding.prefill_backward(t[0], t[1], t[2], o, t[3], lse, causal=causal, scale=sc))
            flops = 10.0 * B * H * N * N * d / (2 if causal else 1)
        else:
            o = torch.empty_like(t[0])
            fn = (lambda t=t, o=o, causal=causal, sc=sc:
                  binding.prefill(t[0], t[1], t[2], causal=causal, scale=sc, out=o))
            flops = prefill_flops(B, H, N, d, causal)
        extras.append((c, fn, flops, "TFLOP/s"))

    def step(record):
        ev = []
        for N in do_pre:
            q, k, v = pre[N]
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            binding.prefill(q, k, v, causal=False, scale=scale_p, out=outs[N])
            e1.record(stream)
            ev.append(("prefill", N, e0, e1))
        if do_dec:
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            binding.decode(dq, dk, dv, lens, scale=scale_d, num_splits=splits, workspace=ws,
                           out=dout)
            e1.record(stream)
            ev.append(("decode", 0, e0, e1))
        for name, fn, _, _ in extras:
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ev.append(("extra", name, e0, e1))
        if record is not None:
            record.append(ev)

    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()
    assert binding.fa_device_status(False) == 0

    sampler = ClockSampler(local) if not args.no_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    records = []
    t_start.record(stream)
    for _ in range(args.steps):
        step(records)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    step_ms = t_start.elapsed_time(t_end) / args.steps

    pre_ms = {N: [] for N in do_pre}
    dec_ms = []
    extra_ms = {name: [] for name, _, _, _ in extras}
    for ev in records:
        for kind, N, e0, e1 in ev:
            {"prefill": pre_ms.get(N), "decode": dec_ms, "extra": extra_ms.get(N)}[kind].append(
                e0.elapsed_time(e1))
    pre_time_s = sum(sum(v) for v in pre_ms.values()) / 1e3
    pre_flops = sum(prefill_flops(PREFILL_B, PREFILL_H, N, PREFILL_D) for N in do_pre) * args.steps
    dec_time_s = sum(dec_ms) / 1e3
    dec_bytes = decode_bytes(lens_np, DECODE_H, DECODE_D) * (args.steps if do_dec else 0)

    # ---- end to end through the public call with pinned host buffers: every
    # step copies its inputs in and its outputs back.  The three calls of a step
    # go on streams of their own (the call is stream-ordered, as in C), so one
    # call's copies can run under another's kernels; each step ends with a
    # device synchronisation, so steps do not overlap.
    e2e = None
    if not args.no_e2e and do_pre:
        host = {N: [x.cpu().pin_memory() for x in pre[N]] for N in do_pre}
        host_out = {N: torch.empty(outs[N].shape, dtype=outs[N].dtype, pin_memory=True) for N in do_pre}
        h2d = sum(x.numel() * x.element_size() for N in do_pre for x in host[N])
        d2h = sum(host_out[N].numel() * host_out[N].element_size() for N in do_pre)
        streams = {N: torch.cuda.Stream(device=device) for N in do_pre}

        def e2e_step():
            # the largest problem first: its copies in are the longest, and the
            # smaller problems' copies then run under its kernels
            for N in sorted(do_pre, reverse=True):
                with torch.cuda.stream(streams[N]):
                    binding.prefill(*host[N], causal=False, scale=scale_p, out=host_out[N], sync=False)
            torch.cuda.synchronize()

        e2e_step()  # warm the host path once
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        e2e_s = time.perf_counter() - t0
        e2e_s, e2e_flops = aggregate(e2e_s, pre_flops, world, device)
        e2e = {"value": e2e_flops / e2e_s / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    tot_s, tot_flops = aggregate(pre_time_s, pre_flops, world, device)
    _, tot_dec_bytes = aggregate(dec_time_s, dec_bytes, world, device)
    dec_s_max, _ = aggregate(dec_time_s, 0.0, world, device)
    step_ms_max, _ = aggregate(step_ms, 0.0, world, device)

    peaks, peak_src = load_peaks()
    configs = None
    if rank == 0 and not args.no_configs and not args.case:
        configs = measure_configs(torch, binding, device, stream, flush, peaks)
        assert binding.fa_device_status(False) == 0

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    value = tot_flops / tot_s / 1e12 if do_pre else None
    # our kernels per step: each prefill launch, plus its fixup pass when the
    # library's plan cuts units between CTAs; decode split + merge; backward
    # prep + dK/dV + dQ
    per_step = 0
    for N in do_pre:
        _, info, _ = binding.fa_prefill_plan(PREFILL_B, PREFILL_H, N, N, 0, 0, 0)
        per_step += 1 + (1 if info[0] and info[5] > 0 else 0)
    per_step += 2 if do_dec else 0
    for name, _, _, _ in extras:  # backward: prep + dK/dV + dQ; decode: split + merge
        if name.startswith("backward"):
            per_step += 3
        elif name.startswith("decode"):
            per_step += 2
        else:
            B, H, N, d = (int(x) for x in name.split(":")[1].split("x"))
            _, info, _ = binding.fa_prefill_plan(B, H, N, N, int(name.endswith(":causal")), 0, 0)
            per_step += 1 + (1 if info[0] and info[5] > 0 else 0)
    n_launch = per_step * args.steps
    detail = {}
    for N in do_pre:
        ms = statistics.median(pre_ms[N])
        tf = prefill_flops(PREFILL_B, PREFILL_H, N, PREFILL_D) / (ms / 1e3) / 1e12
        detail[f"prefill_N{N}"] = {"median_ms": round(ms, 4), "min_ms": round(min(pre_ms[N]), 4),
                                   "tflops": round(tf, 1)}
    traffic = None
    rec = NCU_TRAFFIC.get("prefill")
    if rec and rec.get("src_sha") == src_sha(rec["src"]) and do_pre:
        per = [rec["bytes_per_launch"].get(str(N)) for N in do_pre]
        if all(x is not None for x in per):
            traffic = sum(per) / len(per)
    line = {
        "metric": METRIC,
        "value": round(value, 2) if value is not None else None,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": ("dense non-causal prefill B=1 H=16 d=128 bf16 N=4096,8192,16384 "
                         "+ ragged split-K decode B=32 H=14 d=64 fp16 max_len=4096"),
            "prefill_shapes": [[PREFILL_B, PREFILL_H, N, PREFILL_D] for N in do_pre],
            "decode_shape": [DECODE_B, DECODE_H, DECODE_L, DECODE_D] if do_dec else None,
            "decode_splits": splits,
            "l2": "flushed before every timed kernel (2 x L2 buffer written, outside the events)",
            "ms_per_step_includes": "L2 flushes between kernels",
        },
        "roofline": {
            "bound": "tensor",
            "achieved": round(value, 2) if value is not None else None,
            "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": round(value / peaks["bf16_tflops"], 4) if value is not None else None,
            "traffic": traffic,
            "peak_source": f"{peak_src} bf16 dense burst (kernels timed alone)",
            "frac_of_sustained": (round(value / peaks["bf16_tflops_sustained"], 4)
                                  if value is not None else None),
            "kernel": "fa::prefill_kernel<128>",
        },
        "decode": None,
        "detail": detail,
        "configs": configs,
        "e2e": e2e,
        "gpu_launches": n_launch,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if do_dec:
        drec = NCU_TRAFFIC.get("decode")
        dec_traffic = (drec["bytes_per_launch"] if drec and drec["src_sha"] == src_sha(drec["src"])
                       else None)
        gbs = tot_dec_bytes / dec_s_max / 1e9
        line["decode"] = {
            "value": round(gbs, 1), "unit": "GB/s", "dtype": "f16",
            "median_us": round(statistics.median(dec_ms) * 1e3, 2),
            "kv_bytes_per_step": decode_bytes(lens_np, DECODE_H, DECODE_D),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": dec_traffic, "peak_source": f"{peak_src} copy bandwidth"},
        }
    if extras:
        line["extras"] = {}
        for name, _, amount, unit in extras:
            ms = statistics.median(extra_ms[name])
            key, scale = ("gbs", 1e9) if unit == "GB/s" else ("tflops", 1e12)
            line["extras"][name] = {"median_ms": round(ms, 4), key: round(amount / (ms / 1e3) / scale, 1)}
    if world > 1:
        dist.destroy_process_group()
    return line


# ------------------------------------------------------------------ every config
def time_kernel(torch, stream, flush, fn, reps):
    """Median and min device time (ms) of fn() over reps runs, L2 flushed before each."""
    ms = []
    for _ in range(reps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    return statistics.median(ms), min(ms)


def measure_configs(torch, binding, device, stream, flush, peaks, reps=7):
    """The other workloads of the target (tiny, GPT-2 shape, stress, every decode
    batch), timed one kernel at a time outside the main timed region."""
    import numpy as np

    from attention_forward_prefill_gb300 import inputs as fin
    res = {}
    n_extra = [100]

    def rnd(shape, dtype, cfg=7):
        # the seeded generator; every call draws its own stream
        n_extra[0] += 1
        return gen_tensor(torch, device, shape, cfg, 0, dtype, 0, n_extra[0])

    pre_cases = [("tiny", CFG_TINY, 1, 2, 128, 64, torch.float16, torch.float32, 0.125),
                 ("gpt2_b1", CFG_GPT2, 1, 12, 2048, 64, torch.float16, torch.float16, 0.125),
                 ("gpt2_b4", CFG_GPT2, 4, 12, 2048, 64, torch.float16, torch.float16, 0.125),
                 ("stress", CFG_STRESS, 8, 32, 8192, 128, torch.bfloat16, torch.bfloat16,
                  float(1.0 / math.sqrt(128)))]
    for name, cfg, B, H, N, d, dt, odt, scale in pre_cases:
        q, v = (gen_tensor(torch, device, (B, H, N, d), cfg, t, dt) for t in (fin.TENSOR_Q, fin.TENSOR_V))
        if name == "stress":
            # 1% of the key rows of every (b, h), chosen per head, x20 before rounding
            import numpy as np
            kb, _ = fin.keys_with_outliers((B, H, N, d), fin.seed_for(cfg, fin.TENSOR_K),
                                           fin.seed_for(cfg, fin.TENSOR_OUTLIER), "bf16",
                                           threads=GEN_THREADS)
            k = torch.from_numpy(kb.view(np.int16)).view(dt).to(device)
            del kb
        else:
            k = gen_tensor(torch, device, (B, H, N, d), cfg, fin.TENSOR_K, dt)
        out = torch.empty((B, H, N, d), dtype=odt, device=device)
        for causal in ((True,) if name == "stress" else (False, True)):
            def fn():
                binding.prefill(q, k, v, causal=causal, scale=scale, out=out, out_dtype=odt)
            fn()
            med, mn = time_kernel(torch, stream, flush, fn, reps)
            tf = prefill_flops(B, H, N, d, causal) / (med / 1e3) / 1e12
            res[f"{name}_{'causal' if causal else 'full'}"] = {
                "shape": [B, H, N, d], "median_us": round(med * 1e3, 2),
                "min_us": round(mn * 1e3, 2), "tflops": round(tf, 1),
                "frac_of_peak": round(tf / peaks["bf16_tflops"], 4)}
        del q, k, v, out
    # the general prefill forms: grouped heads, a prompt chunk over a longer
    # cache, and a packed batch of ragged sequences (FLOPs = 4 d per visible
    # (query, key) pair, counted exactly)
    def gen_case(name, q, k, v, fn, pairs, d, H):
        fn()
        med, mn = time_kernel(torch, stream, flush, fn, reps)
        tf = 4.0 * d * H * pairs / (med / 1e3) / 1e12
        res[name] = {"shape": [list(q.shape), list(k.shape)], "median_us": round(med * 1e3, 2),
                     "min_us": round(mn * 1e3, 2), "tflops": round(tf, 1),
                     "frac_of_peak": round(tf / peaks["bf16_tflops"], 4)}
    B, Hq, Hkv, N, d = 4, 14, 2, 4096, 64
    q = rnd((B, Hq, N, d), torch.float16)
    k, v = rnd((B, Hkv, N, d), torch.float16), rnd((B, Hkv, N, d), torch.float16)
    o = torch.empty_like(q)
    gen_case("gqa_prefill_b4_h14_kv2_causal", q, k, v,
             lambda: binding.prefill(q, k, v, causal=True, scale=0.125, out=o),
             B * N * (N + 1) / 2, d, Hq)
    Nq, Nk, H, d = 1024, 8192, 16, 128
    q = rnd((1, H, Nq, d), torch.bfloat16)
    k, v = rnd((1, H, Nk, d), torch.bfloat16), rnd((1, H, Nk, d), torch.bfloat16)
    o = torch.empty_like(q)
    gen_case("chunk_prefill_1024_over_8192_causal", q, k, v,
             lambda: binding.prefill(q, k, v, causal=True, scale=1 / math.sqrt(d), out=o),
             Nq * (Nk - Nq) + Nq * (Nq + 1) / 2, d, H)
    lens = fin.seq_lens(0xFA00F00D, 16, 4096)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(device)
    T, H, d = int(lens.sum()), 16, 128
    q = rnd((T, H, d), torch.bfloat16)
    k, v = rnd((T, H, d), torch.bfloat16), rnd((T, H, d), torch.bfloat16)
    o = torch.empty_like(q)
    mx = int(lens.max())
    gen_case("varlen_prefill_16seqs_causal", q, k, v,
             lambda: binding.prefill_varlen(q, k, v, cu, cu, mx, mx, causal=True,
                                            scale=1 / math.sqrt(d), out=o),
             float(sum(int(n) * (int(n) + 1) / 2 for n in lens)), d, H)
    del q, k, v, o
    # backward pass (training): dQ, dK, dV from the forward's output and
    # log-sum-exp; FLOPs counted as five N^2 d products (10 B H N^2 d, halved
    # for causal), the algorithmic count of a backward that recomputes S
    for name, B, H, N, d, dt, causal in [("backward_long_n8192_full", 1, 16, 8192, 128, torch.bfloat16, False),
                                         ("backward_long_n8192_causal", 1, 16, 8192, 128, torch.bfloat16, True),
                                         ("backward_gpt2_b4_causal", 4, 12, 2048, 64, torch.float16, True)]:
        q, k, v, do = (rnd((B, H, N, d), dt) for _ in range(4))
        out, lse = binding.prefill_with_lse(q, k, v, causal=causal, scale=1 / math.sqrt(d))

        def fn():
            binding.prefill_backward(q, k, v, out, do, lse, causal=causal, scale=1 / math.sqrt(d))
        fn()
        med, mn = time_kernel(torch, stream, flush, fn, reps)
        fl = 10.0 * B * H * N * N * d / (2 if causal else 1)
        tf = fl / (med / 1e3) / 1e12
        res[name] = {"shape": [B, H, N, d], "median_us": round(med * 1e3, 2), "min_us": round(mn * 1e3, 2),
                     "tflops": round(tf, 1), "frac_of_peak": round(tf / peaks["bf16_tflops"], 4)}
        del q, k, v, do, out, lse
    for B in (1, 8, 32):
        for H in (14, 12):
            shp = (B, H, DECODE_L, DECODE_D)
            dq = rnd((B, H, 1, DECODE_D), torch.float16)
            dk, dv = rnd(shp, torch.float16), rnd(shp, torch.float16)
            lens_np = fin.seq_lens(fin.seed_for(3, fin.TENSOR_SEQLEN) + B, B, DECODE_L)
            lens = torch.from_numpy(lens_np).to(device)
            out = torch.empty_like(dq)
            splits = binding.fa_decode_choose_splits(B, H, DECODE_L, -1)
            ws = torch.empty(binding.fa_decode_workspace_bytes(B, H, DECODE_L, DECODE_D, splits),
                             dtype=torch.uint8, device=device)

            def fn():
                binding.decode(dq, dk, dv, lens, scale=0.125, num_splits=splits, workspace=ws,
                               out=out)
            fn()
            med, mn = time_kernel(torch, stream, flush, fn, reps)
            gbs = decode_bytes(lens_np, H, DECODE_D) / (med / 1e3) / 1e9
            res[f"decode_b{B}_h{H}"] = {
                "shape": list(shp), "splits": splits, "median_us": round(med * 1e3, 2),
                "min_us": round(mn * 1e3, 2), "gbs": round(gbs, 1),
                "frac_of_peak": round(gbs / peaks["hbm_gbs"], 4)}
    # grouped decode, Qwen2.5-0.5B-like heads (14 query heads over 2 cache
    # heads): bytes are the K and V rows actually read (per cache head)
    for B in (8, 32):
        Hq, Hkv = 14, 2
        dq = rnd((B, Hq, 1, DECODE_D), torch.float16)
        dk = rnd((B, Hkv, DECODE_L, DECODE_D), torch.float16)
        dv = rnd((B, Hkv, DECODE_L, DECODE_D), torch.float16)
        lens_np = fin.seq_lens(fin.seed_for(3, fin.TENSOR_SEQLEN) + B, B, DECODE_L)
        lens = torch.from_numpy(lens_np).to(device)
        out = torch.empty_like(dq)
        splits = binding.fa_decode_gqa_choose_splits(B, Hq, Hkv, DECODE_L, -1)
        ws = torch.empty(binding.fa_decode_workspace_bytes(B, Hq, DECODE_L, DECODE_D, splits),
                         dtype=torch.uint8, device=device)

        def fn():
            binding.decode(dq, dk, dv, lens, scale=0.125, num_splits=splits, workspace=ws, out=out)
        fn()
        med, mn = time_kernel(torch, stream, flush, fn, reps)
        gbs = decode_bytes(lens_np, Hkv, DECODE_D) / (med / 1e3) / 1e9
        res[f"decode_gqa_b{B}_h{Hq}_kv{Hkv}"] = {
            "shape": [B, Hq, Hkv, DECODE_L, DECODE_D], "splits": splits,
            "median_us": round(med * 1e3, 2), "min_us": round(mn * 1e3, 2), "gbs": round(gbs, 1),
            "frac_of_peak": round(gbs / peaks["hbm_gbs"], 4)}
    # read-only streaming probe beside decode: the library's own kernel, with
    # the decode loads (16-byte, non-caching), over 4 GiB
    x = torch.ones(1 << 31, dtype=torch.float16, device=device)
    xo = torch.zeros(1, dtype=torch.int32, device=device)
    nbytes = x.numel() * 2

    def probe():
        rc = binding.fa_read_probe(x.data_ptr(), nbytes, xo.data_ptr(), stream.cuda_stream)
        assert rc == 0
    med, _ = time_kernel(torch, stream, flush, probe, reps)
    res["read_probe"] = {"what": "fa_read_probe over 4 GiB (16-byte non-caching loads, "
                                 "XOR checksum)", "gbs": round(nbytes / (med / 1e3) / 1e9, 1),
                         "frac_of_peak": round(nbytes / (med / 1e3) / 1e9 / peaks["hbm_gbs"], 4)}
    del x
    return res


# ------------------------------------------------------------------ oracle legs
def oracle_sample(seconds: float, N: int = 16384, threads: int = 1):
    """Time the fp64 oracle on whole rows of the N-length prefill (one head).

    threads > 1 spreads blocks of rows over host threads (the C routine runs
    outside the GIL), the row-parallel form of the same oracle.
    """
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    from attention_forward_prefill_gb300 import inputs as fin
    from oracle import oracle

    d = PREFILL_D
    rows_per_call = 8
    k = oracle.bf16_bits_to_f64(fin.normal_bits((N, d), fin.seed_for(2, 1), "bf16"))
    v = oracle.bf16_bits_to_f64(fin.normal_bits((N, d), fin.seed_for(2, 2), "bf16"))
    q = oracle.bf16_bits_to_f64(fin.normal_bits((N, d), fin.seed_for(2, 0), "bf16"))
    scale = float(np.float32(1.0 / math.sqrt(d)))
    oracle.attention(q, k, v, False, scale, rows=[0])  # load / build
    done = 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        while time.perf_counter() - t0 < seconds:
            blocks = [np.arange(done + i * rows_per_call, done + (i + 1) * rows_per_call) % N
                      for i in range(threads)]
            list(ex.map(lambda r: oracle.attention(q, k, v, False, scale, rows=r, threads=1),
                        blocks))
            done += rows_per_call * threads
    dt = time.perf_counter() - t0
    flops = 4.0 * N * d * done
    return flops / dt / 1e12, done, dt


def cpu_baseline(seconds: float):
    value, rows, dt = oracle_sample(seconds)
    cores = os.cpu_count() or 1
    par, prow, pdt = oracle_sample(max(2.0, seconds / 4), threads=cores)
    return {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": (f"{rows} query rows of one head of the N=16384 d=128 dense prefill "
                       f"({dt:.1f} s single-threaded fp64 C oracle); FLOPs counted as 4*N*d "
                       "per row"),
            "all_cores": {"value": par, "unit": "TFLOP/s", "cores": cores,
                          "sample": f"{prow} rows, row blocks over {cores} host threads, "
                                    f"{pdt:.1f} s"}}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    per_step = max(0.5, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        oracle_sample(min(0.5, per_step))
    vals, rows_total, t_total = [], 0, 0.0
    for _ in range(args.steps):
        v, rows, dt = oracle_sample(per_step)
        vals.append(v)
        rows_total += rows
        t_total += dt
    value = 4.0 * 16384 * PREFILL_D * rows_total / t_total / 1e12
    sample = (f"{rows_total} query rows of one head of the N=16384 d=128 dense prefill over "
              f"{args.steps} steps of ~{per_step:.1f} s (single-threaded fp64 C oracle)")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_total / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": ("dense non-causal prefill B=1 H=16 d=128 bf16 N=4096,8192,16384 "
                                "+ ragged split-K decode B=32 H=14 d=64 fp16 max_len=4096"),
                   "reference": "the fp64 CPU oracle, as it stands, on sampled rows"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--case", default="", help="subset, e.g. prefill:8192 or decode")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config table (tiny, GPT-2 shape, stress, decode batches)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours" and not args.case:
        ap.error("--warmup must be >= 3")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
