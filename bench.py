"""Benchmark of the paged-KV hot path on GB300.

One step = one pass of the whole path over one batch: staged block-table diffs
+ gather (pa_apply_staged_writes), KV write of the step's tokens
(pa_write_kv), attention (pa_forward). Workload: the 256-request decode batch
of a 7B-like layer (32/32 heads, D 128, B 16, contexts U[128, 2048]); the
metric is KV bytes the step's attention must read per second (GB/s), whole
job over all GPUs (replicas: every rank runs its own batch).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl libpa|reference]

--impl reference times the CPU oracle (fp64, all host cores) on the same
256-request step and prints the same line with "impl": "reference". The GPU
line also carries, for the headline batch and for every secondary workload
(tiny decode, mixed chunked prefill, long context bf16 / E4M3, prefix-shared
sampling), the oracle's time for that workload's whole step on the host
cores: measured whole where that takes about ten seconds or less, else
measured on a stated uniform sample of output rows and scaled by visible
(row, key) pairs (oracle_baseline).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn decode KV GB/s vs HBM peak; mixed-batch tokens/s (1×GB300)"
UNIT = "GB/s"
CONFIG_ID = 2


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def combine_ranks(times, units, world, device):
    """Whole-job view of a replicated step: every time is the slowest rank's
    (max over ranks) and the work is what all ranks processed together (sum
    over ranks; each rank runs its own seeded batch, so the ranks' units
    differ). world == 1 returns the inputs."""
    times = [float(x) for x in times]
    if world == 1:
        return times, float(units)
    import torch
    import torch.distributed as dist
    t = torch.tensor(times, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.cpu()], float(u.cpu()[0])


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def traffic_for(kernel: str, src_files):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[kernel]
    except Exception:
        return None
    h = hashlib.sha256()
    for p in src_files:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return t["bytes_per_launch"] if t.get("src_sha256") == h.hexdigest() else None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed
    region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.proc = None
        self.uuid = uuid

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.uuid:
            cmd[1:1] = ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4)
                          if r[i].lower() in ("active", "0x1") or r[i] == "1"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ GPU arm

class Step:
    """Device buffers of one step and the three C-ABI calls of the hot path."""

    def __init__(self, w, dev, max_splits=32):
        import torch
        from paged_kv_cache_143_gb300 import pa
        from workloads.generate import NAN_BF16, NAN_E4M3
        self.w, self.pa = w, pa
        shape = w.pool_shape()
        if w.kv_dtype == "bf16":
            k = torch.full(shape, NAN_BF16, dtype=torch.int16, device=dev).view(torch.bfloat16)
            v = torch.full(shape, NAN_BF16, dtype=torch.int16, device=dev).view(torch.bfloat16)
        else:
            k = torch.full(shape, NAN_E4M3, dtype=torch.uint8, device=dev)
            v = torch.full(shape, NAN_E4M3, dtype=torch.uint8, device=dev)
        self.pool = pa.KVPool(k, v, w.k_scale, w.v_scale)
        if w.ctx_slots.numel():  # the cache before the step
            pa.write_kv(self.pool, w.ctx_k, w.ctx_v, w.ctx_slots.to(dev))
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
        self.table = i32(w.table_before)
        self.rows, self.starts = i32(w.diff_rows), i32(w.diff_starts)
        self.offs, self.vals = i32(w.diff_val_offsets), i32(w.diff_vals)
        self.idx = i32(w.idx_mapping)
        self.gathered = torch.empty((w.R, w.max_blocks), dtype=torch.int32, device=dev)
        self.qsl, self.seq = i32(w.qsl), i32(w.seq_lens)
        self.q = w.q.to(dev).contiguous()
        self.new_k, self.new_v = w.new_k.to(dev).contiguous(), w.new_v.to(dev).contiguous()
        self.slots = w.slot_mapping.to(dev)
        self.out = torch.empty_like(self.q)
        n = pa.forward_workspace_size(w.R, w.Hq, w.D, max_splits)
        self.ws = torch.empty(n, dtype=torch.uint8, device=dev) if n else None

    def run(self, cascade=False):
        pa, w = self.pa, self.w
        pa.apply_staged_writes(self.table, self.rows, self.starts, self.offs, self.vals,
                               self.idx, self.gathered)
        pa.write_kv(self.pool, self.new_k, self.new_v, self.slots)
        self.forward(cascade)

    def forward(self, cascade=False):
        pa, w = self.pa, self.w
        if cascade:  # groups of consecutive requests sharing their prompt blocks
            first = [min(m) for m in w.groups]
            size = [len(m) for m in w.groups]
            prefix_blocks = [p // w.B for p in w.group_prefix]
            pa.forward_shared_prefix(self.q, self.out, self.qsl, self.seq, w.qsl, w.seq_lens,
                                     self.gathered, self.pool, w.scale, first, size,
                                     prefix_blocks, causal=w.causal, workspace=self.ws)
        else:
            pa.forward(self.q, self.out, self.qsl, self.seq, w.qsl, w.seq_lens, self.gathered,
                       self.pool, w.scale, w.causal, workspace=self.ws)


def run_libpa(args):
    import torch
    import torch.distributed as dist

    import workloads
    from paged_kv_cache_143_gb300 import accounting, pa

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    w = workloads.make(CONFIG_ID, device=dev, sub=rank, num_requests=args.requests)
    kv_bytes = accounting.decode_kv_bytes(w.seq_lens, w.Hkv, w.D, w.elt_bytes)

    step = Step(w, dev, max_splits=32)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step.run()
    if pa.get_error() != pa.PA_OK:
        raise RuntimeError("device error during warm-up")

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = pa.kernel_launches()
    t0.record(stream)
    for i in range(args.steps):
        pa.apply_staged_writes(step.table, step.rows, step.starts, step.offs, step.vals,
                               step.idx, step.gathered)
        pa.write_kv(step.pool, step.new_k, step.new_v, step.slots)
        ev[i][0].record(stream)
        pa.forward(step.q, step.out, step.qsl, step.seq, w.qsl, w.seq_lens, step.gathered,
                   step.pool, w.scale, w.causal, workspace=step.ws)
        ev[i][1].record(stream)
    t1.record(stream)
    launches = pa.kernel_launches() - launches0
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    if pa.get_error() != pa.PA_OK:
        raise RuntimeError("device error in the timed region")
    ms = t0.elapsed_time(t1) / args.steps
    fwd_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    (ms, fwd_ms), total_kv = combine_ranks((ms, fwd_ms), kv_bytes, world, dev)

    # ---- end to end through the C ABI with host buffers (pinned), copies inside
    e2e = run_e2e(args, w, step, dev, kv_bytes, world)
    # the oracle beside it, on the host cores (rank 0 of a one-GPU run only)
    args.cpu_legs = args.cpu_legs and world == 1 and rank == 0
    cpu = cpu_baseline(w, kv_bytes) if args.cpu_legs else None

    peak, peak_kind = load_peaks()
    achieved = total_kv / world / (fwd_ms * 1e-3) / 1e9  # per GPU
    line = {
        "metric": METRIC, "value": round(total_kv / (ms * 1e-3) / 1e9, 2),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"decode-7b-like: {w.R} requests x 1 token, 32/32 heads, "
                               f"head_dim 128, block 16, contexts U[128,2048] "
                               f"({int(w.seq_lens.sum())} keys), bf16 KV",
                   "kv_bytes_per_step": kv_bytes, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (KV read per step >> 129 MB)",
                   "step": "pa_apply_staged_writes + pa_write_kv + pa_forward"},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"hbm_gbs ({peak_kind})",
                     "kernel": "decode split-KV (pa_forward on a decode-only batch)",
                     "ms_per_launch": round(fwd_ms, 5),
                     "traffic": traffic_for("decode_kernel", [
                         "paged_kv_cache_143_gb300/csrc/decode.cu",
                         "paged_kv_cache_143_gb300/csrc/decode_rows.cuh",
                         "paged_kv_cache_143_gb300/csrc/pa_device.cuh"])},
        "e2e": e2e,
        "clocks": clk,
    }
    del step
    torch.cuda.empty_cache()
    line["mixed_batch"] = run_mixed(args, dev, 3)
    line["long_context"] = {"bf16": run_mixed(args, dev, 5, "bf16"),
                            "fp8": run_mixed(args, dev, 5, "fp8")}
    line["prefix_shared"] = run_prefix_shared(args, dev)
    line["tiny_decode"] = run_tiny(args, dev)
    line["serving"] = run_serving(args, dev)
    if rank == 0:
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def timed(fn, steps, warmup, stream):
    """Mean ms of fn() over `steps` calls after `warmup`, CUDA events on `stream`."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def timed_flushed(fn, steps, warmup, stream):
    """Mean ms of fn() over `steps` calls after `warmup`, each call timed alone
    by CUDA events on `stream` after a 512 MB write that evicts L2 (for
    workloads whose inputs fit in the 129 MB L2)."""
    import torch
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=torch.cuda.current_device())
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush.fill_(1)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / steps


def run_decode(args, dev):
    """The decode batch of the benchmark line alone, one whole step (staged
    diffs, KV write, forward) per iteration: a narrow command for profiler
    captures (no e2e leg, no secondary workloads, no clock sampling)."""
    import torch

    import workloads
    from paged_kv_cache_143_gb300 import accounting, pa

    w = workloads.make(CONFIG_ID, device=dev, num_requests=args.requests)
    kv = accounting.decode_kv_bytes(w.seq_lens, w.Hkv, w.D, w.elt_bytes)
    step = Step(w, dev, max_splits=32)
    ms = timed(step.run, args.steps, args.warmup, torch.cuda.current_stream())
    if pa.get_error() != pa.PA_OK:
        raise RuntimeError("device error in the decode batch")
    return {"workload": f"decode-7b-like: {w.R} requests x 1 token", "kv_bytes": kv,
            "ms_per_step": round(ms, 5), "gbs": round(kv / (ms * 1e-3) / 1e9, 1)}


def run_mixed(args, dev, cfg, kv_dtype=None):
    """Mixed decode + prefill step of config `cfg` (tokens/s of the whole step),
    and the prefill kernel alone on the same chunks (causal TFLOP/s)."""
    import torch
    import workloads
    from paged_kv_cache_143_gb300 import accounting, pa
    stream = torch.cuda.current_stream()
    n_req = getattr(args, "long_requests", None) if cfg == 5 else None
    w = workloads.make(cfg, device=dev, kv_dtype=kv_dtype, num_requests=n_req)
    step = Step(w, dev, max_splits=32)
    ms = timed(step.run, args.steps, args.warmup, stream)
    if pa.get_error() != pa.PA_OK:
        raise RuntimeError("device error in the mixed step")
    ql = np.diff(w.qsl)
    chunks = np.nonzero(ql > 1)[0]
    pairs = sum(accounting.causal_pairs(int(ql[r]), int(w.seq_lens[r])) for r in chunks)
    flops = accounting.attention_flops(pairs, w.Hq, w.D)
    dec = np.nonzero(ql == 1)[0]
    dec_bytes = accounting.decode_kv_bytes(w.seq_lens[dec], w.Hkv, w.D, w.elt_bytes)
    # the chunks alone: only the prefill kernel runs in pa_forward
    wp = workloads.build(w.seq_lens[chunks], ql[chunks], w.Hq, w.Hkv, w.D, w.B,
                         kv_dtype=w.kv_dtype, seed=workloads.config_seed(cfg, 1), device=dev)
    sp = Step(wp, dev, max_splits=32)
    sp.run()
    fwd = lambda: pa.forward(sp.q, sp.out, sp.qsl, sp.seq, wp.qsl, wp.seq_lens, sp.gathered,
                             sp.pool, wp.scale, wp.causal, workspace=sp.ws)
    ms_pre = timed(fwd, args.steps, args.warmup, stream)
    # the decodes alone
    wd = workloads.build(w.seq_lens[dec], ql[dec], w.Hq, w.Hkv, w.D, w.B, kv_dtype=w.kv_dtype,
                         seed=workloads.config_seed(cfg, 2), device=dev)
    sd = Step(wd, dev, max_splits=32)
    sd.run()
    fwd_d = lambda: pa.forward(sd.q, sd.out, sd.qsl, sd.seq, wd.qsl, wd.seq_lens, sd.gathered,
                               sd.pool, wd.scale, wd.causal, workspace=sd.ws)
    ms_dec = timed(fwd_d, args.steps, args.warmup, stream)
    if pa.get_error() != pa.PA_OK:
        raise RuntimeError("device error in the split runs")
    peak_t = load_peaks_tensor()
    peak_h, peak_kind = load_peaks()
    tf = flops / (ms_pre * 1e-3) / 1e12
    gbs_dec = dec_bytes / (ms_dec * 1e-3) / 1e9
    del step, sp, sd
    torch.cuda.empty_cache()
    cpu = None
    if getattr(args, "cpu_legs", False):
        cpu = oracle_baseline(w, seed=cfg)
        cpu.update({"value": round(w.T / cpu["seconds_per_step"], 2), "unit": "tokens/s"})
    return {"cpu_baseline": cpu,
        "workload": w.name, "tokens_per_step": int(w.T), "ms_per_step": round(ms, 4),
        "tokens_per_s": round(w.T / (ms * 1e-3), 1),
        "step": "pa_apply_staged_writes + pa_write_kv + pa_forward (decodes and chunks)",
        "prefill_only": {"ms": round(ms_pre, 4), "causal_flops": int(flops),
                         "tflops": round(tf, 1),
                         "roofline": {"bound": "tensor", "achieved": round(tf, 1),
                                      "peak": peak_t, "unit": "TFLOP/s",
                                      "frac": round(tf / peak_t, 4),
                                      "peak_source": "bf16_tflops (measured, burst)"}},
        **({"prefill_e4m3_peak": {
            "peak": round(peak_t * 2 / 2.5, 1), "unit": "TFLOP/s",
            "frac": round(tf / (peak_t * 2 / 2.5), 4),
            "how": "the MMA work of an E4M3 pool's chunk: S as three E4M3 products "
                   "(query split in three terms) at twice the bf16 rate, 1.5 bf16 S "
                   "equivalents, plus P.V on f16 operands: 2.5 units against bf16's 2, "
                   "so the measured bf16 peak x 2 / 2.5"}} if w.kv_dtype == "fp8" else {}),
        "decode_only": {"ms": round(ms_dec, 4), "kv_bytes": int(dec_bytes),
                        "gbs": round(dec_bytes / (ms_dec * 1e-3) / 1e9, 1),
                        "roofline": {"bound": "hbm", "achieved": round(gbs_dec, 1),
                                     "peak": peak_h, "unit": "GB/s",
                                     "frac": round(gbs_dec / peak_h, 4),
                                     "peak_source": f"hbm_gbs ({peak_kind})"}},
    }


def run_prefill_only(args, dev, cfg, kv_dtype=None, n_chunks=None):
    """The prefill chunks of config `cfg` alone (the first n_chunks of them):
    pa_forward on the chunks' step, causal TFLOP/s (a narrow command for
    profiler captures of the tensor-core prefill kernel)."""
    import torch
    import workloads
    from paged_kv_cache_143_gb300 import accounting, pa
    w = workloads.make(cfg, device=dev, kv_dtype=kv_dtype)
    ql = np.diff(w.qsl)
    chunks = np.nonzero(ql > 1)[0][:n_chunks]
    seq, name = w.seq_lens[chunks], w.name
    Hq, Hkv, D, B, kvd = w.Hq, w.Hkv, w.D, w.B, w.kv_dtype
    pairs = sum(accounting.causal_pairs(int(ql[r]), int(w.seq_lens[r])) for r in chunks)
    flops = accounting.attention_flops(pairs, Hq, D)
    del w
    torch.cuda.empty_cache()
    wp = workloads.build(seq, ql[chunks], Hq, Hkv, D, B, kv_dtype=kvd,
                         seed=workloads.config_seed(cfg, 1), device=dev)
    sp = Step(wp, dev, max_splits=32)
    sp.run()
    fwd = lambda: pa.forward(sp.q, sp.out, sp.qsl, sp.seq, wp.qsl, wp.seq_lens, sp.gathered,
                             sp.pool, wp.scale, wp.causal, workspace=sp.ws)
    ms = timed(fwd, args.steps, args.warmup, torch.cuda.current_stream())
    if pa.get_error() != pa.PA_OK:
        raise RuntimeError("device error in the prefill chunks")
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": f"{name} prefill chunks x{len(chunks)}", "ms": round(ms, 4),
            "causal_flops": int(flops), "tflops": round(tf, 1),
            "frac": round(tf / load_peaks_tensor(), 4)}


def run_prefix_shared(args, dev):
    """Prefix-shared parallel sampling (8 groups x 16 samples, FP8 KV): decode
    step time, logical KV bytes (what every request reads) and unique KV bytes
    (shared prompt blocks counted once); through pa_forward (every request
    reads its whole context) and through pa_forward_shared_prefix (each
    group's prompt read once)."""
    import torch
    import workloads
    from paged_kv_cache_143_gb300 import accounting, pa
    stream = torch.cuda.current_stream()
    w = workloads.make(4, device=dev)
    step = Step(w, dev, max_splits=32)
    logical = accounting.decode_kv_bytes(w.seq_lens, w.Hkv, w.D, w.elt_bytes)
    unique = accounting.unique_kv_bytes(w.tables, w.seq_lens, w.B, w.Hkv, w.D, w.elt_bytes)
    peak, _ = load_peaks()
    res = {"workload": w.name, "logical_kv_bytes": int(logical), "unique_kv_bytes": int(unique)}
    res["l2"] = "flushed before every timed call (unique KV < 129 MB)"
    for key, cascade in (("pa_forward", False), ("shared_prefix", True)):
        ms = timed_flushed(lambda: step.run(cascade), args.steps, args.warmup, stream)
        ms_fwd = timed_flushed(lambda: step.forward(cascade), args.steps, args.warmup, stream)
        if pa.get_error() != pa.PA_OK:
            raise RuntimeError("device error in the prefix-shared step")
        res[key] = {"ms_per_step": round(ms, 4), "forward_ms": round(ms_fwd, 4),
                    "effective_gbs": round(logical / (ms_fwd * 1e-3) / 1e9, 1),
                    "unique_gbs": round(unique / (ms_fwd * 1e-3) / 1e9, 1),
                    "unique_frac_of_hbm": round(unique / (ms_fwd * 1e-3) / 1e9 / peak, 4)}
    del step
    torch.cuda.empty_cache()
    if getattr(args, "cpu_legs", False):
        cpu = oracle_baseline(w, seed=4)
        cpu.update({"value": round(logical / cpu["seconds_per_step"] / 1e9, 4),
                    "unit": "GB/s (logical KV bytes)"})
        res["cpu_baseline"] = cpu
    return res


def run_tiny(args, dev, graph_steps=8):
    """The tiny decode batch (4 requests): latency of one step, in
    microseconds, issued call by call, and the same decode steps replayed
    `graph_steps` at a time from one CUDA graph (pa_decode_graph_*)."""
    import torch
    import workloads
    from paged_kv_cache_143_gb300 import pa
    stream = torch.cuda.current_stream()
    w = workloads.make(1, device=dev)
    step = Step(w, dev, max_splits=8)
    us = timed(step.run, max(args.steps, 20), args.warmup, stream) * 1e3
    # the same requests with graph_steps decode steps ahead (same shapes, seed)
    N = graph_steps
    ctx = [int(x) - 1 for x in w.seq_lens]
    wg = workloads.build([c + N for c in ctx], [N] * w.R, w.Hq, w.Hkv, w.D, w.B,
                         pool_blocks=w.num_blocks, seed=w.seed, device=dev)
    sg = Step(wg, dev, max_splits=8)
    pa.apply_staged_writes(sg.table, sg.rows, sg.starts, sg.offs, sg.vals, sg.idx, sg.gathered)
    nc0 = torch.zeros(wg.max_reqs, dtype=torch.int32, device=dev)
    nc0[sg.idx.long()] = torch.tensor(ctx, dtype=torch.int32, device=dev)
    nc = nc0.clone()
    per_step = lambda t: t.view(wg.R, N, *t.shape[1:]).transpose(0, 1).contiguous()
    q, k, v = per_step(sg.q), per_step(sg.new_k), per_step(sg.new_v)
    out = torch.empty_like(q)
    g = pa.DecodeGraph(sg.pool, wg.scale, nc, sg.table, sg.idx, sg.gathered,
                       [c + N for c in ctx], q, k, v, out, workspace=sg.ws)

    def replay():
        nc.copy_(nc0)  # every launch starts from the same slot state
        g.launch()
    us_graph = timed(replay, max(args.steps, 20), args.warmup, stream) * 1e3 / N
    if pa.get_error() != pa.PA_OK:
        raise RuntimeError("device error in the tiny decode runs")
    kernels = g.kernels
    g.close()
    cpu = None
    if getattr(args, "cpu_legs", False):
        cpu = oracle_baseline(w, budget_s=2.0, seed=1)
        cpu.update({"value": round(cpu["seconds_per_step"] * 1e6, 2), "unit": "us per step"})
    return {"workload": w.name, "us_per_step": round(us, 2), "cpu_baseline": cpu,
            "graph": {"steps_per_launch": N, "us_per_step": round(us_graph, 2),
                      "kernels_per_launch": kernels,
                      "step": "pa_prepare_inputs + pa_write_kv + pa_forward, captured"}}


def run_serving(args, dev, steps=30):
    """Multi-step serving loop (native scheduler + device calls, engine.py)
    on a stream shaped like the mixed chunked-prefill step: 64 long-running
    requests (prompts U[1024, 4096]) decoding while prompts of U[1024, 8192]
    tokens arrive, 32/8 heads, head_dim 128, block 16, budget 4096 tokens,
    chunk cap 2048. Whole-loop tokens/s (host scheduling, one pinned upload,
    the device calls and the read-back of each entry's last output row, per
    step), KV waste and preemptions from the scheduler's block statistics."""
    import time
    import torch
    from paged_kv_cache_143_gb300 import pa
    from paged_kv_cache_143_gb300.engine import Engine
    Hq, Hkv, D, B, NB = 32, 8, 128, 16, 40000
    max_reqs, max_blocks, max_tokens = 256, 1024, 4096
    rng = np.random.default_rng(143300)
    k_pool = torch.zeros((NB, Hkv, B, D), dtype=torch.bfloat16, device=dev)
    v_pool = torch.zeros_like(k_pool)
    pool = pa.KVPool(k_pool, v_pool)
    sched = pa.Scheduler(NB, B, max_reqs, max_blocks, token_budget=4096, chunk_cap=2048)
    eng = Engine(sched, pool, Hq, max_reqs, max_blocks, max_tokens, scale=D ** -0.5,
                 device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(143300)
    q = torch.randn((max_tokens, Hq, D), generator=gen, device=dev).bfloat16()
    k = torch.randn((max_tokens, Hkv, D), generator=gen, device=dev).bfloat16()
    v = torch.randn((max_tokens, Hkv, D), generator=gen, device=dev).bfloat16()
    out = torch.empty_like(q)
    rid = 0
    for _ in range(64):
        sched.add_request(rid, rng.integers(0, 32000, size=int(rng.integers(1024, 4097))), 4000)
        rid += 1

    def one_step():
        nonlocal rid
        if rng.random() < 0.35:
            sched.add_request(rid, rng.integers(0, 32000, size=int(rng.integers(1024, 8193))),
                              int(rng.integers(16, 256)))
            rid += 1
        b = eng.step(q, k, v, out)
        eng.sync()
        sched.commit(rng.integers(0, 32000, size=b.num_reqs))
        return b
    # warm-up: until the 64 long requests decode
    for _ in range(200):
        if one_step().num_decode >= 64:
            break
    for _ in range(3):
        one_step()
    if pa.get_error() != pa.PA_OK:
        raise RuntimeError("device error in the serving warm-up")
    st0 = sched.stats()
    h2d0, d2h0 = eng.h2d_bytes, eng.d2h_bytes
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    toks = dec = 0
    for _ in range(steps):
        b = one_step()
        toks += b.num_tokens
        dec += b.num_decode
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    if pa.get_error() != pa.PA_OK:
        raise RuntimeError("device error in the serving loop")
    st = sched.stats()
    used_slots = st["used_blocks"] * B
    return {"workload": "serving loop, mixed-chunked-prefill-like stream",
            "steps": steps, "tokens_per_s": round(toks / dt, 1),
            "ms_per_step": round(dt * 1e3 / steps, 4),
            "tokens_per_step": round(toks / steps, 1), "decodes_per_step": round(dec / steps, 1),
            "h2d_bytes_per_step": int((eng.h2d_bytes - h2d0) / steps),
            "d2h_bytes_per_step": int((eng.d2h_bytes - d2h0) / steps),
            "kv_waste_frac": round(st["wasted_slots"] / max(used_slots, 1), 5),
            "kv_used_blocks": st["used_blocks"], "preemptions": st["preemptions"] -
            st0["preemptions"],
            "step": "pa_sched_step + one pinned upload + pa_apply_staged_writes x2 + "
                    "pa_copy_blocks + pa_prepare_inputs + pa_write_kv + pa_forward + "
                    "pa_gather_rows + read-back"}


def load_peaks_tensor():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def run_e2e(args, w, step, dev, kv_bytes, world):
    """Same metric with the step's inputs copied from pinned host memory and the
    output read back, inside the timed region, through the public C ABI."""
    import torch
    from paged_kv_cache_143_gb300 import pa

    def pinned(t):
        return t.detach().cpu().contiguous().pin_memory()
    host_in = {
        "q": pinned(w.q), "new_k": pinned(w.new_k), "new_v": pinned(w.new_v),
        "slots": pinned(w.slot_mapping),
        "rows": pinned(torch.from_numpy(w.diff_rows)),
        "starts": pinned(torch.from_numpy(w.diff_starts)),
        "offs": pinned(torch.from_numpy(w.diff_val_offsets)),
        "vals": pinned(torch.from_numpy(w.diff_vals if w.diff_vals.size else
                                        np.zeros(1, np.int32))),
        "idx": pinned(torch.from_numpy(w.idx_mapping)),
        "qsl": pinned(torch.from_numpy(w.qsl)), "seq": pinned(torch.from_numpy(w.seq_lens)),
    }
    dev_in = {k: torch.empty_like(v, device=dev) for k, v in host_in.items()}
    out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = out_host.numel() * out_host.element_size()
    stream = torch.cuda.current_stream()

    def one():
        for k, v in host_in.items():
            dev_in[k].copy_(v, non_blocking=True)
        d = dev_in
        pa.apply_staged_writes(step.table, d["rows"][:w.diff_rows.size],
                               d["starts"][:w.diff_starts.size], d["offs"], d["vals"],
                               d["idx"], step.gathered)
        pa.write_kv(step.pool, d["new_k"], d["new_v"], d["slots"])
        pa.forward(d["q"], step.out, d["qsl"], d["seq"], w.qsl, w.seq_lens, step.gathered,
                   step.pool, w.scale, w.causal, workspace=step.ws)
        out_host.copy_(step.out, non_blocking=True)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        one()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    (ms,), total_kv = combine_ranks((ms,), kv_bytes, world, dev)
    return {"value": round(total_kv / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h)}


# ------------------------------------------------------------- oracle arms

CPU_SAMPLE_SECONDS = 10.0  # oracle seconds per workload (about; whole configs may take less)


def visible_pairs(w):
    """Visible (query row, key) pairs of every output row, token-major
    [T * Hq]: the oracle's work per row is proportional to them."""
    per_tok = np.zeros(int(w.T), np.int64)
    for r in range(w.R):
        a, b = int(w.qsl[r]), int(w.qsl[r + 1])
        if b == a:
            continue
        seq = int(w.seq_lens[r])
        P = seq - (b - a)
        per_tok[a:b] = P + 1 + np.arange(b - a) if (w.causal and b - a > 1) else seq
    return np.repeat(per_tok, w.Hq)


class OracleStep:
    """The oracle's copy of one step's inputs (prepared outside any timing)
    and one timed pass: staged diffs + gather, KV write, attention over all
    output rows or a subset."""

    def __init__(self, w):
        from tests.helpers import bits, oracle_pool
        self.w = w
        self.pool = oracle_pool(w, include_new=False)
        self.k_new, self.v_new = bits(w.new_k), bits(w.new_v)
        self.slots, self.q = w.slot_mapping.cpu().numpy(), bits(w.q)

    def run(self, rows=None):
        from oracle import oracle as O
        w = self.w
        table = w.table_before.copy()
        t = time.perf_counter()
        gathered = O.apply_staged_writes(table, w.diff_rows, w.diff_starts, w.diff_val_offsets,
                                         w.diff_vals, w.idx_mapping)
        O.write_kv(self.pool, self.k_new, self.v_new, self.slots)
        O.paged_attention(self.q, w.qsl, w.seq_lens, gathered, self.pool, w.scale, w.causal,
                          rows=rows)
        return time.perf_counter() - t


def oracle_baseline(w, budget_s=CPU_SAMPLE_SECONDS, seed=0):
    """Times the fp64 C oracle on the host cores on workload `w`: the whole
    step if it fits in about `budget_s` seconds, else a uniform random sample
    of output rows (token, head) sized to the budget. For a sample, the step's
    fixed part (staged diffs + KV write, timed with a one-row attention) is
    kept and the attention part is scaled by visible (row, key) pairs, to
    which the oracle's work per row is proportional. Returns the seconds of
    one whole step and a description of what ran."""
    from oracle import oracle as O
    st = OracleStep(w)
    pairs = visible_pairs(w)
    total = int(pairs.sum())
    rng = np.random.default_rng(143000 + seed)
    one = np.zeros(1, np.int64)
    t_fixed = min(st.run(one) for _ in range(3))
    # calibration: about two million pairs' worth of rows
    n_cal = int(min(pairs.size, max(64, 2_000_000 * pairs.size // max(total, 1))))
    cal = np.sort(rng.choice(pairs.size, size=n_cal, replace=False)) if n_cal < pairs.size else None
    t_cal = st.run(cal)
    cal_pairs = int(pairs[cal].sum()) if cal is not None else total
    rate = cal_pairs / max(t_cal - t_fixed, 1e-9)  # attention pairs per second
    frac = min(1.0, max(budget_s - t_fixed, 0.1) * rate / max(total, 1))
    if frac >= 0.999 or cal is None:
        rows, sample_pairs = None, total
    else:
        n = max(1, int(pairs.size * frac))
        rows = np.sort(rng.choice(pairs.size, size=n, replace=False))
        sample_pairs = int(pairs[rows].sum())
    secs = []
    while not secs or (rows is None and sum(secs) < budget_s and len(secs) < 50):
        secs.append(st.run(rows))
    s_sample = sum(secs) / len(secs)
    if rows is None:
        whole = s_sample
        what = f"the whole step, {len(secs)} run(s)"
    else:
        whole = t_fixed + max(s_sample - t_fixed, 0.0) * total / sample_pairs
        what = (f"{rows.size} of {pairs.size} output rows (token x head) drawn uniformly, "
                f"{sample_pairs} of {total} visible (row, key) pairs; whole-step time = "
                f"fixed part ({t_fixed:.4f} s: diffs, KV write) + attention part scaled by "
                f"pairs")
    return {"seconds_per_step": round(whole, 5), "measured_seconds": round(s_sample, 5),
            "sampled": rows is not None, "cores": O.max_threads(), "kind": "oracle",
            "sample": f"fp64 C oracle (staged diffs + KV write + attention) on {what}"}


def cpu_baseline(w, kv_bytes):
    """The oracle beside the headline decode batch: KV GB/s of the whole step."""
    b = oracle_baseline(w)
    b.update({"value": round(kv_bytes / b["seconds_per_step"] / 1e9, 4), "unit": UNIT})
    return b


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import workloads
    from oracle import oracle as O
    from paged_kv_cache_143_gb300 import accounting
    w = workloads.make(CONFIG_ID, device="cpu", num_requests=args.requests)
    kv = accounting.decode_kv_bytes(w.seq_lens, w.Hkv, w.D, w.elt_bytes)
    st = OracleStep(w)
    for _ in range(args.warmup):
        st.run()
    secs = [st.run() for _ in range(args.steps)]
    s = sum(secs) / len(secs)
    value = round(kv / s / 1e9, 4)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(s * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": f"decode-7b-like: {w.R} requests x 1 token, 32/32 heads, "
                               f"head_dim 128, block 16, contexts U[128,2048] "
                               f"({int(w.seq_lens.sum())} keys), bf16 KV",
                   "kv_bytes_per_step": kv,
                   "step": "staged diffs + KV write + attention, fp64 C oracle"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": O.max_threads(),
                         "kind": "oracle",
                         "sample": f"the whole {w.R}-request step, {args.steps} timed steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["libpa", "reference"], default="libpa")
    ap.add_argument("--requests", type=int, default=256,
                    help="decode batch size (256 is the benchmark workload; smaller sizes "
                         "are for profiling captures)")
    ap.add_argument("--long-requests", type=int, default=None,
                    help="long-context legs: requests of 32768 tokens (32 is the benchmark "
                         "workload; fewer are for profiling captures)")
    ap.add_argument("--no-cpu", dest="cpu_legs", action="store_false",
                    help="skip the oracle timings on the host cores (profiling runs)")
    ap.add_argument("--chunks", type=int, default=None,
                    help="prefill-long: how many of the long-context prefill chunks to run")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="prefill-long: KV cache element type")
    ap.add_argument("--only", choices=["decode", "mixed", "long-bf16", "long-fp8",
                                       "prefill-long", "prefix-shared", "tiny", "serving"],
                    default=None,
                    help="run one workload alone (the benchmark's decode batch or a "
                         "secondary workload) and print its object (a narrow command for "
                         "profiler captures; not the benchmark line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.only:
        args.cpu_legs = False
        import torch
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        run = {"decode": lambda: run_decode(args, dev),
               "mixed": lambda: run_mixed(args, dev, 3),
               "long-bf16": lambda: run_mixed(args, dev, 5, "bf16"),
               "long-fp8": lambda: run_mixed(args, dev, 5, "fp8"),
               "prefill-long": lambda: run_prefill_only(args, dev, 5, args.kv, args.chunks),
               "prefix-shared": lambda: run_prefix_shared(args, dev),
               "tiny": lambda: run_tiny(args, dev),
               "serving": lambda: run_serving(args, dev)}[args.only]
        print(json.dumps({"only": args.only, "result": run()}), flush=True)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_libpa(args)


if __name__ == "__main__":
    main()
