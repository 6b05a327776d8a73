#!/usr/bin/env python3
"""Benchmark of the MiniMax-H3 DiT block / 50-block denoiser step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on rank 0.  A "step" is one pass of the hot path over one batch
of seeded synthetic input; the headline workload is one full-width BF16 DiT
block at the 512x512x22-frame class (d 5120, 40 x 128 heads, MLP 20480,
N 6912 = 6x32x32 video + 512 text + 256 audio) and `value` is its throughput
in TFLOP/s (4 projections + 2 attention contractions per block).  The
50-block step latency at the 864x480 class (N 10488) with and without token
reduction is reported under "step".

Multi-GPU: the block does not shard (one request per GPU); N GPUs run N
independent replicas with no collective on the data path, launched by
torchrun, barrier + max-over-ranks timing, `value` = all ranks' FLOPs / time.

--impl reference times the fp64 CPU oracle (the deliberately slow
correctness baseline) on the host cores on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DiT block TFLOP/s (BF16/INT8) and 50-block step ms; % of tensor/HBM roofline"
WORKLOAD_DESC = ("block_512: one BF16 MiniMax-H3 DiT block, d=5120, 40x128 heads, MLP 20480 GELU-tanh, "
                 "N=6912 tokens (video 6x32x32 + 512 text + 256 audio), 3D RoPE, full attention")
CPU_SAMPLE_TOKENS = 1024


def block_flops(n, d, f):
    return 2.0 * n * d * (3 * d) + 2.0 * n * d * d + 4.0 * n * d * f + 4.0 * n * n * d


def gemm_flops(n, d, f):
    return 2.0 * n * d * (3 * d) + 2.0 * n * d * d + 4.0 * n * d * f


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return j.get("bf16_tflops", 1800.0), j.get("bf16_tflops_sustained", 1400.0), j.get("hbm_gbs", 6400.0), "measured"
    return 1800.0, 1400.0, 6400.0, "fallback"


def kernel_source_hash():
    csrc = os.path.join(ROOT, "audio_diffusion_transformer_fwd_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu capture, if it was taken
    on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        j = json.load(fh)
    if j.get("source_hash") != kernel_source_hash():
        return None
    return j.get("kernels", {}).get(kernel_key)


def write_traffic(csv_path):
    """profiles/ncu_traffic.json from an ncu --csv capture of
    dram__bytes_read.sum and dram__bytes_write.sum over the launches of one
    block (the command is in profiles/dram_traffic_block_512.md): DRAM bytes
    per launch by kernel class (attention: its launches of the block added),
    and the four GEMM launches' sum, stamped with the hash of the kernel
    sources they were taken on."""
    import csv
    import re
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1024.0, "MB": 1024.0 ** 2}
    with open(csv_path) as fh:
        rows = [r for r in csv.reader(fh)]
    hi = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    hdr = rows[hi]
    ki, mi, vi, ui = (hdr.index(c) for c in ("Kernel Name", "Metric Name", "Metric Value", "Metric Unit"))
    per_launch = {}
    for r in rows[hi + 1:]:
        if r[mi] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        per_launch.setdefault(r[0], [r[ki], 0.0])[1] += float(r[vi].replace(",", "")) * scale.get(r[ui], 1.0)
    order = ["qkv_gemm", "out_proj_gemm", "fc1_gemm", "fc2_gemm"]
    gemms = [(name, b) for name, b in per_launch.values() if "gemm" in name]
    out = {"source_hash": kernel_source_hash(), "unit": "bytes per launch", "kernels": {}}
    for key, (name, b) in zip(order, gemms[:4]):
        out["kernels"][key] = b
    if len(gemms) >= 4:
        out["kernels"]["gemm_per_block"] = sum(b for _, b in gemms[:4])
    for name, b in per_launch.values():
        m = re.search(r"(attn_fwd|gate_adaln_kernel<[^>]*>|rope_table)", name)
        if m and m.group(1) == "attn_fwd":
            # the full waves and, when the last wave is short, its key-split tail
            out["kernels"]["attn_fwd"] = out["kernels"].get("attn_fwd", 0.0) + b
        elif m:
            out["kernels"].setdefault(m.group(1), b)
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json"), "w") as fh:
        json.dump(out, fh, indent=1)
    print(json.dumps(out))
    return 0


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []          # (host time, csv line)
        self.window = None

    def start(self):
        """Start sampling (before the warm-up, so that nvidia-smi is already
        running when the timed region opens)."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self, t0, t1):
        """The host-time window of the timed region."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)   # let the sample that closes the window arrive
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        lines = self.lines
        if self.window is not None:
            t0, t1 = self.window
            inside = [x for x in lines if t0 <= x[0] <= t1 + 0.1]
            lines = inside if inside else sorted(lines, key=lambda x: abs(x[0] - t1))[:1]
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


class Ranks:
    """The replica plumbing of the bench: one process per GPU (torchrun),
    a barrier that also drains the local device, and max-over-ranks timing,
    so the slowest replica sets the time and `value` is the work of all
    ranks divided by it.  `dist` is torch.distributed once initialised (NCCL
    on GPUs, gloo in the CPU tests), or None for one process."""

    def __init__(self, world_size, rank, dist=None, device="cuda"):
        self.world_size, self.rank, self.dist, self.device = world_size, rank, dist, device

    def barrier(self):
        import torch
        if self.dist is not None:
            self.dist.barrier()
        if self.device == "cuda":
            torch.cuda.synchronize()

    def max(self, v):
        if self.dist is None:
            return v
        import torch
        t = torch.tensor([v], device=self.device, dtype=torch.float64)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return t.item()

    def throughput(self, work_per_rank, ms):
        """Whole-job rate: every rank's work over the slowest rank's time."""
        return work_per_rank * self.world_size / (ms * 1e-3)


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------------------- CPU oracle arm
class OracleSample:
    """The fp64 oracle block at a workload's widths (d 5120, 40 x 128 heads,
    F 20480 for the 512 class) over the workload's tokens or a bounded prefix
    of them; weights drawn once.  Attention runs over the sampled tokens
    only."""

    def __init__(self, workload="block_512"):
        import oracle as O
        from audio_diffusion_transformer_fwd_b300 import synth
        self.O = O
        self.name = workload
        self.w = w = synth.WORKLOADS[workload]
        self.cfg = O.BlockConfig(d=w.d, heads=w.heads, head_dim=w.head_dim, ffn=w.ffn, eps=w.eps,
                                 rope_sections=w.sections, rope_theta=w.theta)
        self.wt = synth.host_block_weights(w.d, w.ffn, seed=0)
        self.mod = synth.host_mod(w.d, seed=0)
        self.x = synth.host_activations(w.n_tokens, w.d, seed=0)
        self.pos = synth.positions(w.video, w.n_text, w.n_audio)
        self.cores = os.cpu_count()
        try:
            import threadpoolctl
            info = threadpoolctl.threadpool_info()
            self.cores = max((i.get("num_threads", 0) for i in info), default=self.cores) or self.cores
        except Exception:
            pass

    def run(self, n):
        t0 = time.perf_counter()
        self.O.block_forward(self.x[:n], self.wt, self.mod, self.pos[:n], self.cfg)
        dt = time.perf_counter() - t0
        return block_flops(n, self.w.d, self.w.ffn), dt

    def desc(self, n):
        w = self.w
        part = (f"all {n} tokens" if n >= w.n_tokens
                else f"the first {n} of the {w.n_tokens} tokens (attention over those {n})")
        return (f"fp64 numpy oracle: one {self.name} block (d={w.d}, {w.heads}x{w.head_dim} heads, F={w.ffn}) over "
                f"{part}, {block_flops(n, w.d, w.ffn):.3e} FLOP")


def run_reference(args):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return 0
    sample = OracleSample()
    # size the per-step sample so that warm-up + timed steps take ~2.5 minutes
    fl, dt = sample.run(256)
    per_token_s = dt / 256
    n = int(150.0 / max(1, args.steps + args.warmup) / per_token_s) // 64 * 64
    n = max(64, min(CPU_SAMPLE_TOKENS, n))
    for _ in range(args.warmup):
        sample.run(n)
    tot_fl, tot_s = 0.0, 0.0
    for _ in range(args.steps):
        fl, dt = sample.run(n)
        tot_fl += fl
        tot_s += dt
    value = tot_fl / tot_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot_s / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD_DESC, "sample_tokens": n},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": sample.cores, "kind": "oracle",
                         "sample": sample.desc(n)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    from audio_diffusion_transformer_fwd_b300 import h3dit as H
    from audio_diffusion_transformer_fwd_b300 import synth

    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    ranks = Ranks(ws, rank, dist)
    barrier, max_over_ranks = ranks.barrier, ranks.max

    burst, sustained, hbm, peak_src = measured_peaks()
    w = synth.WORKLOADS["block_512"]
    n, d, f = w.n_tokens, w.d, w.ffn
    shape = H.BlockShape(w.d, w.heads, w.head_dim, w.ffn, w.eps, w.sections, w.theta)
    stream = torch.cuda.current_stream()
    wdev = synth.device_block_weights(d, f, seed=rank, block=0)
    bw = H.block_weights(wdev["w_qkv"], wdev["w_o"], wdev["w1"], wdev["w2"])
    mod = synth.device_mods(1, d, seed=rank)
    x = synth.device_activations(n, d, seed=rank)
    pos = torch.from_numpy(synth.positions(w.video, w.n_text, w.n_audio)).cuda()
    nbytes = H.h3dit_workspace_size(shape, n)
    wsb = torch.empty(nbytes, device="cuda", dtype=torch.uint8)

    def step():
        H.h3dit_block_forward(shape, bw, mod, x, pos, n, wsb, nbytes, stream)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        step()
    H.h3dit_check_device_error(stream)

    # ---- device-timed region (inputs resident; weights 629 MB > L2 per step),
    # no per-kernel events inside it
    barrier()
    t_host0 = time.monotonic()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    barrier()
    sampler.mark(t_host0, time.monotonic())
    H.h3dit_check_device_error(stream)
    ms = max_over_ranks(ev0.elapsed_time(ev1)) / args.steps

    # ---- per-kernel breakdown: the same blocks again with CUDA events around
    # every launch on the launch stream (the library's per-class timing)
    H.h3dit_timing_reset()
    H.h3dit_timing_enable(True)
    barrier()
    for _ in range(args.steps):
        step()
    barrier()
    H.h3dit_timing_enable(False)
    clocks = sampler.stop()
    H.h3dit_check_device_error(stream)
    per_class = {name: H.h3dit_timing_read(k) for name, k in
                 (("rows", H.KC_ROWS), ("qkv", H.KC_QKV), ("attention", H.KC_ATTN), ("out_proj", H.KC_OPROJ),
                  ("fc1", H.KC_FC1), ("fc2", H.KC_FC2))}
    launches = sum(c for _, c in per_class.values())
    fl = block_flops(n, d, f)
    value = ranks.throughput(fl, ms) / 1e12

    gemm_ms = sum(per_class[k][0] for k in ("qkv", "out_proj", "fc1", "fc2")) / args.steps
    gemm_launch = sum(per_class[k][1] for k in ("qkv", "out_proj", "fc1", "fc2")) / args.steps
    attn_ms = per_class["attention"][0] / args.steps
    rows_ms = per_class["rows"][0] / args.steps
    gfl = gemm_flops(n, d, f)
    achieved = gfl / (gemm_ms * 1e-3) / 1e12
    kernels = {
        "qkv_gemm": {"ms": per_class["qkv"][0] / args.steps, "tflops": 2.0 * n * d * 3 * d / (per_class["qkv"][0] / args.steps * 1e-3) / 1e12},
        "out_proj_gemm": {"ms": per_class["out_proj"][0] / args.steps, "tflops": 2.0 * n * d * d / (per_class["out_proj"][0] / args.steps * 1e-3) / 1e12},
        "fc1_gemm": {"ms": per_class["fc1"][0] / args.steps, "tflops": 2.0 * n * d * f / (per_class["fc1"][0] / args.steps * 1e-3) / 1e12},
        "fc2_gemm": {"ms": per_class["fc2"][0] / args.steps, "tflops": 2.0 * n * d * f / (per_class["fc2"][0] / args.steps * 1e-3) / 1e12},
        "attention": {"ms": attn_ms, "tflops": 4.0 * n * n * d / (attn_ms * 1e-3) / 1e12,
                      "frac_of_sustained": 4.0 * n * n * d / (attn_ms * 1e-3) / 1e12 / sustained,
                      "frac_of_burst": 4.0 * n * n * d / (attn_ms * 1e-3) / 1e12 / burst},
        "row_kernels": {"ms": rows_ms, "note": "rope table + AdaLN-1 + gated residual fused with AdaLN-2 + "
                        "final gated residual per block"},
    }
    # attention's second roofline: one exponential per score (N^2 per head)
    # on the MUFU pipe, 16 results per clock per SM, at the run's median SM clock
    sm_mhz = clocks.get("sm_mhz") if isinstance(clocks, dict) else None
    if sm_mhz and attn_ms > 0:
        n_sm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        exps = float(n) * n * w.heads
        kernels["attention"]["mufu"] = {
            "exp2_per_block": exps, "rate": f"16 per clock per SM x {n_sm} SMs at {sm_mhz:.0f} MHz",
            "min_ms": exps / (16.0 * n_sm * sm_mhz * 1e6) * 1e3,
            "frac": exps / (attn_ms * 1e-3) / (16.0 * n_sm * sm_mhz * 1e6)}
    # algorithmic bytes of the row kernels of one block: AdaLN-1 reads x and
    # writes h (4 N d), the fused gated residual + AdaLN-2 reads x and the
    # branch and writes x and h2 (8 N d), the final gated residual reads x and
    # the branch and writes x (6 N d); the RoPE table reads the positions and
    # writes N * Dh/2 (cos, sin) fp32 pairs
    rows_bytes = 18.0 * n * d + n * (12.0 + (w.head_dim // 2) * 8.0)
    rows_gbs = None
    if rows_ms > 0:
        rows_gbs = rows_bytes / (rows_ms * 1e-3) / 1e9
        kernels["row_kernels"]["bytes_per_block"] = rows_bytes
        kernels["row_kernels"]["gbs"] = rows_gbs
        kernels["row_kernels"]["frac_of_hbm"] = rows_gbs / hbm
        kernels["row_kernels"]["timing"] = ("CUDA events around each launch inside the block loop, at the "
                                            "power-capped SM clock of the run (the row kernels' two block "
                                            "reductions make them slower at lower SM clocks)")

    # The denominator follows the length of the timed region: the measured
    # sustained BF16 rate (cuBLAS back to back for 4 s under the power cap) only
    # for a region of a second or more, the burst rate for anything shorter.
    region_s = ms * args.steps / 1e3
    long_region = region_s >= 1.0
    peak = sustained if long_region else burst
    roofline = {"kernel": "tcgen05 BF16 GEMM (QKV+RoPE, out-proj, FC1+GELU, FC2), all launches of a block",
                "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "frac_of_burst": achieved / burst, "frac_of_sustained": achieved / sustained,
                "peak_source": (f"{peak_src} bf16 {'sustained' if long_region else 'burst'} "
                                f"(timed region {region_s:.2f} s; sustained = cuBLAS 8192^3 back to back for 4 s "
                                f"under the power cap, used for regions of 1 s or more; burst = best of 10)"),
                "traffic": ncu_traffic("gemm_per_block"), "algorithmic_flops_per_block": gfl,
                "launches_per_block": gemm_launch}

    # ---- end-to-end through the C ABI with host buffers.  Every step copies
    # its input (x, mod, pos) from pinned host memory and its result back.
    # The copies run on their own streams and the device buffers are double
    # buffered, so step i+1's upload and step i-1's download overlap step i's
    # blocks -- the pipelining a serving loop would use.
    xh = torch.empty((n, d), dtype=torch.bfloat16).pin_memory()
    xh.copy_(x.cpu())
    modh = mod.cpu().pin_memory()
    posh = pos.cpu().pin_memory()
    xo = [torch.empty((n, d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xb = [x, x.clone()]
    mb = [mod, mod.clone()]
    pb = [pos, pos.clone()]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    e2e_steps = max(2, args.steps)   # as long as the device-timed run, so both see the same power state
    ev_in = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_done = [torch.cuda.Event() for _ in range(e2e_steps)]
    ev_out = [torch.cuda.Event() for _ in range(e2e_steps)]
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)
    for i in range(e2e_steps):
        k = i % 2
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(ev_out[i - 2])     # buffer k's previous result has been read back
            xb[k].copy_(xh, non_blocking=True)
            mb[k].copy_(modh, non_blocking=True)
            pb[k].copy_(posh, non_blocking=True)
            ev_in[i].record(up)
        stream.wait_event(ev_in[i])
        H.h3dit_block_forward(shape, bw, mb[k], xb[k], pb[k], n, wsb, nbytes, stream)
        ev_done[i].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[i])
            xo[k].copy_(xb[k], non_blocking=True)
            ev_out[i].record(down)
    stream.wait_event(ev_out[e2e_steps - 1])
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1)) / e2e_steps
    h2d = xh.numel() * 2 + modh.numel() * 4 + posh.numel() * 4
    d2h = xo[0].numel() * 2

    del wsb
    # ---- the same block on the dynamic-int8 path
    int8_res = run_int8_block(args, H, synth, torch, stream, barrier, max_over_ranks, rank, wdev, mod, x, pos)

    # ---- the final layer (video and audio heads) on the block's output
    final_res = run_final_layer(args, H, torch, stream, barrier, max_over_ranks, shape, x, n, d, hbm)

    # ---- 50-block steps (864x480 class), latency
    step_res = {}
    if not args.skip_step:
        step_res = run_steps(args, H, synth, torch, stream, barrier, max_over_ranks, rank)

    cpu = None
    if rank == 0 and not args.skip_cpu:
        # one whole block_512 block (the bench workload, every token, attention
        # over all 6912) and one whole tiny block; the 50-block step times are
        # extrapolated from the measured block rate and labelled as such
        sample = OracleSample()
        fl_c, dt_c = sample.run(n)
        tiny = OracleSample("tiny_block")
        fl_t, dt_t = tiny.run(tiny.w.n_tokens)
        cpu = {"value": fl_c / dt_c / 1e12, "unit": "TFLOP/s", "cores": sample.cores, "kind": "oracle",
               "sample": sample.desc(n), "seconds": dt_c,
               "tiny_block": {"value": fl_t / dt_t / 1e12, "unit": "TFLOP/s", "seconds": dt_t,
                              "sample": tiny.desc(tiny.w.n_tokens)}}
        if step_res.get("step_864"):
            st = synth.WORKLOADS["step_864"]
            cpu["step_864_extrapolated_s"] = st.n_blocks * block_flops(st.n_tokens, st.d, st.ffn) / (fl_c / dt_c)
            cpu["extrapolation"] = ("50 x the FLOP of one 10488-token block at the measured rate of the whole "
                                    "block_512 block: an estimate, not a measurement")

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,0.1) AdaLN, N(0,1) x)",
            "config": {"workload": WORKLOAD_DESC, "parallelism": f"replicas x{ws}",
                       "l2": "inputs larger than L2: 629 MB of block weights streamed every step"},
            "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu,
            "e2e": {"value": ranks.throughput(fl, e2e_ms) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "pipelining": "uploads and downloads on their own streams, device buffers double-buffered"},
            "gpu_launches": int(launches), "clocks": clocks, "int8": int8_res, "final_layer": final_res,
            "step": step_res,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_final_layer(args, H, torch, stream, barrier, max_over_ranks, shape, x, n, d, hbm):
    """The final layer at the 512 class: a video head over rows 0..6143 and
    an audio head over rows 6656..6911, 64 output channels each, AdaLN fused
    into the projection's operand load.  HBM-bound: the algorithmic bytes are
    the head rows read once plus the weights and the outputs."""
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    specs = ((0, 6144, 64), (6656, 256, 64))
    heads, keep = [], []
    for r0, rows, c in specs:
        sh = torch.randn(d, device="cuda", generator=g) * 0.1
        sc = torch.randn(d, device="cuda", generator=g) * 0.1
        wt = (torch.randn((c, d), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        out = torch.empty((rows, c), device="cuda", dtype=torch.bfloat16)
        heads.append(H.final_head(r0, rows, sh, sc, wt, c, out))
        keep += [sh, sc, wt, out]
    # three copies of the stream (210 MB, more than L2) used in turn
    xs = [x] + [x.clone() for _ in range(2)]
    for i in range(args.warmup):
        H.h3dit_final_layer(shape, xs[i % 3], n, heads, stream)
    H.h3dit_check_device_error(stream)
    steps = max(1, min(args.steps, 51))
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        H.h3dit_final_layer(shape, xs[i % 3], n, heads, stream)
    e1.record(stream)
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1)) / steps
    byts = sum(rows * d * 2 + c * d * 2 + rows * c * 2 + 8 * d for _, rows, c in specs)
    flops = sum(2.0 * rows * d * c for _, rows, c in specs)
    return {"workload": "video head rows 0..6143 + audio head rows 6656..6911 of the 512-class stream, "
                        "64 output channels each",
            "ms": ms, "gbs": byts / (ms * 1e-3) / 1e9, "frac_of_hbm": byts / (ms * 1e-3) / 1e9 / hbm,
            "tflops": flops / (ms * 1e-3) / 1e12, "bytes": byts, "steps": steps,
            "l2": "three copies of the stream used in turn (210 MB, more than L2)"}


def run_int8_block(args, H, synth, torch, stream, barrier, max_over_ranks, rank, wdev, mod, x, pos):
    """The 512-class block on the dynamic-int8 paths: all four projections in
    int8 (config 3), the MLP alone and QKV alone.  The BF16 weights are
    quantised per output channel by the library and widened to operand form
    once, outside the timed region; each variant is timed like the BF16 block."""
    w = synth.WORKLOADS["block_512_int8"]
    n, d, f = w.n_tokens, w.d, w.ffn
    codes, scales, bytes8 = {}, {}, {}
    for k, t in wdev.items():
        q8 = torch.empty(t.shape, device="cuda", dtype=torch.int8)
        sc = torch.empty(t.shape[0], device="cuda", dtype=torch.float32)
        H.h3dit_quantize_weight(t, t.shape[0], t.shape[1], q8, sc, stream)
        cb = torch.empty(t.shape, device="cuda", dtype=torch.bfloat16)
        H.h3dit_widen_codes(q8, q8.numel(), cb, stream)
        codes[k], scales[k], bytes8[k] = cb, sc, q8
    names = ("w_qkv", "w_o", "w1", "w2")
    # int8_resident: the same block with the weights kept as int8 bytes,
    # widened into the workspace before each projection
    variants = (("int8", H.INT8, names), ("int8_mlp", H.INT8_MLP, ("w1", "w2")), ("int8_qkv", H.INT8_QKV, ("w_qkv",)),
                ("int8_resident", H.INT8, names))
    burst, sustained, _, peak_src = measured_peaks()
    gops = gemm_flops(n, d, f)
    res = {"workload": "block_512_int8: the block_512 shapes with int8 QKV/out-proj/FC1/FC2 (per-token activation "
                       "scales, per-output-channel weight scales, FC2 one scale per 1024 input channels), BF16 attention; "
                       "variants with the MLP alone and QKV alone in int8",
           "peak_note": f"int8 codes run exactly on the BF16 tensor path (sm_103a has no integer tcgen05 MMA): "
                        f"peaks = {peak_src} bf16 sustained {sustained} / burst {burst}"}
    for name, prec, q_names in variants:
        shape = H.BlockShape(w.d, w.heads, w.head_dim, w.ffn, w.eps, w.sections, w.theta, prec)
        as_bytes = name == "int8_resident"
        src = bytes8 if as_bytes else codes
        ptr = [src[k] if k in q_names else wdev[k] for k in names]
        sc = [scales[k] if k in q_names else None for k in names]
        bw = H.block_weights(*ptr, *sc, codes_int8=as_bytes)
        weight_bytes = sum(p.numel() * p.element_size() for p in ptr) + sum(x.numel() * 4 for x in sc if x is not None)
        nbytes = H.h3dit_workspace_size(shape, n)
        wsb = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
        x8 = x.clone()

        def step():
            H.h3dit_block_forward(shape, bw, mod, x8, pos, n, wsb, nbytes, stream)

        for _ in range(args.warmup):
            step()
        H.h3dit_check_device_error(stream)
        steps = max(1, min(args.steps, 100 if name == "int8" else 30))
        H.h3dit_timing_reset()
        H.h3dit_timing_enable(True)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        barrier()
        H.h3dit_timing_enable(False)
        H.h3dit_check_device_error(stream)
        ms = max_over_ranks(e0.elapsed_time(e1)) / steps
        cls = {c: H.h3dit_timing_read(k) for c, k in
               (("qkv", H.KC_QKV), ("out_proj", H.KC_OPROJ), ("fc1", H.KC_FC1), ("fc2", H.KC_FC2),
                ("attention", H.KC_ATTN), ("rows", H.KC_ROWS), ("quant", H.KC_QUANT))}
        gemm_ms = sum(cls[k][0] for k in ("qkv", "out_proj", "fc1", "fc2")) / steps
        res[name] = {"ms": ms, "tops": block_flops(n, d, f) / (ms * 1e-3) / 1e12,
                     "gemm_ms": gemm_ms, "gemm_tops": gops / (gemm_ms * 1e-3) / 1e12,
                     "gemm_frac_of_bf16_sustained": gops / (gemm_ms * 1e-3) / 1e12 / sustained,
                     "gemm_frac_of_bf16_burst": gops / (gemm_ms * 1e-3) / 1e12 / burst,
                     "quant_ms": cls["quant"][0] / steps, "rows_ms": cls["rows"][0] / steps,
                     "attention_ms": cls["attention"][0] / steps, "steps": steps,
                     "weight_bytes_resident": weight_bytes}
        if as_bytes:
            res[name]["note"] = ("weights kept as int8 bytes (half the operand form) and widened into the "
                                 "workspace before each projection; quant_ms includes the widening")
        del wsb
    del codes, bytes8
    torch.cuda.empty_cache()
    return res


def run_steps(args, H, synth, torch, stream, barrier, max_over_ranks, rank):
    """50-block step latency at the 864x480 class, without and with token
    reduction (same weights)."""
    w = synth.WORKLOADS["step_864"]
    n, d, f, nb = w.n_tokens, w.d, w.ffn, w.n_blocks
    shape = H.BlockShape(w.d, w.heads, w.head_dim, w.ffn, w.eps, w.sections, w.theta)
    wdev = [synth.device_block_weights(d, f, seed=100 + rank, block=b) for b in range(nb)]
    bws = [H.block_weights(t["w_qkv"], t["w_o"], t["w1"], t["w2"]) for t in wdev]
    mods = synth.device_mods(nb, d, seed=100 + rank)
    x0 = synth.device_activations(n, d, seed=100 + rank)
    x = x0.clone()
    pos = torch.from_numpy(synth.positions(w.video, w.n_text, w.n_audio)).cuda()
    T, Hh, W = w.video
    out = {}
    _, sustained, _, _ = measured_peaks()
    for name, tr in (("step_864", None),
                     ("step_864_token_reduction", H.reduction(H.video_grid(0, T, Hh, W), 3, 40))):
        nbytes = H.h3dit_workspace_size(shape, n, tr)
        wsb = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
        reps = max(1, min(3, args.steps))
        for _ in range(max(1, min(2, args.warmup))):
            x.copy_(x0)
            H.h3dit_step_forward(shape, bws, mods, x, pos, n, tr, wsb, nbytes, stream)
        H.h3dit_check_device_error(stream)
        barrier()
        tot = 0.0
        for _ in range(reps):
            x.copy_(x0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            H.h3dit_step_forward(shape, bws, mods, x, pos, n, tr, wsb, nbytes, stream)
            e1.record(stream)
            barrier()
            tot += e0.elapsed_time(e1)
        ms = max_over_ranks(tot / reps)
        if tr is None:
            fl = nb * block_flops(n, d, f)
        else:
            nr = H.h3dit_reduced_tokens(n, H.video_grid(0, T, Hh, W))
            fl = 4 * block_flops(n, d, f) + 36 * block_flops(nr, d, f) + 10 * block_flops(n, d, f)
        out[name] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "frac_of_sustained": fl / (ms * 1e-3) / 1e12 / sustained,
                     "n_tokens": n, "blocks": nb, "reps": reps}
        del wsb
    del wdev
    torch.cuda.empty_cache()
    return out


def run_profile(args):
    """The 512-class block, BF16 or int8, run warmup + steps times with no
    timing: a short, fixed launch sequence for ncu (one block = rope table,
    AdaLN, QKV GEMM, attention, out-proj GEMM, fused residual + AdaLN, FC1,
    FC2, residual; int8 adds the quantisers)."""
    import torch
    from audio_diffusion_transformer_fwd_b300 import h3dit as H
    from audio_diffusion_transformer_fwd_b300 import synth
    torch.cuda.set_device(0)
    w = synth.WORKLOADS["block_512"]
    n, d, f = w.n_tokens, w.d, w.ffn
    if args.profile == "final":
        return run_profile_final(args, H, synth, torch, w)
    if args.tokens:
        n = max(1, min(n, args.tokens))
    prec = H.INT8 if args.profile == "int8" else H.BF16
    shape = H.BlockShape(w.d, w.heads, w.head_dim, w.ffn, w.eps, w.sections, w.theta, prec)
    wdev = synth.device_block_weights(d, f, seed=0, block=0)
    if prec == H.INT8:
        codes, scales = {}, {}
        for k, t in wdev.items():
            q8 = torch.empty(t.shape, device="cuda", dtype=torch.int8)
            sc = torch.empty(t.shape[0], device="cuda", dtype=torch.float32)
            H.h3dit_quantize_weight(t, t.shape[0], t.shape[1], q8, sc)
            cb = torch.empty(t.shape, device="cuda", dtype=torch.bfloat16)
            H.h3dit_widen_codes(q8, q8.numel(), cb)
            codes[k], scales[k] = cb, sc
        bw = H.block_weights(codes["w_qkv"], codes["w_o"], codes["w1"], codes["w2"],
                             scales["w_qkv"], scales["w_o"], scales["w1"], scales["w2"])
    else:
        bw = H.block_weights(wdev["w_qkv"], wdev["w_o"], wdev["w1"], wdev["w2"])
    mod = synth.device_mods(1, d, seed=0)
    x = synth.device_activations(n, d, seed=0)
    pos = torch.from_numpy(synth.positions(w.video, w.n_text, w.n_audio)[:n]).cuda()
    nbytes = H.h3dit_workspace_size(shape, n)
    wsb = torch.empty(nbytes, device="cuda", dtype=torch.uint8)
    for _ in range(args.warmup + args.steps):
        H.h3dit_block_forward(shape, bw, mod, x, pos, n, wsb, nbytes)
    H.h3dit_check_device_error()
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.profile, "tokens": n, "blocks": args.warmup + args.steps}))
    return 0


def run_profile_final(args, H, synth, torch, w):
    """The final layer of the 512 class (video head rows 0..6143, audio head
    rows 6656..6911, 64 channels each) run warmup + steps times, no timing:
    two launches per layer (row statistics, head GEMM)."""
    n, d = w.n_tokens, w.d
    shape = H.BlockShape(w.d, w.heads, w.head_dim, w.ffn, w.eps, w.sections, w.theta)
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    heads, keep = [], []
    for r0, rows, c in ((0, 6144, 64), (6656, 256, 64)):
        sh = torch.randn(d, device="cuda", generator=g) * 0.1
        sc = torch.randn(d, device="cuda", generator=g) * 0.1
        wt = (torch.randn((c, d), device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        out = torch.empty((rows, c), device="cuda", dtype=torch.bfloat16)
        heads.append(H.final_head(r0, rows, sh, sc, wt, c, out))
        keep += [sh, sc, wt, out]
    x = synth.device_activations(n, d, seed=0)
    for _ in range(args.warmup + args.steps):
        H.h3dit_final_layer(shape, x, n, heads)
    H.h3dit_check_device_error()
    torch.cuda.synchronize()
    print(json.dumps({"profile": "final", "tokens": n, "layers": args.warmup + args.steps}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-step", action="store_true", help="omit the 50-block step latencies")
    ap.add_argument("--skip-cpu", action="store_true", help="omit the oracle CPU baseline")
    ap.add_argument("--tokens", type=int, default=None,
                    help="with --profile: run the block on the first TOKENS tokens of the workload (a small case)")
    ap.add_argument("--profile", choices=["bf16", "int8", "final"], default=None,
                    help="run only WARMUP + STEPS forwards of the 512-class block, or of its final layer "
                         "(no report): the command the ncu captures under profiles/ run")
    ap.add_argument("--traffic-from", default=None,
                    help="write profiles/ncu_traffic.json from an ncu DRAM-bytes CSV of one block and exit")
    args = ap.parse_args()
    if args.traffic_from:
        return write_traffic(args.traffic_from)
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
