#!/usr/bin/env python
"""Benchmark of the KDA hot path on GB300: prefill tokens/s (T=8192, H=96, d=128, bf16) and
decode state GB/s (N=256, H=96), against the HBM roofline.

One step = one kda_prefill of the 8192-token, 96-head workload (inputs resident in HBM).
The same step through kda_prefill_precise, the decode (256 sequences x 96 heads, 1.6 GB fp32
state updated in place), a checkpoint restore (kda_state_copy of 64 states), the pre-mixer and the
output gate on the same token grid, a prefix-reuse (cache-hit) prefill, the context-parallel
prefill of one 262,144-token sequence at 8 heads (and its scan and output correction alone), and
the varlen x8 and 262,144-token (64 checkpoints) prefills at 96 heads are timed in the same run
and reported beside it.  The CPU-baseline leg times the fp64 oracle on the step's own inputs and
compares the step's results with it, and those of the varlen x8, 262,144-token and
context-parallel figures on sampled heads.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

N > 1 runs under torchrun: every rank processes its own copy of the workload (the heads and
sequences of the path are independent, so ranks exchange nothing); value = all ranks'
tokens / the slowest rank's time.  --impl reference times the fp64 CPU oracle instead.
The pages report no throughput or kernel measurement for KDA, so vs_baseline is null.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s at H=96,d=128; decode state HBM GB/s vs peak"
PUBLISHED = "none: the pages report no KDA throughput, latency or kernel measurement"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

H, D = 96, 128
T1 = 8192                      # prefill workload: one sequence of 8192 tokens
N_DEC = 256                    # decode workload: 256 sequences
FLOP_PER_TOKEN_HEAD = 6 * D * D + 8 * 16 * D        # 114,688 (chunk C = 16 accounting)
BYTES_PER_TOKEN_HEAD = 4 * D * 2 + 2 + D * 2        # q, k, v, g, o bf16 + beta bf16 = 1,282
BYTES_PER_TOKEN_HEAD_FP32_OUT = 4 * D * 2 + 2 + D * 4   # the same with o in fp32, as written = 1,538
STATE_BYTES = D * D * 4                             # 65,536 per (sequence, head)
DECODE_BYTES_PER_SEQ_HEAD = 2 * STATE_BYTES + 4 * D * 2 + 2 + D * 4   # 132,610
PREMIX_BYTES_PER_TOKEN_HEAD = 2 * (4 * D * 2 + 2)    # xq, xk, xv, a, b in; q, k, v, g, beta out: 2,052
TOL_OUT, TOL_STATE = 2e-2, 1e-2   # bf16-input bounds: max|err| / RMS on outputs and on states
E2E_CHUNK = 1024               # tokens per chunk of the staged (copy-overlapped) end-to-end prefill


def set_heads(heads: int) -> None:
    global H
    if heads < 1:
        raise SystemExit("--heads must be positive")
    H = heads


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(value: float, device=None) -> float:
    """The maximum of `value` over all ranks of the default process group (any backend: a CPU
    tensor for gloo, a device tensor for NCCL).  Replicas finish when the slowest one does."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: float, slowest_ms: float, world: int) -> float:
    """Whole-job throughput of `world` replicas that each process `units_per_rank` units, over
    the slowest rank's time (weak scaling: the work per rank is fixed)."""
    return world * units_per_rank / (slowest_ms / 1e3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (the library nvidia-smi uses) every
    2 ms on a thread, so that a timed region of a few milliseconds still gets samples.  Read only;
    unavailable where the driver library is missing."""

    # clock-event reason bits of the NVML API
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_index: int, period_s: float = 0.002):
        import ctypes
        import threading

        self.samples = []
        self.max_mhz = None
        self.period = period_s
        self._stop = threading.Event()
        self._thread = None
        self._lib = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(gpu_index), ctypes.byref(handle)) != 0:
                return
            self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
            mx = ctypes.c_uint(0)
            if lib.nvmlDeviceGetMaxClockInfo(handle, ctypes.c_int(1), ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._lib, self._handle = lib, handle
        except (OSError, AttributeError):
            self._lib = None

    def _run(self):
        import ctypes
        import time

        mhz, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self._stop.is_set():
            if self._lib.nvmlDeviceGetClockInfo(self._handle, ctypes.c_int(1), ctypes.byref(mhz)) == 0:
                r = 0
                if self._reasons_fn is not None and self._reasons_fn(self._handle, ctypes.byref(rs)) == 0:
                    r = rs.value
                self.samples.append((float(mhz.value), r))
            time.sleep(self.period)

    def start(self):
        import threading

        if self._lib is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        return self.samples


class ClockSampler:
    """Clock / throttle samples during the timed region: nvidia-smi every 100 ms, and NVML every
    2 ms (the timed region of a default run is shorter than nvidia-smi's start-up)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.nvml = NvmlSampler(gpu_index)

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.nvml.start()

    def stop(self):
        fast = self.nvml.stop()
        rows = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        if self.path is not None and os.path.exists(self.path):   # also when nvidia-smi never ran
            os.unlink(self.path)
        self.path = None
        return summarize_clocks(rows, fast, self.nvml.max_mhz)


def summarize_clocks(smi_rows, nvml_samples, nvml_max_mhz):
    """Median SM clock, maximum SM clock and the throttle reasons seen, over nvidia-smi rows
    (`ClockSampler.FIELDS`, as strings) and NVML samples (MHz, reason bits)."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    sm = [float(r[1]) for r in smi_rows if r[1].replace(".", "").isdigit()]
    sm += [m for m, _ in nvml_samples]
    maxes = [float(r[2]) for r in smi_rows if r[2].replace(".", "").isdigit()]
    if nvml_max_mhz is not None:
        maxes.append(nvml_max_mhz)
    reasons = {names[i] for r in smi_rows for i in range(4) if r[5 + i].lower() == "active"}
    reasons |= {n for _, bits in nvml_samples for b, n in NvmlSampler.REASON_BITS.items() if bits & b}
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    sm.sort()
    return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(maxes) if maxes else None,
            "reasons": sorted(reasons), "samples": len(sm),
            "sources": {"nvidia_smi_100ms": len(smi_rows), "nvml_2ms": len(nvml_samples)}}


def cuda_time_ms(fn, steps, stream):
    """CUDA-event time of `steps` calls of fn on `stream`, plus the per-call average."""
    import torch

    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    stop.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(stop)
    return total, total / steps


def cuda_time_ms_queued(fn, steps, stream, hold_cycles=4_000_000):
    """As cuda_time_ms, for calls shorter than their host-side cost: a spin of `hold_cycles` GPU
    cycles holds the stream while the calls are queued, so the events time the calls back to back
    on the device rather than the rate at which the host submits them."""
    import torch

    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(hold_cycles)
    start.record(stream)
    for _ in range(steps):
        fn()
    stop.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(stop)
    return total, total / steps


def oracle_sample(tokens: int, heads: int, seed: int = 1, threads=None):
    """Run the fp64 oracle on the first `tokens` tokens of `heads` heads of the prefill
    workload's distributions; returns (seconds, threads used)."""
    import oracle
    from kimi_delta_attention_13_gb300 import synth

    x = synth.make_inputs([tokens], heads=heads, dtype="bf16", seed=seed, device="cpu")
    orc = oracle.default()
    nthreads = int(threads or os.cpu_count() or 1)
    t0 = time.perf_counter()
    orc.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], threads=nthreads)
    return time.perf_counter() - t0, min(nthreads, heads)


def rel_err(got, ref) -> float:
    """max |got - ref| / RMS(ref) over a tensor."""
    import numpy as np

    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref)) / rms) if rms > 0 else float(np.max(np.abs(got)))


def cpu_baseline(step, target_s: float = 10.0):
    """The oracle timed on a bounded sample of the timed step's own inputs (its first tokens, all
    96 heads), scaled to tokens/s; the step's GPU results on the same tokens are compared with the
    oracle's (outputs, and the final state when the sample is the whole sequence)."""
    import oracle

    orc = oracle.default()
    cores = int(os.cpu_count() or 1)
    x = step["inputs"]

    def run(tokens):
        sl = [x[k][:tokens] for k in ("q", "k", "v", "g", "beta")]
        t0 = time.perf_counter()
        o, f, _ = orc.prefill(*sl, threads=cores)
        return time.perf_counter() - t0, o, f

    t_small, _, _ = run(64)
    tokens = int(max(64, min(T1, 64 * target_s / max(t_small, 1e-3))))
    secs, o, f = run(tokens)
    base = {"value": tokens / secs, "unit": "tokens/s", "cores": min(cores, H), "kind": "oracle",
            "sample": f"fp64 oracle on the timed step's inputs: first {tokens} tokens x all {H} heads "
                      f"of the T=8192 workload ({secs:.1f} s)"}
    out_err = rel_err(step["out"][:tokens].numpy(), o)
    fin_err = rel_err(step["final"].numpy(), f) if tokens == T1 else None
    ok = out_err <= TOL_OUT and (fin_err is None or fin_err <= TOL_STATE)
    parity = {"vs": "fp64 oracle, same inputs", "tokens": tokens, "heads": H,
              "metric": "max|gpu - oracle| / RMS(oracle)", "out": out_err, "final_state": fin_err,
              "out_precise_mode": (rel_err(step["out_precise"][:tokens].numpy(), o)
                                   if "out_precise" in step else None),
              "tolerance": {"out": TOL_OUT, "final_state": TOL_STATE}, "pass": ok}
    return base, parity


def other_parity(named) -> None:
    """The CPU-baseline leg's oracle comparison for the other workloads: each figure's kept head
    sample against the fp64 oracle on the same inputs (outputs, final states, checkpoints), as
    max|gpu - oracle| / RMS(oracle) against the same bounds."""
    import oracle

    orc = oracle.default()
    cores = int(os.cpu_count() or 1)
    for fig in named.values():
        c = fig.pop("_check", None)
        if c is None:
            continue
        x = c["inputs"]
        t0 = time.perf_counter()
        ro, rf, rc = orc.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], c["cu"], c["init"],
                                 ckpt_stride=c["ckpt_stride"], threads=cores)
        par = {"vs": "fp64 oracle, same inputs", "heads": c["heads"],
               "metric": "max|gpu - oracle| / RMS(oracle)",
               "out": rel_err(c["out"].numpy(), ro), "final_state": rel_err(c["final"].numpy(), rf),
               "oracle_s": time.perf_counter() - t0}
        if c["ckpts"] is not None and rc is not None:
            par["ckpts"] = rel_err(c["ckpts"].numpy(), rc)
        par["pass"] = (par["out"] <= TOL_OUT and par["final_state"] <= TOL_STATE and
                       par.get("ckpts", 0.0) <= TOL_STATE)
        fig["parity"] = par


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    per_step_tokens = 256
    for _ in range(args.warmup):
        oracle_sample(per_step_tokens, H)
    secs = []
    cores = 1
    for _ in range(args.steps):
        s, cores = oracle_sample(per_step_tokens, H)
        secs.append(s)
    total = sum(secs)
    value = per_step_tokens * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"prefill T={T1} H={H} d={D} (oracle sample: {per_step_tokens} tokens "
                               f"x {H} heads per step)", "global_batch": 1, "seq_len": T1,
                   "parallelism": "cpu threads"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {per_step_tokens} tokens x {H} heads per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "published": PUBLISHED,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gb300(args):
    import torch

    import kimi_delta_attention_13_gb300 as kda
    from kimi_delta_attention_13_gb300 import build as kbuild
    from kimi_delta_attention_13_gb300 import synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    kbuild.build()
    kda.load()
    peaks, peak_kind = load_peaks()
    stream = torch.cuda.current_stream(dev)

    # ---- prefill workload (inputs resident in HBM, 1.0 GB: larger than L2) -----------------
    x = synth.make_inputs([T1], heads=H, dtype="bf16", seed=1, device=dev)
    out = torch.empty(T1, H, D, device=dev, dtype=torch.float32)
    fin = torch.empty(1, H, D, D, device=dev, dtype=torch.float32)

    def prefill_step():
        kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], out=out, final_state=fin, stream=stream)

    for _ in range(max(args.warmup, 3)):
        prefill_step()
    torch.cuda.synchronize()
    assert kda.device_status() == 0

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    total_ms, per_ms = cuda_time_ms(prefill_step, args.steps, stream)
    barrier()
    clk = clocks.stop()
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
        per_ms = total_ms / args.steps
    tokens_per_s = replica_throughput(T1 * args.steps, total_ms, world)
    # the roofline counts o in bf16 (the workload's byte budget); the kernel writes fp32 o, whose
    # fraction, on the bytes actually written, is reported beside it
    bytes_alg = T1 * H * BYTES_PER_TOKEN_HEAD + H * STATE_BYTES
    bytes_fp32_out = T1 * H * BYTES_PER_TOKEN_HEAD_FP32_OUT + H * STATE_BYTES
    flops_alg = T1 * H * FLOP_PER_TOKEN_HEAD
    achieved_gbs = bytes_alg / (per_ms / 1e3) / 1e9
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    t_bytes = bytes_alg / (hbm_peak * 1e9)
    t_flops = flops_alg / (float(peaks.get("bf16_tflops", 1900.0)) * 1e12)
    path = "tensor-core chunked" if kda.prefill_path(D, D, torch.bfloat16) == 1 else "per-token"

    # the same step in the kernel's precise mode (kda_prefill_precise), timed beside it
    out_p = torch.empty_like(out)

    def precise_step():
        kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], out=out_p, final_state=fin,
                    stream=stream, precise=True)

    for _ in range(3):
        precise_step()
    _, precise_ms = cuda_time_ms(precise_step, max(5, args.steps // 2), stream)
    assert kda.device_status() == 0

    # ---- end to end through the public API: pinned host inputs -> device -> host outputs -----
    hx = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}
    h_out = torch.empty(T1, H, D, dtype=torch.float32).pin_memory()
    h_fin = torch.empty(1, H, D, D, dtype=torch.float32).pin_memory()
    del x
    # the timed step's inputs and results, for the oracle comparison of the CPU-baseline leg
    with_base = rank == 0 and world == 1 and not args.no_cpu_baseline
    step = {"inputs": hx, "out": out.cpu(), "final": fin.cpu(), "out_precise": out_p.cpu()} \
        if with_base else None
    del out_p

    # the staged prefill: chunks whose uploads, prefills and downloads overlap; device
    # staging buffers are allocated once, as a serving loop would
    fin_d = torch.empty(1, H, D, D, device=dev, dtype=torch.float32)
    staged = {"buffers": None}

    def e2e_step():
        _, _, staged["buffers"] = kda.prefill_staged(
            hx["q"], hx["k"], hx["v"], hx["g"], hx["beta"], None, None, device=dev,
            chunk_tokens=E2E_CHUNK, buffers=staged["buffers"], h_out=h_out, final_state=fin_d,
            stream=stream)
        with torch.cuda.stream(stream):
            h_fin.copy_(fin_d, non_blocking=True)

    for _ in range(2):
        e2e_step()
    barrier()
    # one event pair per step on the caller's stream (a step's copies and prefills all finish
    # before the stream moves on): the mean over the steps is the figure, the spread is reported
    # beside it, since a shared host's memory traffic can slow single steps
    n_e2e = max(3, args.steps // 2)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e + 1)]
    torch.cuda.synchronize()
    marks[0].record(stream)
    for i in range(n_e2e):
        e2e_step()
        marks[i + 1].record(stream)
    torch.cuda.synchronize()
    e2e_steps = sorted(marks[i].elapsed_time(marks[i + 1]) for i in range(n_e2e))
    e2e_ms = marks[0].elapsed_time(marks[-1])
    e2e_per = e2e_ms / n_e2e
    if world > 1:
        e2e_per = max_over_ranks(e2e_per, dev)
    h2d = sum(v.numel() * v.element_size() for v in hx.values())
    d2h = h_out.numel() * 4 + h_fin.numel() * 4
    del h_out, h_fin, staged, fin_d
    hx = None
    torch.cuda.empty_cache()

    # ---- decode workload: 256 x 96 states (1.6 GB fp32), updated in place -----------------
    d = synth.make_decode_inputs(N_DEC, heads=H, seed=3, device=dev)
    dout = torch.empty(N_DEC, H, D, device=dev, dtype=torch.float32)

    def decode_step():
        kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"], out=dout, stream=stream)

    for _ in range(3):
        decode_step()
    _, dec_ms = cuda_time_ms(decode_step, max(5, args.steps), stream)
    dec_bytes = N_DEC * H * DECODE_BYTES_PER_SEQ_HEAD
    dec_gbs = dec_bytes / (dec_ms / 1e3) / 1e9
    del d, dout
    torch.cuda.empty_cache()

    # ---- checkpoint restore: 64 states of 96 heads (403 MB) gathered by index --------------
    src = torch.randn(64, H, D, D, device=dev)
    dst = torch.empty_like(src)
    idx = torch.randperm(64, device=dev)

    def copy_step():
        kda.state_copy(dst, src, idx, idx, stream=stream)

    for _ in range(3):
        copy_step()
    _, cp_ms = cuda_time_ms(copy_step, 10, stream)
    cp_gbs = 2 * src.numel() * 4 / (cp_ms / 1e3) / 1e9
    assert kda.device_status() == 0
    del src, dst
    torch.cuda.empty_cache()

    # ---- pre-mixer and output gate on the T = 8192, H = 96 token grid ----------------------
    px = synth.make_premix_inputs([T1], heads=H, d=D, dtype="bf16", seed=7, device=dev)
    pout = tuple(torch.empty_like(px["xq"]) for _ in range(4)) + (torch.empty_like(px["b"]),)

    def premix_step():
        kda.premix(px["xq"], px["xk"], px["xv"], px["a"], px["b"], px["w"], out=pout, stream=stream)

    for _ in range(3):
        premix_step()
    _, pm_ms = cuda_time_ms(premix_step, max(5, args.steps), stream)
    pm_bytes = PREMIX_BYTES_PER_TOKEN_HEAD * T1 * H + 3 * H * D * 4 * 4
    del px, pout
    torch.cuda.empty_cache()
    gx = synth.make_gate_inputs((T1, H, D), "f32", "bf16", seed=8, device=dev)
    gout = torch.empty(T1, H, D, device=dev, dtype=torch.bfloat16)

    def gate_step():
        kda.output_gate(gx["o"], gx["z"], out=gout, stream=stream)

    for _ in range(3):
        gate_step()
    _, og_ms = cuda_time_ms(gate_step, max(5, args.steps), stream)
    og_bytes = T1 * H * D * (4 + 2 + 2)
    assert kda.device_status() == 0
    del gx, gout
    torch.cuda.empty_cache()

    reuse = prefix_reuse_figure(dev, stream)
    assert kda.device_status() == 0
    torch.cuda.empty_cache()
    cp = context_parallel_figure(dev, stream, hbm_peak=hbm_peak, keep=with_base)
    assert kda.device_status() == 0
    torch.cuda.empty_cache()
    named = named_workload_figures(dev, stream, hbm_peak, keep=with_base)
    assert kda.device_status() == 0
    torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    base, parity = cpu_baseline(step) if with_base else (None, None)
    if with_base:
        other_parity(named)
        other_parity({"context_parallel": cp})
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "prefill_traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tr = json.load(f)
        if tr.get("kernel_source_hash") == kbuild_source_hash():
            traffic = tr.get("dram_bytes_per_launch")
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": per_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"prefill T={T1} H={H} d_k=d_v={D}: bf16 q/k/v/g/beta, fp32 out and "
                               "state, zero initial state, final state written (one sequence)",
                   "global_batch": world, "seq_len": T1, "heads": H, "head_dim": D,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2 ({T1 * H * (4 * D * 2 + 2) / 1e9:.2f} GB read per step), "
                         "no flush needed",
                   "prefill_kernel": path},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved_gbs / hbm_peak, "traffic": traffic,
                     "bytes_basis": "1,282 B per token-head: q, k, v, g, o in bf16, beta bf16; "
                                    "+ the fp32 final state",
                     "frac_fp32_out": bytes_fp32_out / (per_ms / 1e3) / 1e9 / hbm_peak,
                     "frac_fp32_out_basis": "1,538 B per token-head: o counted in fp32, as the "
                                            "kernel writes it",
                     "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                     "bytes_alg_per_launch": bytes_alg, "flops_alg_per_launch": flops_alg,
                     "t_bytes_us": t_bytes * 1e6, "t_flops_us": t_flops * 1e6,
                     "roofline_fraction": max(t_bytes, t_flops) / (per_ms / 1e3)},
        "e2e": {"value": world * T1 / (e2e_per / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_per,
                "step_ms": {"steps": len(e2e_steps), "min": e2e_steps[0],
                            "median": e2e_steps[len(e2e_steps) // 2], "max": e2e_steps[-1]},
                "path": f"kda_prefill_staged from pinned host buffers, {E2E_CHUNK}-token chunks whose "
                        "uploads, prefills and downloads overlap"},
        "precise_mode": {"workload": "the same prefill through kda_prefill_precise (Aqk carried in "
                                    "two fp16 parts; outputs' error in parity.out_precise_mode)",
                         "ms": precise_ms, "tokens_per_s": world * T1 / (precise_ms / 1e3),
                         "frac": bytes_alg / (precise_ms / 1e3) / 1e9 / hbm_peak,
                         "time_vs_default": precise_ms / per_ms},
        "premix": {"workload": f"pre-mixer T={T1} H={H} d={D}: width-4 causal conv of xq/xk/xv, "
                               "q/k L2 norm, decay and write gates, bf16 in and out",
                   "GB/s": pm_bytes / (pm_ms / 1e3) / 1e9, "peak": hbm_peak,
                   "frac": pm_bytes / (pm_ms / 1e3) / 1e9 / hbm_peak, "ms": pm_ms,
                   "bytes_alg": pm_bytes},
        "output_gate": {"workload": f"output gate T={T1} H={H} d={D}: fp32 o, bf16 z, bf16 out",
                        "GB/s": og_bytes / (og_ms / 1e3) / 1e9, "peak": hbm_peak,
                        "frac": og_bytes / (og_ms / 1e3) / 1e9 / hbm_peak, "ms": og_ms,
                        "bytes_alg": og_bytes},
        "decode": {"workload": f"decode N={N_DEC} H={H} d={D}, fp32 state in place",
                   "GB/s": dec_gbs, "peak": hbm_peak, "frac": dec_gbs / hbm_peak, "ms": dec_ms,
                   "bytes_alg": dec_bytes},
        "state_copy": {"workload": "64 states x 96 heads gathered by index (403 MB)",
                       "GB/s": cp_gbs, "frac": cp_gbs / hbm_peak, "ms": cp_ms},
        "prefix_reuse": reuse,
        "context_parallel": cp,
        "other_workloads": named,
        "gpu_launches": args.steps,
        "clocks": clk,
        "cpu_baseline": base,
        "parity": parity,
        "published": PUBLISHED,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def prefix_reuse_figure(dev, stream, n_req: int = 4, prefix: int = 16384, new_tokens: int = 1024,
                        stride: int = 4096):
    """Cache-hit prefill: `n_req` requests share a cached `prefix`-token sequence (checkpoints
    every `stride` tokens) and each adds `new_tokens` tokens. The cache-hit path restores the
    state at the prefix boundary (one kda_state_copy) and prefills only the new tokens; the full
    path prefills prefix + new tokens of every request."""
    import torch

    import kimi_delta_attention_13_gb300 as kda
    from kimi_delta_attention_13_gb300 import synth
    from kimi_delta_attention_13_gb300.prefix_cache import CheckpointStore, resume_prefill

    keys = ("q", "k", "v", "g", "beta")
    base = synth.make_inputs([prefix], heads=H, dtype="bf16", seed=7, device=dev)
    _, _, ck = kda.prefill(*[base[k] for k in keys], ckpt_stride=stride, lengths=[prefix], stream=stream)
    store = CheckpointStore(prefix // stride, H, device=dev)
    store.add_checkpoints(["base"], ck, stride, [prefix], stream=stream)
    del ck
    new = synth.make_inputs([new_tokens] * n_req, heads=H, dtype="bf16", seed=8, device=dev)
    slot, covered = store.lookup("base", prefix)
    lens_hit = [new_tokens] * n_req
    full = {k: torch.cat([t for i in range(n_req)
                          for t in (base[k], new[k][i * new_tokens:(i + 1) * new_tokens])], 0)
            for k in keys}
    lens_full = [prefix + new_tokens] * n_req
    cu_full = torch.tensor([0] + [sum(lens_full[:i + 1]) for i in range(n_req)], device=dev,
                           dtype=torch.int32)
    out_hit = torch.empty(n_req * new_tokens, H, D, device=dev)
    out_full = torch.empty(sum(lens_full), H, D, device=dev)
    fin = torch.empty(n_req, H, D, D, device=dev)

    def hit():
        resume_prefill(store, [slot] * n_req, *[new[k] for k in keys], new["cu_seqlens"], lens_hit,
                       out=out_hit, final_state=fin, stream=stream)

    def miss():
        kda.prefill(*[full[k] for k in keys], cu_full, None, out=out_full, final_state=fin,
                    lengths=lens_full, stream=stream)

    for fn in (hit, miss):
        fn()
    _, hit_ms = cuda_time_ms(hit, 5, stream)
    _, miss_ms = cuda_time_ms(miss, 3, stream)
    served = n_req * (prefix + new_tokens)
    return {"workload": f"{n_req} requests x ({prefix}-token cached prefix, checkpoints every "
                        f"{stride}) + {new_tokens} new tokens, H={H}",
            "cache_hit_ms": hit_ms, "full_prefill_ms": miss_ms,
            "cache_hit_tokens_per_s": served / (hit_ms / 1e3),
            "new_tokens_per_s": n_req * new_tokens / (hit_ms / 1e3),
            "speedup": miss_ms / hit_ms, "restored_from_tokens": covered}


def named_workload_figures(dev, stream, hbm_peak, keep: bool = False):
    """The other two prefill workloads beside the T=8192 step, timed the same way (CUDA events on
    the launching stream, 2 warm-ups, 3 launches): varlen x8 (8 sequences of U[1024, 32768] tokens,
    initial and final states) and one sequence of 262,144 tokens with a checkpoint every 4096.
    Algorithmic bytes: 1,282 B per token-head (bf16 o) plus 64 KB per state read or written.
    With `keep`, each figure also keeps host copies of its inputs and GPU results on 8 sampled heads
    (the long workload's oracle heads) for the oracle comparison of the CPU-baseline leg."""
    import torch

    import kimi_delta_attention_13_gb300 as kda
    from kimi_delta_attention_13_gb300 import synth

    res = {}
    ws = synth.workloads()
    for w, key in ((ws[2], "varlen8"), (ws[4], "long_T262144_ckpt4096")):
        lengths = [int(L) for L in w.lengths]
        T, N = sum(lengths), len(lengths)
        x = synth.make_inputs(lengths, heads=H, dtype="bf16", seed=w.seed, device=dev,
                              init_state=w.init_state)
        n_ck = kda.num_checkpoints(lengths, w.ckpt_stride) if w.ckpt_stride else 0
        o = torch.empty(T, H, D, device=dev)
        fin = torch.empty(N, H, D, D, device=dev)
        ck = torch.empty(n_ck, H, D, D, device=dev) if n_ck else None

        def step():
            kda.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], x["state"],
                        out=o, final_state=fin, ckpt_stride=w.ckpt_stride, ckpts=ck,
                        lengths=lengths, stream=stream)

        for _ in range(2):
            step()
        _, ms = cuda_time_ms(step, 3, stream)
        states = N * (2 if w.init_state else 1) + n_ck
        b = T * H * BYTES_PER_TOKEN_HEAD + states * H * STATE_BYTES
        if keep:
            hs = synth.long_context_oracle_heads() if H == 96 else list(range(min(H, 8)))
            idx = torch.tensor(hs, device=dev)
            check = {"heads": hs, "ckpt_stride": w.ckpt_stride,
                     "inputs": {k_: x[k_].index_select(1, idx).cpu() for k_ in ("q", "k", "v", "g", "beta")},
                     "cu": x["cu_seqlens"].cpu().long(),
                     "init": None if x["state"] is None else x["state"].index_select(1, idx).cpu(),
                     "out": o.index_select(1, idx).cpu(), "final": fin.index_select(1, idx).cpu(),
                     "ckpts": ck.index_select(1, idx).cpu() if ck is not None else None}
        res[key] = {"workload": f"{w.name}: {N} sequence(s), {T} tokens, H={H}, "
                                f"{n_ck} checkpoints, fp32 out",
                    "ms": ms, "tokens_per_s": T / (ms / 1e3), "bytes_alg": b,
                    "GB/s": b / (ms / 1e3) / 1e9, "frac": b / (ms / 1e3) / 1e9 / hbm_peak,
                    "longest_sequence": max(lengths)}
        if keep:
            res[key]["_check"] = check
        del x, o, fin, ck
        torch.cuda.empty_cache()
    return res


def context_parallel_figure(dev, stream, T=262144, heads=8, hbm_peak=None, keep=False):
    """One long sequence at a low head count: the plain prefill runs one CTA per head; the
    context-parallel prefill cuts the sequence into segments that prefill side by side.  The scan
    and the output correction are also timed alone.  With `keep`, 4 of the heads' inputs and
    results stay on the host for the CPU-baseline leg's oracle comparison."""
    import torch

    import kimi_delta_attention_13_gb300 as kda
    from kimi_delta_attention_13_gb300 import synth
    from kimi_delta_attention_13_gb300.context_parallel import (auto_seg_len, cp_combine, cp_correct,
                                                                prefill_cp)

    seg_len = auto_seg_len(T, heads, torch.cuda.get_device_properties(dev).multi_processor_count)

    x = synth.make_inputs([T], heads=heads, dtype="bf16", seed=9, device=dev)
    args = [x[k_] for k_ in ("q", "k", "v", "g", "beta")]

    def plain():
        kda.prefill(*args, stream=stream)

    def split():
        prefill_cp(*args, seg_len=seg_len, lengths=[T], stream=stream)

    plain()
    split()
    _, plain_ms = cuda_time_ms(plain, 2, stream)
    _, cp_ms = cuda_time_ms(split, 3, stream)
    check = None
    if keep:
        out, fin = prefill_cp(*args, seg_len=seg_len, lengths=[T], stream=stream)
        hs = [0, 3, 5, 7][: heads]
        idx = torch.tensor(hs, device=dev)
        check = {"heads": hs, "ckpt_stride": 0,
                 "inputs": {k_: x[k_].index_select(1, idx).cpu() for k_ in ("q", "k", "v", "g", "beta")},
                 "cu": torch.tensor([0, T], dtype=torch.int64), "init": None,
                 "out": out.index_select(1, idx).cpu(), "final": fin.index_select(1, idx).cpu(),
                 "ckpts": None}
        del out, fin
    del x, args
    # the scan alone, on states of the same shape (its time does not depend on the values)
    n_seg = -(-T // seg_len)
    gen = torch.Generator(device=dev).manual_seed(10)
    s_loc = torch.randn(n_seg, heads, D, D, device=dev, generator=gen)
    m = torch.randn(n_seg, heads, D, D, device=dev, generator=gen) / D ** 0.5
    s_start = torch.empty_like(s_loc)
    seq_seg = torch.tensor([0, n_seg], dtype=torch.int32, device=dev)

    def scan():
        cp_combine(s_loc, m, seq_seg, s_start, stream=stream)

    for _ in range(3):
        scan()
    _, scan_ms = cuda_time_ms_queued(scan, 10, stream)
    del s_loc, m
    # the output correction alone: every segment but the first; its bytes are u read and the
    # outputs read and written, fp32
    u = torch.randn(T, heads, D, device=dev, generator=gen)
    o = torch.zeros(T, heads, D, device=dev)
    cu_seg = torch.tensor(list(range(0, T, seg_len)) + [T], dtype=torch.int32, device=dev)

    def correct():
        cp_correct(o, u, s_start, cu_seg, [0], stream=stream)

    correct()
    _, corr_ms = cuda_time_ms(correct, 5, stream)
    corr_bytes = (T - min(seg_len, T)) * heads * D * 4 * 3
    del u, o, s_start
    fig = {"workload": f"one sequence T={T} H={heads} d={D} bf16, fp32 out and final state; "
                       f"segments of {seg_len} tokens",
           "plain_ms": plain_ms, "cp_ms": cp_ms, "speedup": plain_ms / cp_ms,
           "scan_ms": scan_ms, "scan_segments": n_seg,
           "correct_ms": corr_ms, "correct_GB/s": corr_bytes / (corr_ms / 1e3) / 1e9,
           "cp_tokens_per_s": T / (cp_ms / 1e3), "plain_tokens_per_s": T / (plain_ms / 1e3)}
    if hbm_peak:
        fig["correct_frac"] = fig["correct_GB/s"] / hbm_peak
    if check is not None:
        fig["_check"] = check
    return fig


def kbuild_source_hash() -> str:
    """Hash of the prefill kernel sources: a stored ncu traffic figure applies only to them."""
    import hashlib

    from kimi_delta_attention_13_gb300 import build as kbuild

    h = hashlib.sha256()
    for p in kbuild.sources():
        if "prefill" in os.path.basename(p) or "internal" in os.path.basename(p):
            with open(p, "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=H,
                    help="head count of every workload (default 96; smaller values make a short "
                         "case for profiling)")
    args = ap.parse_args()
    set_heads(args.heads)
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
