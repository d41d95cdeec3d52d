#!/usr/bin/env python
"""Benchmark of the 2Mamba second-order mixer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tm2|reference]

One step = one pass of the whole training hot path over one synthetic batch:
forward + backward of the 2Mamba mixer at B=2, H=16, T=8192, d=dv=64, bf16 inputs,
normalised ("2Mamba2Furious" Sec. 5; App. B shapes: 16 heads of dimension 64;
sequence length 8192).  `value` is tokens/s over all ranks (weak scaling: each rank
runs its own replica on its own batch; the path has no exchange step).  The same
line carries the decode step (256 sequences x 16 heads, fp32 d^2 x dv state) in GB/s
and 2Mamba-E fwd+bwd (B=2, H=16, T=4096) in tokens/s.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events on the
launching stream; a 256 MiB buffer is written between timed steps to flush the
126 MB L2.  Per-kernel device times come from the library's own launch trace (CUDA
events recorded around every kernel on its stream).  Rank 0 prints one JSON line.

--impl reference times the CPU fp64 oracle (the only executable reference of this
method; the paper's code is not available) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
import synth_inputs as si  # noqa: E402

METRIC = "2Mamba fwd+bwd tokens/s at T=8192 on 1 B300; % bf16 tensor peak; decode GB/s"
FLUSH_BYTES = 256 << 20


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "sm_max_mhz": p.get("sm_max_mhz", 2032.0), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "sm_max_mhz": 2032.0, "source": "fallback"}


# ----------------------------------------------------------------------------- counting
def fwd_flops(d, dv, C, normalize=True):
    """Algorithmic flops per token-head of the chunked forward (causal pairs only)."""
    dv1 = dv + 1 if normalize else dv
    return 4 * d * d * dv1 + (C + 1) * (d + dv) + 2 * d * d * dv1 / C


def bwd_flops(d, dv, C, normalize=True):
    dv1 = dv + 1 if normalize else dv
    return 8 * d * d * dv1 + (C + 1) * (3 * d + 2 * dv) + 4 * d * d * dv1 / C


def kernel_flops(name, d, dv, C, tokens):
    """Algorithmic flops of one launch of a named kernel over `tokens` token-heads: the
    method's own work at chunk length C (causal pairs only, no recompute counted twice;
    the tensor-core kernels' hi + lo split of operands is not counted)."""
    dv1 = dv + 1
    state = 2 * d * d * dv1          # one d^2 x (dv+1) contraction per token
    per = {
        "tc_state_scan_fwd": state + 2 * d * d * dv1 / C,
        "tc_state_scan_bwd": state + 2 * d * d * dv1 / C,
        "tc_chunk_out": state + (C + 1) * (d + dv),
        "tc_bwd_dq": state + (C + 1) * (d + dv),
        "tc_bwd_dkdv": 2 * state + (C + 1) * (2 * d + dv),
        "state_scan_fwd": state + 2 * d * d * dv1 / C,
        "chunk_out": state + (C + 1) * (d + dv),
        "state_scan_bwd": state + 2 * d * d * dv1 / C,
        "bwd_chunk": 3 * state + (C + 1) * (3 * d + 2 * dv),
    }.get(name)
    return None if per is None else per * tokens


def kernel_bytes(name, d, dv, C, tokens, in_bytes=2):
    """Algorithmic HBM bytes of one launch over `tokens` token-heads: the token rows the kernel
    must read or write, plus the chunk states it must write or read (two fp16 planes of
    d^2 x dv and the fp32 normaliser column per chunk, amortised over the C tokens of a
    chunk).  Scratch the implementation adds (operand blocks) is not counted."""
    state = (2 * 2 * d * d * dv + 4 * d * d) / C
    per = {
        "tc_state_scan_fwd": state + in_bytes * (d + dv),
        "tc_state_scan_bwd": state + in_bytes * (d + dv) + 4 * 2,
        "tc_chunk_out": state + in_bytes * (2 * d + dv) + 4 * (dv + 1),
        "tc_bwd_dq": state + in_bytes * (2 * d + 2 * dv) + 4 * (d + 2),
        "tc_bwd_dkdv": state + in_bytes * (2 * d + 2 * dv) + 4 * (d + dv + 4),
    }.get(name)
    return None if per is None else per * tokens


def decode_bytes_per_head(d, dv):
    return 2 * d * d * dv * 4 + 2 * d * d * 4 + 3 * d * 4 + 4 + dv * 4 + 4


def roofline(kernel, kf, kb, ms_per_launch, pk, tc):
    """Roofline entry of one kernel from its algorithmic flops kf and bytes kb per launch and its
    live launch time.  Tensor-core kernels (timed inside a long step) are measured against the
    sustained bf16 figure or the HBM copy bandwidth, whichever bound takes longer for the
    kernel's algorithmic work; CUDA-core kernels against the fp32 FMA rate derived from the SM
    count and clock.  None when the kernel's work is not counted."""
    if kf is None:
        return None
    sec = ms_per_launch * 1e-3
    if tc:
        t_flop = kf / (pk["bf16_tflops_sustained"] * 1e12)
        t_byte = kb / (pk["hbm_gbs"] * 1e9)
        if t_byte > t_flop:
            roof = {"kernel": kernel, "bound": "hbm", "achieved": kb / sec / 1e9, "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": kb / sec / 1e9 / pk["hbm_gbs"],
                    "peak_source": "MEASURED_PEAKS.json hbm_gbs (%s)" % pk["source"]}
        else:
            roof = {"kernel": kernel, "bound": "tensor", "achieved": kf / sec / 1e12,
                    "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                    "frac": kf / sec / 1e12 / pk["bf16_tflops_sustained"],
                    "peak_source": "MEASURED_PEAKS.json bf16_tflops_sustained (%s)" % pk["source"]}
        roof["algorithmic_flops_per_launch"] = kf
        roof["algorithmic_bytes_per_launch"] = kb
        roof["tensor_frac"] = kf / sec / 1e12 / pk["bf16_tflops_sustained"]
        roof["hbm_frac"] = kb / sec / 1e9 / pk["hbm_gbs"]
        return roof
    peak = 148 * 128 * 2 * pk["sm_max_mhz"] * 1e6 / 1e12   # FFMA, TFLOP/s
    return {"kernel": kernel, "bound": "alu", "achieved": kf / sec / 1e12, "peak": peak, "unit": "TFLOP/s",
            "frac": kf / sec / 1e12 / peak,
            "peak_source": "derived: 148 SMs x 128 fp32 FMA/clk x 2 flop x %.0f MHz" % pk["sm_max_mhz"],
            "algorithmic_flops_per_launch": kf}


# ----------------------------------------------------------------------------- tracing
class Trace:
    def __init__(self, lib):
        self.lib = lib
        lib.tm2_trace_enable.argtypes = [ctypes.c_int]
        lib.tm2_trace_read.argtypes = [ctypes.c_int, ctypes.c_char_p, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_float)]

    def start(self):
        self.lib.tm2_trace_enable(1)

    def stop(self):
        self.lib.tm2_trace_enable(0)
        out = []
        buf = ctypes.create_string_buffer(64)
        ms = ctypes.c_float()
        for i in range(self.lib.tm2_trace_count()):
            if self.lib.tm2_trace_read(i, buf, 64, ctypes.byref(ms)) == 0:
                out.append((buf.value.decode(), float(ms.value)))
        return out


def summarize(trace):
    agg = {}
    for name, ms in trace:
        a = agg.setdefault(name, {"launches": 0, "ms": 0.0})
        a["launches"] += 1
        a["ms"] += ms
    tot = sum(a["ms"] for a in agg.values()) or 1.0
    for a in agg.values():
        a["share"] = a["ms"] / tot
        a["ms_per_launch"] = a["ms"] / a["launches"]
    return agg


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.gpu = str(device)

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            out = parse_clocks(f)
        os.unlink(self.path)
        return out


def parse_clocks(lines):
    """Summary of `nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,nounits`
    samples: median SM clock, the highest max-clock reading, and every throttle reason seen
    Active in any sample (None when no sample parsed)."""
    sm, smax, reasons = [], 0.0, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 7:
            continue
        try:
            sm.append(float(parts[0]))
            smax = max(smax, float(parts[1]))
        except ValueError:
            continue
        for n, v in zip(names, parts[3:7]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
            "samples": len(sm)}


# ----------------------------------------------------------------------------- helpers
def file_sha(name):
    path = os.path.join(ROOT, "ssm_sequence_mixer_chunked_b300", "csrc", name)
    with open(path, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def ncu_traffic(kernel, units_per_launch):
    """DRAM bytes (read + write) per launch of `kernel`, scaled from the committed ncu
    capture (profiles/ncu_traffic.json) by the units the launch processes -- or None when
    there is no capture or the kernel's source file changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel)
        if not rec or rec.get("file_sha") != file_sha(rec["file"]):
            return None
    except (OSError, ValueError, KeyError):
        return None
    return rec["dram_bytes_per_unit"] * units_per_launch


def setup_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, torch.device("cuda", torch.cuda.current_device())


def max_over_ranks(x, world, device="cuda"):
    """Largest value of x over all ranks (the step time the whole job waits for)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base, rank):
    """Seed of the synthetic batch of `rank`: every rank runs its own replica on its own
    batch (the (b, h) problems are independent, so nothing is exchanged)."""
    return base + 1000 * rank


def whole_job_rate(units_per_rank, world, max_ms):
    """Units per second of the whole job: all ranks' units over the slowest rank's time."""
    return world * units_per_rank / (max_ms * 1e-3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle
def oracle_fwd_bwd_sample(inp, heads):
    import oracle
    t0 = time.perf_counter()
    for b, h in heads:
        sel = (slice(b, b + 1), slice(h, h + 1))
        q, k, v, a, dO = (inp[n][sel] for n in ("q", "k", "v", "a", "dO"))
        oracle.fwd_quadratic(q, k, v, a, True)
        oracle.bwd_quadratic(q, k, v, a, dO, True)
    return time.perf_counter() - t0


def cpu_baseline(inp, w):
    import oracle
    heads = [(0, 0), (1, 7)]
    dt = oracle_fwd_bwd_sample(inp, heads)
    frac = len(heads) / (w.B * w.H)
    return {"value": frac * w.B * w.T / dt, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": "fp64 quadratic-form forward+backward of %d of the %d (b,h) heads at full "
                      "T=%d (%.1f s); tokens/s scaled by the head fraction" % (len(heads), w.B * w.H, w.T, dt)}


# ----------------------------------------------------------------------------- arms
def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    w = si.WORKLOADS[3]
    inp = si.workload_inputs(3)
    heads = [(0, 0)]
    for _ in range(min(args.warmup, 1)):
        oracle_fwd_bwd_sample(inp, heads)
    times = [oracle_fwd_bwd_sample(inp, heads) for _ in range(args.steps)]
    step_s = sum(times) / len(times)
    frac = len(heads) / (w.B * w.H)
    value = frac * w.B * w.T / step_s
    sample = ("fp64 quadratic-form forward+backward of 1 of the %d (b,h) heads at full T=%d per step; "
              "tokens/s scaled by the head fraction" % (w.B * w.H, w.T))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_s * 1e3 / frac, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, TC_CHUNK),
            "cpu_baseline": {"kind": "oracle", "cores": oracle.num_threads(), "sample": sample,
                             "value": value, "unit": "tokens/s"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


TC_CHUNK = 256   # the chunk length the library picks for bf16 inputs with d = dv = 64


def config_of(w, C):
    return {"workload": "2Mamba forward+backward, B=%d H=%d T=%d d=dv=%d, bf16 inputs, fp32 "
                        "accumulate, normalised" % (w.B, w.H, w.T, w.d),
            "B": w.B, "H": w.H, "T": w.T, "d": w.d, "dv": w.dv, "chunk": C,
            "global_batch": w.B, "seq_len": w.T, "parallelism": "replicas (one per GPU)",
            "l2": "flushed between timed steps (256 MiB write)"}


def run_tm2(args, world, rank, device):
    import ssm_sequence_mixer_chunked_b300 as tm2
    lib = tm2.lib()
    trace = Trace(lib)
    pk = peaks()
    w = si.WORKLOADS[3]
    C = 0   # library choice: the tensor-core path wherever it applies
    inp_cpu = si.workload_inputs(3, seed=rank_seed(3, rank))
    g = {k: v.to(device) for k, v in inp_cpu.items()}
    B, H, T, d, dv = w.B, w.H, w.T, w.d, w.dv
    o = torch.empty(g["v"].shape, dtype=torch.float32, device=device)
    Z = torch.empty((B, H, T), dtype=torch.float32, device=device)
    grads = tuple(torch.empty(g[n].shape, dtype=torch.float32, device=device) for n in ("q", "k", "v", "a"))
    # one workspace for both calls: the backward reads the chunk states the forward left in it
    ws = torch.empty(tm2.workspace_bytes(B, H, T, d, dv, C), dtype=torch.uint8, device=device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def step(q, k, v, a, dO):
        tm2.forward(q, k, v, a, chunk=C, out=o, Z=Z, workspace=ws)
        tm2.backward(q, k, v, a, o, Z, dO, chunk=C, workspace=ws, grads=grads, reuse_states=True)

    for _ in range(args.warmup):
        step(g["q"], g["k"], g["v"], g["a"], g["dO"])
    torch.cuda.synchronize()

    clocks = ClockSampler(device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    trace.start()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record()
        step(g["q"], g["k"], g["v"], g["a"], g["dO"])
        evs[i][1].record()
    torch.cuda.synchronize()
    recs = trace.stop()
    barrier(world)
    clk = clocks.stop()
    step_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    step_ms = max_over_ranks(step_ms, world)
    tokens = B * T
    value = whole_job_rate(tokens, world, step_ms)
    kern = summarize(recs)
    launches = len(recs)

    # roofline of the dominant kernel (largest share of step time)
    dom = max(kern, key=lambda n: kern[n]["ms"])
    per_launch_tokens = B * H * T
    tc = dom.startswith("tc_")
    kf = kernel_flops(dom, d, dv, 256 if tc else 64, per_launch_tokens)
    kb = kernel_bytes(dom, d, dv, 256, per_launch_tokens) if tc else None
    roof = roofline(dom, kf, kb, kern[dom]["ms_per_launch"], pk, tc)
    if roof is not None:
        roof["traffic"] = ncu_traffic(dom, per_launch_tokens)
    CH = TC_CHUNK
    counted = (fwd_flops(d, dv, CH) + bwd_flops(d, dv, CH)) * B * H * T
    tensor_frac = counted / (step_ms * 1e-3) / (pk["bf16_tflops_sustained"] * 1e12)

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_of(w, CH), "roofline": roof,
            "step_bf16_tensor_peak_frac": tensor_frac,
            "step_tensor_peak": "bf16_tflops_sustained of MEASURED_PEAKS.json (%s)" % pk["source"],
            "step_counted_flops": counted, "gpu_launches": launches,
            "kernels": {n: {k: round(v, 4) if isinstance(v, float) else v for k, v in a.items()}
                        for n, a in kern.items()},
            "clocks": clk}

    if not args.no_e2e:
        line["e2e"] = run_e2e(args, tm2, inp_cpu, device, C, world)
    if not args.no_decode:
        line["decode"] = run_decode(args, tm2, device, trace, pk, world)
    if not args.no_e:
        line["e_variant"] = run_e_variant(args, tm2, device, trace, world)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(inp_cpu, w)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, tm2, inp_cpu, device, C, world):
    """Same metric through the public API with host buffers: every step copies its inputs from
    pinned host memory to the device and its results (o and all gradients) back to pinned host
    memory, inside the timed region.  Steps are pipelined the way an input pipeline feeds a
    model: step i+1's inputs travel in and step i-1's results travel out while step i computes
    (three streams, double-buffered device inputs and host outputs)."""
    host_in = [{k: v.pin_memory() for k, v in inp_cpu.items()} for _ in range(2)]
    host_out = [{n: torch.empty(inp_cpu[src].shape, dtype=torch.float32).pin_memory()
                 for n, src in (("o", "v"), ("dq", "q"), ("dk", "k"), ("dv", "v"), ("da", "a"))} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    dev_in = [{k: torch.empty(v.shape, dtype=v.dtype, device=device) for k, v in inp_cpu.items()} for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_used = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    for e in ev_used:
        e.record(torch.cuda.current_stream())

    def run(n):
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):               # inputs of step i (buffer b free once step i-2 is done)
                s_in.wait_event(ev_used[b])
                for k, t in host_in[b].items():
                    dev_in[b][k].copy_(t, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[b])
                g = dev_in[b]
                o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"], chunk=C)
                dq, dk, dv, da = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], chunk=C)
                ev_used[b].record(s_comp)
                ev_done[b].record(s_comp)
            with torch.cuda.stream(s_out):              # results of step i (host buffer b free once step i-2's are out)
                s_out.wait_event(ev_done[b])
                for name, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv), ("da", da)):
                    host_out[b][name].copy_(t, non_blocking=True)
                    t.record_stream(s_out)              # not reused before its copy has run
        cur = torch.cuda.current_stream()
        for st in (s_in, s_comp, s_out):
            cur.wait_stream(st)

    run(2)
    torch.cuda.synchronize()
    n = max(2, min(args.steps, 6))
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    run(n)
    t1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / n, world)
    B, T = inp_cpu["a"].shape[0], inp_cpu["a"].shape[2]
    return {"value": world * B * T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "pipeline": "copy-in / compute / copy-out on three streams, double-buffered; every step "
                        "moves its own inputs and results"}


def run_decode(args, tm2, device, trace, pk, world):
    w = si.WORKLOADS[4]
    N, H, d, dv = w.B, w.H, w.d, w.dv
    S, z = si.decode_initial_state(N, H, d, dv, S0_std=w.S0_std)
    S, z = S.to(device), z.to(device)
    toks = [{k: v.to(device) for k, v in si.decode_token(t, N, H, d, dv, qkv_std=w.qkv_std).items()}
            for t in range(8)]
    o = torch.empty((N, H, dv), dtype=torch.float32, device=device)
    Zo = torch.empty((N, H), dtype=torch.float32, device=device)
    for t in range(3):
        x = toks[t % 8]
        tm2.step(x["q"], x["k"], x["v"], x["a"], S, z, out=o, Z=Zo)
    torch.cuda.synchronize()
    n = max(args.steps, 10)
    barrier(world)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    trace.start()
    ev0.record()
    for t in range(n):
        x = toks[t % 8]
        tm2.step(x["q"], x["k"], x["v"], x["a"], S, z, out=o, Z=Zo)
    ev1.record()
    torch.cuda.synchronize()
    recs = trace.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / n, world)
    kms = sum(m for _, m in recs) / max(len(recs), 1)
    nbytes = decode_bytes_per_head(d, dv) * N * H
    gbs = nbytes / (kms * 1e-3) / 1e9
    return {"workload": "decode step, N=%d sequences x H=%d, d=dv=%d, fp32 state, %d steps" % (N, H, d, n),
            "ms_per_step": ms, "kernel_ms_per_launch": kms, "bytes_per_step": nbytes,
            "GBps": world * nbytes / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "roofline": {"kernel": "decode_step", "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                         "traffic": ncu_traffic("decode_step", N * H)},
            "tokens_per_s": world * N / (ms * 1e-3), "l2": "state (4.3 GB) larger than L2",
            "gpu_launches": len(recs)}


def run_e_variant(args, tm2, device, trace, world):
    w = si.WORKLOADS[5]
    inp = si.workload_inputs(5)
    g = {k: v.to(device) for k, v in inp.items()}
    B, H, T, d, dv = w.B, w.H, w.T, w.d, w.dv

    def step():
        o, lse = tm2.e_forward(g["q"], g["k"], g["v"], g["a"])
        tm2.e_backward(g["q"], g["k"], g["v"], g["a"], o, lse, g["dO"])

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    n = max(1, min(args.steps, 5))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    barrier(world)
    trace.start()
    for i in range(n):
        flush.zero_()
        evs[i][0].record()
        step()
        evs[i][1].record()
    torch.cuda.synchronize()
    recs = trace.stop()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / n, world)
    flops = ((T + 1) * (d + dv) + (T + 1) * (3 * d + 2 * dv)) * B * H * T
    return {"workload": "2Mamba-E forward+backward, B=%d H=%d T=%d d=dv=%d bf16" % (B, H, T, d),
            "ms_per_step": ms, "tokens_per_s": world * B * T / (ms * 1e-3),
            "counted_flops": flops, "bf16_tensor_peak_frac": flops / (ms * 1e-3) / (peaks()["bf16_tflops"] * 1e12),
            "kernels": {n: round(a["ms"], 3) for n, a in summarize(recs).items()},
            "gpu_launches": len(recs)}


def run_case(name):
    """Small fixed cases for profiler captures (few launches, a few GB at most on the
    device, working sets above the 126 MB L2).  Prints a one-line summary."""
    import ssm_sequence_mixer_chunked_b300 as tm2
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    if name == "decode_small":          # 32 sequences x 16 heads: 545 MB of state
        N, H, d = 32, 16, 64
        S, z = si.decode_initial_state(N, H, d, d, S0_std=0.01)
        S, z = S.to(dev), z.to(dev)
        x = {k: v.to(dev) for k, v in si.decode_token(0, N, H, d, d, qkv_std=0.125).items()}
        for _ in range(3):
            tm2.step(x["q"], x["k"], x["v"], x["a"], S, z)
    elif name == "fwdbwd_small":        # B=1, H=4, T=8192: chunk states well above L2
        inp = si.sequence_inputs(1, 4, 8192, 64, 64, dtype="bf16", qkv_std=0.125, seed=3, with_dO=True)
        g = {k: v.to(dev) for k, v in inp.items()}
        o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"])
        tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"])
    elif name == "e_small":             # 2Mamba-E, B=1, H=4, T=4096
        inp = si.sequence_inputs(1, 4, 4096, 64, 64, dtype="bf16", qkv_std=1.0, seed=5, with_dO=True)
        g = {k: v.to(dev) for k, v in inp.items()}
        o, lse = tm2.e_forward(g["q"], g["k"], g["v"], g["a"])
        tm2.e_backward(g["q"], g["k"], g["v"], g["a"], o, lse, g["dO"])
    else:
        raise SystemExit("unknown case " + name)
    torch.cuda.synchronize()
    print("case %s ok" % name)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="tm2", choices=["tm2", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--case", default=None, help="run one small profiling case and exit")
    args = ap.parse_args()
    if args.case:
        return run_case(args.case)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        return run_reference(args, world, rank)
    world, rank, device = setup_dist()
    run_tm2(args, world, rank, device)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
