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
# kernels launched beside another one (their event-timed span includes sharing the SMs)
OVERLAPPED = {"tc_bwd_dq": "runs beside the reverse state walk (which has stream priority); the span is "
                           "from its first to its last CTA, not its own device time",
              "tc_state_scan_fwd": "two concurrent launches per step (the heads in two halves on two streams); "
                                   "the sum of their spans exceeds the walk's wall time",
              "tc_chunk_out": "two launches per step, the first beside the second half's walk; the sum of "
                              "their spans includes that sharing"}


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


def packed_rows(d):
    """State rows of the block-packed layout the tensor-core forward walk exports (16 x 16
    blocks of the (m, n) index square with bm <= bn): 2560 of the 4096 rows at d = 64."""
    nb = d // 16
    return nb * (nb + 1) // 2 * 256


def kernel_flops(name, d, dv, C, tokens):
    """Algorithmic flops of one launch of a named kernel over `tokens` token-heads: the
    method's own work at chunk length C (causal pairs only, no recompute counted twice;
    the tensor-core kernels' hi + lo split of operands is not counted).  Both walks, the chunk
    output and dq work on the block-packed state (packed_rows of the d^2 rows: the state is
    symmetric in its two key indices); dk/dv contracts the full gradient state once (each stored
    off-diagonal block in both orientations) and takes the key term from the same product
    (2 d dv more per token)."""
    dv1 = dv + 1
    state = 2 * d * d * dv1          # one d^2 x (dv+1) contraction per token
    pstate = 2 * packed_rows(d) * dv1
    per = {
        "tc_state_scan_fwd": pstate + 2 * packed_rows(d) * dv1 / C,
        "tc_state_scan_bwd": pstate + 2 * packed_rows(d) * dv1 / C,
        "tc_chunk_out": pstate + (C + 1) * (d + dv),
        "tc_bwd_dq": pstate + (C + 1) * (d + dv),
        "tc_bwd_dkdv": state + 2 * d * dv + (C + 1) * (2 * d + dv),
        "state_scan_fwd": state + 2 * d * d * dv1 / C,
        "chunk_out": state + (C + 1) * (d + dv),
        "state_scan_bwd": state + 2 * d * d * dv1 / C,
        "bwd_chunk": 3 * state + (C + 1) * (3 * d + 2 * dv),
    }.get(name)
    return None if per is None else per * tokens


def kernel_bytes(name, d, dv, C, tokens, in_bytes=2):
    """Algorithmic HBM bytes of one launch over `tokens` token-heads: the token rows the kernel
    must read or write (inputs and the gradients dq, dk, dv in the input type, o and the
    per-token scalars in fp32), plus the chunk states it must write or read (two fp16 planes of
    d^2 x dv and the fp32 normaliser column per chunk, amortised over the C tokens of a
    chunk).  Every kernel moves the block-packed state (packed_rows of the d^2 rows; the
    normaliser stays full).  Scratch the implementation adds (operand
    blocks) is not counted."""
    state = (2 * 2 * d * d * dv + 4 * d * d) / C
    pstate = (2 * 2 * packed_rows(d) * dv + 4 * d * d) / C
    per = {
        "tc_state_scan_fwd": pstate + in_bytes * (d + dv),
        "tc_state_scan_bwd": pstate + in_bytes * (d + dv) + 4 * 2,
        "tc_chunk_out": pstate + in_bytes * (2 * d + dv) + 4 * (dv + 1),
        "tc_bwd_dq": pstate + in_bytes * (2 * d + 2 * dv) + in_bytes * d + 4 * 2,
        "tc_bwd_dkdv": pstate + in_bytes * (2 * d + 2 * dv) + in_bytes * (d + dv) + 4 * 4,
    }.get(name)
    return None if per is None else per * tokens


def decode_bytes_per_head(d, dv, packed=False):
    """Algorithmic bytes of one decode step of one (sequence, head): the fp32 state S and z read
    and written once (d^2 rows, or d(d+1)/2 symmetric-packed), the token in, y and zeta out."""
    rows = d * (d + 1) // 2 if packed else d * d
    return 2 * rows * dv * 4 + 2 * rows * 4 + 3 * d * 4 + 4 + dv * 4 + 4


def e_decode_bytes_per_head(ctx, d, dv, in_bytes=2):
    """Algorithmic bytes of one 2Mamba-E decode step of one (sequence, head) at context ctx: the
    cached keys, values and running sums read once, the new row appended, q in, o and lse out."""
    return ctx * ((d + dv) * in_bytes + 8) + (d + dv) * in_bytes + 8 + d * in_bytes + 4 + dv * 4 + 4


SUSTAINED_AFTER_MS = 1000.0   # a timed region this long runs under the power cap: sustained peak


def tensor_peak_key(timed_ms):
    """Which measured bf16 figure a tensor-core kernel is held to: the burst one for a timed
    region shorter than a second (the clocks have not settled under the power cap), the
    sustained one for a longer region."""
    return "bf16_tflops_sustained" if timed_ms >= SUSTAINED_AFTER_MS else "bf16_tflops"


def roofline(kernel, kf, kb, ms_per_launch, pk, tc, peak_key="bf16_tflops_sustained"):
    """Roofline entry of one kernel from its algorithmic flops kf and bytes kb per launch and its
    live launch time.  Tensor-core kernels are measured against the measured bf16 figure named by
    peak_key (tensor_peak_key: burst or sustained) or the HBM copy bandwidth, whichever bound takes
    longer for the kernel's algorithmic work; CUDA-core kernels against the fp32 FMA rate derived
    from the SM count and clock.  None when the kernel's work is not counted."""
    if kf is None:
        return None
    sec = ms_per_launch * 1e-3
    if tc:
        tp = pk[peak_key]
        t_flop = kf / (tp * 1e12)
        t_byte = kb / (pk["hbm_gbs"] * 1e9)
        if t_byte > t_flop:
            roof = {"kernel": kernel, "bound": "hbm", "achieved": kb / sec / 1e9, "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": kb / sec / 1e9 / pk["hbm_gbs"],
                    "peak_source": "MEASURED_PEAKS.json hbm_gbs (%s)" % pk["source"]}
        else:
            roof = {"kernel": kernel, "bound": "tensor", "achieved": kf / sec / 1e12,
                    "peak": tp, "unit": "TFLOP/s", "frac": kf / sec / 1e12 / tp,
                    "peak_source": "MEASURED_PEAKS.json %s (%s)" % (peak_key, pk["source"])}
        roof["algorithmic_flops_per_launch"] = kf
        roof["algorithmic_bytes_per_launch"] = kb
        roof["tensor_frac"] = kf / sec / 1e12 / tp
        roof["tensor_peak"] = "%s = %.1f TFLOP/s" % (peak_key, tp)
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
    """SM clock, its maximum, power and the throttle reasons, sampled during the timed region:
    about every millisecond from NVML in a thread (read-only queries; the power reading every
    eighth sample), else every 100 ms by nvidia-smi.  The samples are CSV lines in
    nvidia-smi's format either way (parse_clocks)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits: hw slowdown, hw thermal slowdown, sw thermal slowdown, sw power cap
    BITS = (0x8, 0x40, 0x20, 0x4)

    def __init__(self, device):
        self.proc = None
        self.path = None
        self.thread = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            self.gpu = str(device)

    def _nvml_loop(self, nv, h):
        # the clock and the reasons every sample; the maximum clock once and the power every
        # eighth sample (the slowest query), carried between
        smax, pw, i = None, 0.0, 0
        while not self.stop_flag:
            try:
                if smax is None:
                    smax = nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM)
                if i % 8 == 0:
                    pw = nv.nvmlDeviceGetPowerUsage(h) / 1000.0
                sm = nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM)
                r = nv.nvmlDeviceGetCurrentClocksEventReasons(h)
                flags = ["Active" if r & b else "Not Active" for b in self.BITS]
                self.lines.append("%d, %d, %.1f, %s\n" % (sm, smax, pw, ", ".join(flags)))
            except Exception:
                break
            i += 1
            time.sleep(0.0005)

    def start(self):
        self.stop_flag = False
        self.lines = []
        try:
            import threading
            import pynvml as nv
            nv.nvmlInit()
            try:
                h = nv.nvmlDeviceGetHandleByUUID(self.gpu)
            except Exception:
                h = nv.nvmlDeviceGetHandleByUUID(self.gpu.encode())
            self.thread = threading.Thread(target=self._nvml_loop, args=(nv, h), daemon=True)
            self.thread.start()
            return
        except Exception:
            self.thread = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join(timeout=5)
            return parse_clocks(self.lines)
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
            "outputs": "o fp32, gradients dq dk dv bf16 (TM2_GRADS_INPUT_DTYPE), da fp32",
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
    grads = tuple(torch.empty(g[n].shape, dtype=g[n].dtype if n != "a" else torch.float32, device=device)
                  for n in ("q", "k", "v", "a"))
    # one workspace for both calls: the backward reads the chunk states the forward left in it
    ws = torch.empty(tm2.workspace_bytes(B, H, T, d, dv, C), dtype=torch.uint8, device=device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def step(q, k, v, a, dO):
        tm2.forward(q, k, v, a, chunk=C, out=o, Z=Z, workspace=ws)
        tm2.backward(q, k, v, a, o, Z, dO, chunk=C, workspace=ws, grads=grads, reuse_states=True, lowp_grads=True)

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

    # roofline of the dominant kernel (largest share of step time), among the kernels that run
    # alone: dq runs beside the reverse walk, so its event-timed span includes that sharing
    dom = max((n for n in kern if n not in OVERLAPPED), key=lambda n: kern[n]["ms"])
    per_launch_tokens = B * H * T
    tc = dom.startswith("tc_")
    kf = kernel_flops(dom, d, dv, 256 if tc else 64, per_launch_tokens)
    kb = kernel_bytes(dom, d, dv, 256, per_launch_tokens) if tc else None
    timed_ms = step_ms * args.steps
    peak_key = tensor_peak_key(timed_ms)
    roof = roofline(dom, kf, kb, kern[dom]["ms_per_launch"], pk, tc, peak_key)
    if roof is not None:
        roof["traffic"] = ncu_traffic(dom, per_launch_tokens)
    CH = TC_CHUNK
    counted = (fwd_flops(d, dv, CH) + bwd_flops(d, dv, CH)) * B * H * T
    tensor_frac = counted / (step_ms * 1e-3) / (pk[peak_key] * 1e12)
    per_kernel_roof = {}
    for n, a in kern.items():
        if n.startswith("tc_"):
            # per step: every tc kernel covers the step's B H T token-heads once, in one launch
            # or (the split forward) two; the time is the sum of its launches' spans per step
            r = roofline(n, kernel_flops(n, d, dv, 256, per_launch_tokens), kernel_bytes(n, d, dv, 256, per_launch_tokens),
                         a["ms"] / args.steps, pk, True, peak_key)
            if r is not None:
                per_kernel_roof[n] = {"bound": r["bound"], "frac": round(r["frac"], 4),
                                      "tensor_frac": round(r["tensor_frac"], 4), "hbm_frac": round(r["hbm_frac"], 4)}
                if n in OVERLAPPED:
                    per_kernel_roof[n]["note"] = OVERLAPPED[n]

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_of(w, CH), "roofline": roof,
            "step_bf16_tensor_peak_frac": tensor_frac,
            "step_tensor_peak": "%s of MEASURED_PEAKS.json (%s): timed region %.0f ms (%s a second)" % (
                peak_key, pk["source"], timed_ms, "over" if timed_ms >= SUSTAINED_AFTER_MS else "under"),
            "kernel_roofline": per_kernel_roof,
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
    if not args.no_decode:
        line["e_decode"] = run_e_decode(args, tm2, device, trace, pk, world)
    if not args.no_quadratic:
        line["quadratic_form"] = run_quadratic(args, tm2, device, trace, pk, world)
    if not args.no_conv:
        line["conv"] = run_conv(args, tm2, device, trace, pk, world)
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
    out_types = {"o": torch.float32, "dq": inp_cpu["q"].dtype, "dk": inp_cpu["k"].dtype, "dv": inp_cpu["v"].dtype,
                 "da": torch.float32}
    host_out = [{n: torch.empty(inp_cpu[src].shape, dtype=out_types[n]).pin_memory()
                 for n, src in (("o", "v"), ("dq", "q"), ("dk", "k"), ("dv", "v"), ("da", "a"))} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in[0].values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    dev_in = [{k: torch.empty(v.shape, dtype=v.dtype, device=device) for k, v in inp_cpu.items()} for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_used = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    B0, H0, T0, d0 = inp_cpu["q"].shape
    ws = torch.empty(tm2.workspace_bytes(B0, H0, T0, d0, inp_cpu["v"].shape[-1], C), dtype=torch.uint8,
                     device=device)   # one workspace: the backward reads the forward's chunk states
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
                o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"], chunk=C, workspace=ws)
                dq, dk, dv, da = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], chunk=C, workspace=ws,
                                              reuse_states=True, lowp_grads=True)
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
                        "moves its own inputs and results (o and da fp32, dq dk dv bf16); the backward "
                        "reuses the forward's chunk states"}


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
    out = {"workload": "decode step, N=%d sequences x H=%d, d=dv=%d, fp32 state, %d steps" % (N, H, d, n),
           "ms_per_step": ms, "kernel_ms_per_launch": kms, "bytes_per_step": nbytes,
           "GBps": world * nbytes / (ms * 1e-3) / 1e9, "unit": "GB/s",
           "roofline": {"kernel": "decode_step", "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"],
                        "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                        "traffic": ncu_traffic("decode_step", N * H)},
           "tokens_per_s": world * N / (ms * 1e-3), "l2": "state (4.3 GB) larger than L2",
           "gpu_launches": len(recs)}
    # the same workload on the symmetric-packed state (the outputs are the full state's)
    Sp, zp = tm2.state_pack(S, z)
    del S, z
    torch.cuda.synchronize()
    for t in range(3):
        x = toks[t % 8]
        tm2.step(x["q"], x["k"], x["v"], x["a"], Sp, zp, packed=True, out=o, Z=Zo)
    torch.cuda.synchronize()
    barrier(world)
    trace.start()
    ev0.record()
    for t in range(n):
        x = toks[t % 8]
        tm2.step(x["q"], x["k"], x["v"], x["a"], Sp, zp, packed=True, out=o, Z=Zo)
    ev1.record()
    torch.cuda.synchronize()
    recs = trace.stop()
    pms = max_over_ranks(ev0.elapsed_time(ev1) / n, world)
    pkms = sum(m for _, m in recs) / max(len(recs), 1)
    pbytes = decode_bytes_per_head(d, dv, packed=True) * N * H
    pgbs = pbytes / (pkms * 1e-3) / 1e9
    out["packed"] = {"ms_per_step": pms, "kernel_ms_per_launch": pkms, "bytes_per_step": pbytes,
                     "tokens_per_s": world * N / (pms * 1e-3),
                     "effective_GBps": world * nbytes / (pms * 1e-3) / 1e9,
                     "roofline": {"kernel": "decode_step_packed", "bound": "hbm", "achieved": pgbs,
                                  "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": pgbs / pk["hbm_gbs"],
                                  "traffic": ncu_traffic("decode_step_packed", N * H)},
                     "note": "symmetric-packed state (d(d+1)/2 of d^2 rows); effective_GBps counts the full "
                             "state's bytes, roofline the bytes actually moved"}
    return out


def conv_bytes_per_element(backward=False):
    """Algorithmic bytes per (b, h, t, channel) element of the size-2 input convolution with bf16
    tensors: forward x in, y out; backward dy in and fp32 dx out (dx pass), x and dy in (weight
    gradient pass).  The weights, biases and per-head gradients are negligible."""
    return (2 + 4) + (2 + 2) if backward else 2 + 2


def run_conv(args, tm2, device, trace, pk, world):
    """The size-2 input convolution over q, k and v at the main workload's shape (forward), its
    backward for one tensor, and the decode step with the fused convolution."""
    w = si.WORKLOADS[3]
    B, H, T, C = w.B, w.H, w.T, w.d
    gen = torch.Generator(device).manual_seed(7)
    xs = [torch.randn(B, H, T, C, generator=gen, device=device).to(torch.bfloat16) for _ in range(3)]
    dy = torch.randn(B, H, T, C, generator=gen, device=device).to(torch.bfloat16)
    wt = torch.randn(H, C, 2, generator=gen, device=device) * 0.7
    bt = torch.randn(H, C, generator=gen, device=device) * 0.1
    n = max(args.steps, 10)

    def timed(fn, name):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        barrier(world)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        trace.start()
        ev0.record()
        for _ in range(n):
            fn()
        ev1.record()
        torch.cuda.synchronize()
        recs = [m for nm, m in trace.stop() if nm == name]
        return max_over_ranks(ev0.elapsed_time(ev1) / n, world), sum(recs) / max(len(recs), 1), len(recs)

    fwd_ms, fwd_kms, nf = timed(lambda: [tm2.conv2_forward(x, wt, bt) for x in xs], "conv2_fwd")
    bwd_ms, bwd_kms, nb = timed(lambda: tm2.conv2_backward(xs[0], wt, dy), "conv2_bwd")
    elems = B * H * T * C
    fb, bb = conv_bytes_per_element() * elems, conv_bytes_per_element(True) * elems
    out = {"workload": "size-2 input convolution, B=%d H=%d T=%d C=%d bf16: forward of q, k, v; backward of one "
                       "tensor (dx, dw, db); %d steps" % (B, H, T, C, n),
           "fwd_ms_per_step": fwd_ms, "bwd_ms_per_step": bwd_ms,
           "roofline_fwd": {"kernel": "conv2_fwd", "bound": "hbm", "achieved": fb / (fwd_kms * 1e-3) / 1e9,
                            "peak": pk["hbm_gbs"], "unit": "GB/s",
                            "frac": fb / (fwd_kms * 1e-3) / 1e9 / pk["hbm_gbs"], "traffic": None},
           "roofline_bwd": {"kernel": "conv2_bwd (dx and weight-gradient passes)", "bound": "hbm",
                            "achieved": bb / (bwd_kms * 1e-3) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                            "frac": bb / (bwd_kms * 1e-3) / 1e9 / pk["hbm_gbs"], "traffic": None},
           "gpu_launches": nf + 2 * nb}
    del xs, dy
    # decode step with the fused convolution against the plain step, the decode workload's shape
    wd = si.WORKLOADS[4]
    N, d = wd.B, wd.d
    S, z = si.decode_initial_state(N, wd.H, d, d, S0_std=wd.S0_std)
    S, z = S.to(device), z.to(device)
    tok = {k: v.to(device) for k, v in si.decode_token(0, N, wd.H, d, d, qkv_std=wd.qkv_std).items()}
    cw = tuple(torch.randn(wd.H, d, 2, generator=gen, device=device) * 0.7 for _ in range(3))
    cb = tuple(torch.randn(wd.H, d, generator=gen, device=device) * 0.1 for _ in range(3))
    caches = tuple(torch.zeros(N, wd.H, d, device=device) for _ in range(3))
    o = torch.empty((N, wd.H, d), dtype=torch.float32, device=device)
    Zo = torch.empty((N, wd.H), dtype=torch.float32, device=device)
    conv_ms, conv_kms, _ = timed(lambda: tm2.step_conv(tok["q"], tok["k"], tok["v"], tok["a"], cw, cb, caches, S, z,
                                                       out=o, Z=Zo), "decode_step_conv")
    dbytes = decode_bytes_per_head(d, d) * N * wd.H
    out["decode_step_conv"] = {"ms_per_step": conv_ms, "kernel_ms_per_launch": conv_kms,
                               "roofline": {"kernel": "decode_step (fused convolution)", "bound": "hbm",
                                            "achieved": dbytes / (conv_kms * 1e-3) / 1e9, "peak": pk["hbm_gbs"],
                                            "unit": "GB/s", "frac": dbytes / (conv_kms * 1e-3) / 1e9 / pk["hbm_gbs"],
                                            "traffic": None},
                               "note": "N=%d x H=%d, d=%d, fp32 state; bytes as the plain step (the caches add "
                                       "3 x N x H x d x 8 B)" % (N, wd.H, d)}
    return out


def run_e_decode(args, tm2, device, trace, pk, world):
    """2Mamba-E decoding over a bf16 KV cache: 64 sequences x 16 heads, d = dv = 64, the token at
    position 8191 attends over 8192 cached keys (2.1 GB of cache, larger than L2)."""
    N, H, d, ctx = 64, 16, 64, 8192
    g = torch.Generator(device).manual_seed(rank_seed(6, 0))   # cache drawn on the device (2 GB)
    Kc = torch.randn(N, H, ctx, d, generator=g, device=device).to(torch.bfloat16)
    Vc = torch.randn(N, H, ctx, d, generator=g, device=device).to(torch.bfloat16)
    cc = torch.cumsum(-torch.nn.functional.softplus(torch.randn(N, H, ctx, generator=g, device=device)), -1)
    cum = torch.stack([cc, torch.zeros_like(cc)], -1).contiguous()
    tok = {k: v.to(device) for k, v in si.decode_token(0, N, H, d, d, dtype="bf16", qkv_std=1.0, seed=6).items()}
    o = torch.empty((N, H, d), dtype=torch.float32, device=device)
    lse = torch.empty((N, H), dtype=torch.float32, device=device)
    ws = torch.empty(tm2.lib().tm2e_step_workspace(N, H, ctx, d, d, 1), dtype=torch.uint8, device=device)
    pos = ctx - 1
    for _ in range(3):
        tm2.e_step(tok["q"], tok["k"], tok["v"], tok["a"], Kc, Vc, cum, pos, out=o, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    n = max(args.steps, 10)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    trace.start()
    ev0.record()
    for _ in range(n):
        tm2.e_step(tok["q"], tok["k"], tok["v"], tok["a"], Kc, Vc, cum, pos, out=o, lse=lse, workspace=ws)
    ev1.record()
    torch.cuda.synchronize()
    recs = trace.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / n, world)
    nbytes = e_decode_bytes_per_head(ctx, d, d) * N * H
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "2Mamba-E decode over a bf16 KV cache, N=%d sequences x H=%d, d=dv=%d, context %d, %d steps"
                        % (N, H, d, ctx, n),
            "ms_per_step": ms, "bytes_per_step": nbytes, "tokens_per_s": world * N / (ms * 1e-3),
            "roofline": {"kernel": "e_decode", "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"], "traffic": ncu_traffic("e_decode", N * H)},
            "kernels": {nm: round(a["ms"], 3) for nm, a in summarize(recs).items()}, "gpu_launches": len(recs)}


def run_quadratic(args, tm2, device, trace, pk, world):
    """The quadratic (C = T) form against the chunked form: the forward workload B=4 H=16 T=2048
    (bf16, d = dv = 64) and fwd+bwd at B=2 H=16 T=4096; tokens/s of each and the faster one."""
    out = {}
    for label, wid, bwd in (("fwd_B4_H16_T2048", 2, False), ("fwdbwd_B2_H16_T4096", 5, True)):
        w = si.WORKLOADS[wid]
        inp = si.sequence_inputs(w.B, w.H, w.T, 64, 64, dtype="bf16", qkv_std=0.125, seed=rank_seed(wid, 0),
                                 with_dO=bwd)
        g = {k: v.to(device) for k, v in inp.items()}
        ws = torch.empty(tm2.workspace_bytes(w.B, w.H, w.T, 64, 64), dtype=torch.uint8, device=device)

        def chunked():
            o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"], workspace=ws)
            if bwd:
                tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], workspace=ws, reuse_states=True)

        def quadratic():
            o, Z = tm2.forward_quadratic(g["q"], g["k"], g["v"], g["a"])
            if bwd:
                tm2.backward_quadratic(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"])

        res = {}
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        for name, fn in (("chunked", chunked), ("quadratic", quadratic)):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            n = max(1, min(args.steps, 10))
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            barrier(world)
            for i in range(n):
                flush.zero_()
                evs[i][0].record()
                fn()
                evs[i][1].record()
            torch.cuda.synchronize()
            res[name] = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / n, world)
        T, BH = w.T, w.B * w.H
        qflops = ((T + 1) * 128 + (((T + 1) * (3 * 64 + 2 * 64)) if bwd else 0)) * BH * T
        best = min(res, key=res.get)
        out[label] = {"chunked_ms": res["chunked"], "quadratic_ms": res["quadratic"], "faster": best,
                      "tokens_per_s": world * w.B * T / (res[best] * 1e-3),
                      "quadratic_counted_flops": qflops,
                      "quadratic_bf16_tensor_peak_frac": qflops / (res["quadratic"] * 1e-3) / (pk["bf16_tflops"] * 1e12)}
    return out


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
            "counted_flops": flops,
            "bf16_tensor_peak_frac": flops / (ms * 1e-3) / (peaks()[tensor_peak_key(ms * n)] * 1e12),
            "tensor_peak": tensor_peak_key(ms * n),
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
    elif name == "fwdbwd_h16":          # B=1, H=16, T=8192: 512 MB of chunk states per walk (4x L2)
        inp = si.sequence_inputs(1, 16, 8192, 64, 64, dtype="bf16", qkv_std=0.125, seed=3, with_dO=True)
        g = {k: v.to(dev) for k, v in inp.items()}
        o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"])
        tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], lowp_grads=True)
    elif name == "decode_packed_small":   # 32 sequences x 16 heads, packed state: 272 MB
        N, H, d = 32, 16, 64
        S, z = si.decode_initial_state(N, H, d, d, S0_std=0.01)
        Sp, zp = tm2.state_pack(S.to(dev), z.to(dev))
        x = {k: v.to(dev) for k, v in si.decode_token(0, N, H, d, d, qkv_std=0.125).items()}
        for _ in range(3):
            tm2.step(x["q"], x["k"], x["v"], x["a"], Sp, zp, packed=True)
    elif name == "e_decode_small":      # 2Mamba-E decode, 16 sequences x 16 heads, context 8192: 537 MB cache
        N, H, d, ctx = 16, 16, 64, 8192
        gen = torch.Generator(dev).manual_seed(6)
        Kc = torch.randn(N, H, ctx, d, generator=gen, device=dev).to(torch.bfloat16)
        Vc = torch.randn(N, H, ctx, d, generator=gen, device=dev).to(torch.bfloat16)
        cc = torch.cumsum(-torch.nn.functional.softplus(torch.randn(N, H, ctx, generator=gen, device=dev)), -1)
        cum = torch.stack([cc, torch.zeros_like(cc)], -1).contiguous()
        x = {k: v.to(dev) for k, v in si.decode_token(0, N, H, d, d, dtype="bf16", qkv_std=1.0, seed=6).items()}
        for _ in range(3):
            tm2.e_step(x["q"], x["k"], x["v"], x["a"], Kc, Vc, cum, ctx - 1)
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
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="tm2", choices=["tm2", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-quadratic", action="store_true")
    ap.add_argument("--no-conv", action="store_true")
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
