"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and nothing else: it holds none of the
mixer's arithmetic, so the CUDA path and the CPU oracle can both consume the
exact same buffers without sharing any code that computes the method.

Workload shapes follow the paper's setups ("2Mamba2Furious", App. B: heads of
dimension 64, 16 heads in the small model; Sec. 5 / App. B: sequence lengths
2048, 4096 and 8192).  The paper trains on text; no dataset is needed for the
mixer, whose inputs are the post-projection q, k, v and the A-mask input a, so
these are Gaussian draws.

Draw order for one workload: q, k, v, a, dO (then S0 for decode), each
``torch.randn(shape, dtype=float64, generator=g)`` from one
``torch.Generator('cpu').manual_seed(seed)``; then scaled, cast to fp32 and,
for bf16 workloads, rounded to bf16.  Decode step t draws its token from a
generator seeded ``seed * 1_000_003 + t``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "fwd", "fwdbwd", "decode", "e"
    B: int = 1
    H: int = 1
    T: int = 0
    d: int = 64
    dv: int = 64
    dtype: str = "bf16"  # dtype of q, k, v, o, dO ("f32" or "bf16"); a is always fp32
    qkv_std: float = 1.0
    chunk: int | None = None
    steps: int = 0       # decode steps
    S0_std: float = 0.0  # decode initial-state std
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    1: Workload("fwd_f32_B1_H2_T256_d16", "fwd", B=1, H=2, T=256, d=16, dv=16, dtype="f32",
                qkv_std=1 / math.sqrt(16), chunk=64),
    2: Workload("fwd_bf16_B4_H16_T2048_d64", "fwd", B=4, H=16, T=2048, d=64, dv=64,
                dtype="bf16", qkv_std=1 / math.sqrt(64)),
    3: Workload("fwdbwd_bf16_B2_H16_T8192_d64", "fwdbwd", B=2, H=16, T=8192, d=64, dv=64,
                dtype="bf16", qkv_std=1 / math.sqrt(64)),
    4: Workload("decode_f32_N256_H16_d64_1000steps", "decode", B=256, H=16, d=64, dv=64,
                dtype="f32", qkv_std=1 / math.sqrt(64), steps=1000, S0_std=0.01),
    5: Workload("e_fwdbwd_bf16_B2_H16_T4096_d64", "e", B=2, H=16, T=4096, d=64, dv=64,
                dtype="bf16", qkv_std=1.0),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _round(x64: torch.Tensor, dtype: str) -> torch.Tensor:
    x = x64.to(torch.float32)
    return x.to(TORCH_DTYPE[dtype]) if dtype != "f32" else x


def sequence_inputs(B, H, T, d, dv, *, dtype="bf16", qkv_std=1.0, seed=0, with_dO=False,
                    dO_std=1.0, a_mean=0.0, a_std=1.0):
    """q,k,v (B,H,T,d|dv) in ``dtype``; a (B,H,T) fp32; optional dO (B,H,T,dv)."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = torch.randn((B, H, T, d), dtype=torch.float64, generator=g) * qkv_std
    k = torch.randn((B, H, T, d), dtype=torch.float64, generator=g) * qkv_std
    v = torch.randn((B, H, T, dv), dtype=torch.float64, generator=g) * qkv_std
    a = torch.randn((B, H, T), dtype=torch.float64, generator=g) * a_std + a_mean
    out = {"q": _round(q, dtype), "k": _round(k, dtype), "v": _round(v, dtype),
           "a": a.to(torch.float32)}
    if with_dO:
        dO = torch.randn((B, H, T, dv), dtype=torch.float64, generator=g) * dO_std
        out["dO"] = _round(dO, dtype)
    return out


def workload_inputs(wid: int, seed: int | None = None):
    """Inputs of a sequence workload (ids 1, 2, 3, 5) with the default seed = id."""
    w = WORKLOADS[wid]
    assert w.kind != "decode"
    return sequence_inputs(w.B, w.H, w.T, w.d, w.dv, dtype=w.dtype, qkv_std=w.qkv_std,
                           seed=wid if seed is None else seed,
                           with_dO=w.kind in ("fwdbwd", "e"))


def decode_initial_state(N, H, d, dv, *, S0_std=0.01, seed=4):
    """S0 (N,H,d*d,dv) fp32 ~ N(0, S0_std^2); z0 = 0 (N,H,d*d) fp32."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    S0 = (torch.randn((N, H, d * d, dv), dtype=torch.float64, generator=g) * S0_std)
    return S0.to(torch.float32), torch.zeros((N, H, d * d), dtype=torch.float32)


def decode_token(t, N, H, d, dv, *, dtype="f32", qkv_std=0.125, seed=4):
    """Token of decode step t: q,k (N,H,d), v (N,H,dv) in ``dtype``; a (N,H) fp32."""
    g = torch.Generator("cpu").manual_seed(int(seed) * 1_000_003 + int(t))
    q = torch.randn((N, H, d), dtype=torch.float64, generator=g) * qkv_std
    k = torch.randn((N, H, d), dtype=torch.float64, generator=g) * qkv_std
    v = torch.randn((N, H, dv), dtype=torch.float64, generator=g) * qkv_std
    a = torch.randn((N, H), dtype=torch.float64, generator=g)
    return {"q": _round(q, dtype), "k": _round(k, dtype), "v": _round(v, dtype),
            "a": a.to(torch.float32)}


def rel_err(x, ref) -> float:
    """max|x - ref| / RMS(ref): the parity metric, per output tensor."""
    x = torch.as_tensor(x).double().cpu()
    ref = torch.as_tensor(ref).double().cpu()
    rms = ref.pow(2).mean().sqrt().item()
    err = (x - ref).abs().max().item() if ref.numel() else 0.0
    return err / rms if rms > 0 else err
