"""GPU parity of the quadratic (C = T) form of the mixer against the fp64 oracle.

"2Mamba2Furious", Sec. 1-2: the quadratic form pays O(T^2) flops but fewer than the chunked
form below T = 8192 at d = 64; Sec. 5 (2Mamba, order 2) and Sec. 4 (the first-order mixer of
Mamba-2S, order 1).  bf16 inputs with d = dv = 64 run the tensor-core kernels, everything else
the CUDA-core kernels.  Bars: 2e-2 (bf16 inputs), 1e-4 (fp32 inputs), max|err| / RMS.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import ssm_sequence_mixer_chunked_b300 as tm2
import synth_inputs as si

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def cuda(d):
    return {k: v.cuda() for k, v in d.items()}


def gerr(x, ref, scale):
    """max|x - ref| / RMS(ref), or against `scale` where the exact tensor is zero (T = 1
    normalised: o_0 = v_0 whatever q, k, a are)."""
    r = np.asarray(ref, dtype=np.float64)
    if np.sqrt((r ** 2).mean()) <= 1e-9 * scale:
        return float((torch.as_tensor(x).double() - torch.as_tensor(r)).abs().max()) / scale
    return si.rel_err(x, ref)


def run_and_check(inp, dtype, order, normalize, heads=None):
    g = cuda(inp)
    o, Z = tm2.forward_quadratic(g["q"], g["k"], g["v"], g["a"], order=order, normalize=normalize)
    grads = tm2.backward_quadratic(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], order=order,
                                   normalize=normalize)
    torch.cuda.synchronize()
    sel = (slice(None), slice(None)) if heads is None else heads
    q, k, v, a, dO = (inp[n][sel] for n in ("q", "k", "v", "a", "dO"))
    o_ref, Z_ref = oracle.fwd_quadratic(q, k, v, a, normalize, order=order)
    refs = oracle.bwd_quadratic(q, k, v, a, dO, normalize, order=order)
    scale = float(np.sqrt((refs[2] ** 2).mean()))
    errs = {"o": si.rel_err(o.cpu()[sel], o_ref), "Z": si.rel_err(Z.cpu()[sel], Z_ref)}
    for name, x, ref in zip(("dq", "dk", "dv", "da"), grads, refs):
        errs[name] = gerr(x.cpu()[sel], ref, scale)
    bad = {k: v for k, v in errs.items() if not v <= TOL[dtype]}
    assert not bad, (dtype, order, normalize, errs)
    return o, Z, grads


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("T", [1, 64, 190, 1000])
def test_order2_tensor_core_ragged(T, normalize):
    inp = si.sequence_inputs(2, 2, T, 64, 64, dtype="bf16", qkv_std=0.125, seed=600 + T, with_dO=True)
    run_and_check(inp, "bf16", 2, normalize)


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("normalize", [True, False])
def test_order2_fp32(d, normalize):
    inp = si.sequence_inputs(1, 3, 333, d, d, dtype="f32", qkv_std=1 / math.sqrt(d), seed=610 + d, with_dO=True)
    run_and_check(inp, "f32", 2, normalize)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 130, 700])
def test_order1(dtype, T):
    """The first-order mixer (score, not its square), unnormalised as in Mamba-2S."""
    inp = si.sequence_inputs(2, 2, T, 64, 64, dtype=dtype, qkv_std=0.125, seed=620 + T, with_dO=True)
    run_and_check(inp, dtype, 1, False)


def test_order1_normalised_positive_scores():
    """Normalised first order where every score is positive (q, k drawn with a shared positive
    mean), so Z stays away from zero."""
    inp = si.sequence_inputs(1, 2, 500, 64, 64, dtype="bf16", qkv_std=0.05, seed=630, with_dO=True)
    for n in ("q", "k"):
        inp[n] = (inp[n].float() + 0.125).to(torch.bfloat16)
    run_and_check(inp, "bf16", 1, True)


@pytest.mark.parametrize("case", ["a_plus40", "a_minus40"])
def test_order2_decay_limits(case):
    inp = si.sequence_inputs(1, 2, 777, 64, 64, dtype="bf16", qkv_std=0.125, seed=640, with_dO=True)
    inp["a"] = torch.full_like(inp["a"], 40.0 if case == "a_plus40" else -40.0)
    o, _, _ = run_and_check(inp, "bf16", 2, False)
    if case == "a_plus40":   # only the diagonal weight: o_i = (q_i . k_i)^2 v_i
        s = (inp["q"].double() * inp["k"].double()).sum(-1, keepdim=True)
        assert si.rel_err(o.cpu(), s ** 2 * inp["v"].double()) <= 2e-2


def test_order2_equals_chunked_forward():
    """The quadratic form and the chunked form (tm2_forward) compute the same function."""
    inp = si.sequence_inputs(2, 4, 1500, 64, 64, dtype="bf16", qkv_std=0.125, seed=650)
    g = cuda(inp)
    oq, Zq = tm2.forward_quadratic(g["q"], g["k"], g["v"], g["a"])
    oc, Zc = tm2.forward(g["q"], g["k"], g["v"], g["a"])
    torch.cuda.synchronize()
    assert si.rel_err(oq.cpu(), oc.cpu()) <= 2e-2 and si.rel_err(Zq.cpu(), Zc.cpu()) <= 2e-2


def test_order2_fwd_B4_H16_T2048_full():
    """The forward workload B=4, H=16, T=2048, d=dv=64 (bf16), every head against the oracle."""
    inp = si.workload_inputs(2)
    g = cuda(inp)
    o, Z = tm2.forward_quadratic(g["q"], g["k"], g["v"], g["a"])
    torch.cuda.synchronize()
    o_ref, Z_ref = oracle.fwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], True)
    assert si.rel_err(o.cpu(), o_ref) <= 2e-2 and si.rel_err(Z.cpu(), Z_ref) <= 2e-2


def test_order2_fwd_bwd_B2_H16_T8192_sampled_heads():
    """fwd+bwd of the quadratic form at B=2, H=16, T=8192, d=dv=64 bf16 on the whole batch; the
    oracle checks two full heads."""
    inp = si.workload_inputs(3)
    g = cuda(inp)
    o, Z = tm2.forward_quadratic(g["q"], g["k"], g["v"], g["a"])
    grads = tm2.backward_quadratic(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"])
    torch.cuda.synchronize()
    for b, h in ((0, 2), (1, 9)):
        sel = (slice(b, b + 1), slice(h, h + 1))
        q, k, v, a, dO = (inp[n][sel] for n in ("q", "k", "v", "a", "dO"))
        o_ref, _ = oracle.fwd_quadratic(q, k, v, a, True)
        refs = oracle.bwd_quadratic(q, k, v, a, dO, True)
        assert si.rel_err(o.cpu()[sel], o_ref) <= 2e-2
        for name, x, ref in zip(("dq", "dk", "dv", "da"), grads, refs):
            e = si.rel_err(x.cpu()[sel], ref)
            assert e <= 2e-2, (name, b, h, e)
