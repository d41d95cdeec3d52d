"""GPU parity at the method's edge cases, on the tensor-core path that the benchmark runs.

The 2Mamba cases run bf16 inputs with d = dv = 64 and chunk 256 (the tensor-core scan,
chunk output, dq and dk/dv kernels), over four chunks with a ragged end (T = 1000), forward
and backward, normalised and not, against the fp64 oracle at the bf16 bar (2e-2):

* a = +40: every decay is e^-40, so only the diagonal weight s_ii^2 survives and the
  normalised output is v itself ("2Mamba2Furious", Sec. 3-5: the softplus A-mask).
* a = -40: no decay; the state sums every earlier token.
* a mixed: each token draws +40 or -40, so runs of no decay are cut by full resets.
* input scale: q, k, v ~ N(0, s^2) with s = 1e-2 and s = 4 (the normalised output does not
  depend on the scale of q and k; the fp16 state planes must not lose it).

The 2Mamba-E cases (Sec. 6) run the tensor-core forward and backward at the decay limits:
a = -40 is plain causal softmax attention, a = +40 gives o_i = v_i.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import ssm_sequence_mixer_chunked_b300 as tm2
import synth_inputs as si

pytestmark = pytest.mark.gpu

BAR = 2e-2


def cuda(d):
    return {k: v.cuda() for k, v in d.items()}


def gerr(x, ref, scale):
    """max|x - ref| / RMS(ref); where the exact tensor is zero up to e^-40-sized terms (for
    example dq, dk when a = +40 leaves only the diagonal weights, or da when sigmoid(-40)
    multiplies it), max|x - ref| is measured against `scale` instead."""
    r = np.asarray(ref, dtype=np.float64)
    if np.sqrt((r ** 2).mean()) <= 1e-9 * scale:
        return float((torch.as_tensor(x).double() - torch.as_tensor(r)).abs().max()) / scale
    return si.rel_err(x, ref)


def f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def well_conditioned_rows(inp, o_ref, Z_ref, refs, frac=0.25):
    """Rows (b, h, t) whose dq and dk the backward can determine to the bar from an fp32
    forward output.  The normalised backward depends on o through D_i = dO_i . o_i, and where
    one weight dominates a row whose score q_i . k_i is nearly zero (a token right after a full
    decay, a = +40) dq_i, dk_i are amplified copies of o_i's last bits: the oracle backward
    evaluated at the exact o rounded once to fp32 already moves them by more than `frac` of
    the bar there.  Such rows are conditioning-limited for any fp32 pipeline (one rounding of
    D_i decides them); they are left out of the dq, dk checks."""
    q, k, v, a, dO = (inp[n] for n in ("q", "k", "v", "a", "dO"))
    r32 = oracle.bwd_quadratic(q, k, v, a, dO, True, o=f32(o_ref), Z=f32(Z_ref))
    ok = np.ones(np.asarray(o_ref).shape[:3], dtype=bool)
    for idx in (0, 1):
        rms = np.sqrt((refs[idx] ** 2).mean())
        ok &= np.abs(r32[idx] - refs[idx]).max(-1) <= frac * BAR * rms
    return ok


def row_err(x, ref, rows):
    """max |x - ref| over the selected rows, over the RMS of ref over all rows."""
    x = torch.as_tensor(x).double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(x - ref)[rows].max() / np.sqrt((ref ** 2).mean()))


def edge_inputs(case, B=1, H=2, T=1000, d=64, seed=0, qkv_std=None):
    std = {"std_1e-2": 1e-2, "std_4": 4.0}.get(case, 1 / math.sqrt(d) if qkv_std is None else qkv_std)
    inp = si.sequence_inputs(B, H, T, d, d, dtype="bf16", qkv_std=std, seed=seed, with_dO=True)
    if case == "a_plus40":
        inp["a"] = torch.full_like(inp["a"], 40.0)
    elif case == "a_minus40":
        inp["a"] = torch.full_like(inp["a"], -40.0)
    elif case == "a_mixed":
        g = torch.Generator().manual_seed(seed + 1)
        pick = torch.rand(inp["a"].shape, generator=g) < 0.5
        inp["a"] = torch.where(pick, torch.tensor(40.0), torch.tensor(-40.0))
    return inp


CASES = ["a_plus40", "a_minus40", "a_mixed", "std_1e-2", "std_4"]


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("case", CASES)
def test_tc_edge_fwd_bwd(case, normalize):
    """Forward and backward against the oracle, end to end; with normalisation also the
    backward as a function of its inputs (the oracle backward at the kernel's own o and Z).
    End-to-end dq, dk are checked on the rows an fp32 forward output determines to the bar
    (well_conditioned_rows); at most 1% of the rows may fall outside."""
    inp = edge_inputs(case, seed=500 + CASES.index(case))
    g = cuda(inp)
    o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"], normalize=normalize, chunk=256)
    grads = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], normalize=normalize, chunk=256)
    torch.cuda.synchronize()
    for x in (o, Z) + tuple(grads):
        assert torch.isfinite(x).all(), case
    q, k, v, a, dO = (inp[n] for n in ("q", "k", "v", "a", "dO"))
    o_ref, Z_ref = oracle.fwd_quadratic(q, k, v, a, normalize)
    refs = oracle.bwd_quadratic(q, k, v, a, dO, normalize)
    scale = float(np.sqrt((refs[2] ** 2).mean()))   # RMS of dv: never degenerate here
    errs = {"o": si.rel_err(o.float().cpu(), o_ref), "Z": si.rel_err(Z.cpu(), Z_ref)}
    degenerate = float(np.sqrt((refs[0] ** 2).mean())) <= 1e-9 * scale   # a = +40: exact dq, dk ~ e^-40
    rows = well_conditioned_rows(inp, o_ref, Z_ref, refs) if normalize and not degenerate else None
    for name, x, ref in zip(("dq", "dk", "dv", "da"), grads, refs):
        if rows is not None and name in ("dq", "dk"):
            errs[name] = row_err(x.float().cpu(), ref, rows)
        else:
            errs[name] = gerr(x.float().cpu(), ref, scale)
    if normalize and not degenerate:   # (at a = +40 every row is conditioning-limited)
        at = oracle.bwd_quadratic(q, k, v, a, dO, True, o=o.cpu(), Z=Z.cpu())
        for name, x, ref in zip(("dq", "dk", "dv", "da"), grads, at):
            if rows is not None and name in ("dq", "dk"):
                errs[name + "@o"] = row_err(x.float().cpu(), ref, rows)
            else:
                errs[name + "@o"] = gerr(x.float().cpu(), ref, scale)
    bad = {k: v for k, v in errs.items() if not v <= BAR}
    assert not bad, (case, normalize, errs)
    if rows is not None:
        assert rows.mean() >= 0.99, (case, float(rows.mean()))
    if case == "a_plus40" and normalize:
        # only the diagonal weight survives: o_i = v_i
        assert si.rel_err(o.float().cpu(), inp["v"]) <= BAR


def test_tc_edge_no_decay_long():
    """a = -40 over T = 4096 (16 chunks): the undecayed state grows with every chunk; the
    normaliser column and the fp16 planes must keep up."""
    inp = edge_inputs("a_minus40", B=1, H=1, T=4096, seed=520)
    g = cuda(inp)
    o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"], chunk=256)
    grads = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], chunk=256)
    torch.cuda.synchronize()
    o_ref, Z_ref = oracle.fwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], True)
    refs = oracle.bwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], inp["dO"], True)
    scale = float(np.sqrt((refs[2] ** 2).mean()))
    assert si.rel_err(o.float().cpu(), o_ref) <= BAR
    assert si.rel_err(Z.cpu(), Z_ref) <= BAR
    for name, x, ref in zip(("dq", "dk", "dv", "da"), grads, refs):
        e = gerr(x.float().cpu(), ref, scale)
        assert e <= BAR, (name, e)


def test_tc_edge_scale_invariance_normalised():
    """The normalised output does not depend on the scale of q and k (w_ij scales by c^4 in
    both N_i and Z_i): the tensor-core forward at q, k scaled by 1/16 and by 16 (powers of two,
    so the bf16 inputs stay exact) agrees with the unscaled run within the bf16 bar."""
    inp = edge_inputs("base", B=1, H=2, T=700, seed=530)
    g = cuda(inp)
    o1, _ = tm2.forward(g["q"], g["k"], g["v"], g["a"], chunk=256)
    for c in (1.0 / 16, 16.0):
        o2, _ = tm2.forward(g["q"] * c, g["k"] * c, g["v"], g["a"], chunk=256)
        torch.cuda.synchronize()
        assert si.rel_err(o2.float().cpu(), o1.float().cpu()) <= BAR, c


# ------------------------------------------------------------------------ 2Mamba-E

E_CASES = ["a_plus40", "a_minus40", "a_mixed", "std_4"]


@pytest.mark.parametrize("case", E_CASES)
def test_tc_e_edge_fwd_bwd(case):
    inp = edge_inputs(case, seed=540 + E_CASES.index(case), qkv_std=1.0)
    g = cuda(inp)
    o, lse = tm2.e_forward(g["q"], g["k"], g["v"], g["a"])
    grads = tm2.e_backward(g["q"], g["k"], g["v"], g["a"], o, lse, g["dO"])
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.e_fwd(inp["q"], inp["k"], inp["v"], inp["a"])
    refs = oracle.e_bwd(inp["q"], inp["k"], inp["v"], inp["a"], inp["dO"])
    scale = float(np.sqrt((refs[2] ** 2).mean()))
    errs = {"o": si.rel_err(o.float().cpu(), o_ref), "lse": si.rel_err(lse.cpu(), lse_ref)}
    for name, x, ref in zip(("dq", "dk", "dv", "da"), grads, refs):
        errs[name] = gerr(x.float().cpu(), ref, scale)
    for x in (o, lse) + tuple(grads):
        assert torch.isfinite(x).all(), (case, errs)
    bad = {k: v for k, v in errs.items() if not v <= BAR}
    assert not bad, (case, errs)
    if case == "a_plus40":
        assert si.rel_err(o.float().cpu(), inp["v"]) <= BAR


def test_tc_e_no_decay_is_causal_softmax():
    """a = -40: 2Mamba-E is textbook causal softmax attention; the tensor-core forward agrees
    with torch's scaled_dot_product_attention (fp64, CPU) on the same bf16 inputs."""
    inp = edge_inputs("a_minus40", B=1, H=2, T=777, seed=550, qkv_std=1.0)
    g = cuda(inp)
    o, _ = tm2.e_forward(g["q"], g["k"], g["v"], g["a"])
    torch.cuda.synchronize()
    ref = torch.nn.functional.scaled_dot_product_attention(
        inp["q"].double(), inp["k"].double(), inp["v"].double(), is_causal=True)
    assert si.rel_err(o.float().cpu(), ref) <= BAR


# ------------------------------------------------------------------------ fp32, long sequences

@pytest.mark.parametrize("d", [16])
def test_fp32_long_sequence(d):
    """fp32 inputs at T = 8192 (the CUDA-core path, chunk 64): forward and backward within the
    fp32 bar 1e-4 over 128 chunks, where the running decay sums are longest."""
    inp = si.sequence_inputs(1, 2, 8192, d, d, dtype="f32", qkv_std=1 / math.sqrt(d), seed=560 + d,
                             with_dO=True)
    g = cuda(inp)
    o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"])
    grads = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"])
    torch.cuda.synchronize()
    o_ref, Z_ref = oracle.fwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], True)
    refs = oracle.bwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], inp["dO"], True)
    errs = {"o": si.rel_err(o.cpu(), o_ref), "Z": si.rel_err(Z.cpu(), Z_ref)}
    for name, x, ref in zip(("dq", "dk", "dv", "da"), grads, refs):
        errs[name] = si.rel_err(x.cpu(), ref)
    bad = {k: v for k, v in errs.items() if not v <= 1e-4}
    assert not bad, errs


def test_fp32_long_sequence_d32_forward():
    """fp32 inputs at T = 8192 with d = dv = 32: the forward within the fp32 bar 1e-4."""
    inp = si.sequence_inputs(1, 2, 8192, 32, 32, dtype="f32", qkv_std=1 / math.sqrt(32), seed=592)
    g = cuda(inp)
    o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"])
    torch.cuda.synchronize()
    o_ref, Z_ref = oracle.fwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], True)
    assert si.rel_err(o.cpu(), o_ref) <= 1e-4 and si.rel_err(Z.cpu(), Z_ref) <= 1e-4


def test_fp32_long_sequence_e():
    """2Mamba-E with fp32 inputs at T = 8192: the global running sums carry their fp32
    residual, so cumA_i - cumA_j keeps fp32 precision over the whole sequence."""
    inp = si.sequence_inputs(1, 1, 8192, 32, 32, dtype="f32", qkv_std=1.0, seed=570, with_dO=True)
    g = cuda(inp)
    o, lse = tm2.e_forward(g["q"], g["k"], g["v"], g["a"])
    grads = tm2.e_backward(g["q"], g["k"], g["v"], g["a"], o, lse, g["dO"])
    torch.cuda.synchronize()
    o_ref, _ = oracle.e_fwd(inp["q"], inp["k"], inp["v"], inp["a"])
    refs = oracle.e_bwd(inp["q"], inp["k"], inp["v"], inp["a"], inp["dO"])
    errs = {"o": si.rel_err(o.cpu(), o_ref)}
    for name, x, ref in zip(("dq", "dk", "dv", "da"), grads, refs):
        errs[name] = si.rel_err(x.cpu(), ref)
    bad = {k: v for k, v in errs.items() if not v <= 1e-4}
    assert not bad, errs
