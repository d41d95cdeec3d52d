"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Metric per output tensor: max|err| / RMS(oracle tensor).  Bars: 2e-2 for bf16 inputs
with fp32 accumulation, 1e-4 for the fp32 mode.  Inputs come from synth_inputs (the
same buffers feed both sides; bf16 values are up-cast exactly for the oracle).
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


def err(x, ref):
    return si.rel_err(x, ref)


def gerr(x, ref, scale):
    """err(), except where the exact gradient is identically zero (T = 1 with
    normalisation: o_0 = v_0 whatever q, k are), where |x| is measured against `scale`."""
    r = np.asarray(ref, dtype=np.float64)
    if np.sqrt((r ** 2).mean()) <= 1e-9 * scale:
        return float(torch.as_tensor(x).double().abs().max()) / scale
    return err(x, ref)


def run_fwd(inp, normalize=True, chunk=0, **kw):
    g = cuda(inp)
    out = tm2.forward(g["q"], g["k"], g["v"], g["a"], normalize=normalize, chunk=chunk, **kw)
    torch.cuda.synchronize()
    return out


def check_fwd(inp, dtype, normalize=True, chunk=0, heads=None):
    o, Z = run_fwd(inp, normalize, chunk)
    sel = (slice(None), slice(None)) if heads is None else heads
    q, k, v, a = (inp[n][sel] for n in ("q", "k", "v", "a"))
    o_ref, Z_ref = oracle.fwd_quadratic(q, k, v, a, normalize)
    eo, ez = err(o.cpu()[sel], o_ref), err(Z.cpu()[sel], Z_ref)
    assert eo <= TOL[dtype], ("o", eo)
    assert ez <= TOL[dtype], ("Z", ez)
    return eo, ez


# ------------------------------------------------------------------------ forward

@pytest.mark.parametrize("normalize", [True, False])
def test_fwd_fp32_d16_T256(normalize):
    """Forward only, fp32: B=1, H=2, T=256, d=dv=16, chunk 64, against both oracle forms."""
    inp = si.workload_inputs(1)
    o, Z = run_fwd(inp, normalize, chunk=64)
    o_q, Z_q = oracle.fwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], normalize)
    o_r, Z_r, _, _ = oracle.fwd_recurrent(inp["q"], inp["k"], inp["v"], inp["a"], normalize)
    for ref_o, ref_Z in ((o_q, Z_q), (o_r, Z_r)):
        assert err(o.cpu(), ref_o) <= 1e-4
        assert err(Z.cpu(), ref_Z) <= 1e-4


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("T", [1, 64, 200, 333])
def test_fwd_small_ragged(dtype, d, T):
    """Several chunks and a ragged last chunk (T % 64 != 0), every supported head dim."""
    inp = si.sequence_inputs(2, 3, T, d, d, dtype=dtype, qkv_std=1 / math.sqrt(d), seed=100 + T + d)
    for normalize in (True, False):
        check_fwd(inp, dtype, normalize)


def test_fwd_bf16_B4_H16_T2048_full():
    """bf16 forward at B=4, H=16, T=2048, d=dv=64 checked on every head."""
    inp = si.workload_inputs(2)
    check_fwd(inp, "bf16", True)


def test_fwd_initial_and_final_state():
    """Prefill with an initial state; the final state equals the oracle recurrence's."""
    B, H, T, d = 2, 2, 150, 16
    inp = si.sequence_inputs(B, H, T, d, d, dtype="f32", qkv_std=0.25, seed=7)
    g = torch.Generator().manual_seed(8)
    S0 = torch.randn(B, H, d * d, d, generator=g) * 0.1
    z0 = torch.rand(B, H, d * d, generator=g) * 0.1
    gi = cuda(inp)
    o, Z, Sf, zf = tm2.forward(gi["q"], gi["k"], gi["v"], gi["a"], normalize=True, S0=S0.cuda(),
                               z0=z0.cuda(), return_state=True)
    torch.cuda.synchronize()
    o_r, Z_r, Sf_r, zf_r = oracle.fwd_recurrent(inp["q"], inp["k"], inp["v"], inp["a"], True, S0=S0, z0=z0)
    assert err(o.cpu(), o_r) <= 1e-4 and err(Z.cpu(), Z_r) <= 1e-4
    assert err(Sf.cpu(), Sf_r) <= 1e-4 and err(zf.cpu(), zf_r) <= 1e-4


def test_fwd_bf16_d64_initial_and_final_state():
    """bf16, d = dv = 64 (the tensor-core path): continue a sequence from the state a prefix
    left behind (the oracle recurrence over 300 tokens gives S0, z0), over three chunks with
    a ragged end; outputs and the final state against the oracle recurrence.  (A state that
    no sequence can produce -- e.g. z0 with random signs -- lets Z cross zero, where o = N/Z
    has no usable precision in any arithmetic.)"""
    B, H, T, d = 1, 2, 600, 64
    pre = si.sequence_inputs(B, H, 300, d, d, dtype="bf16", qkv_std=0.125, seed=16)
    _, _, S0, z0 = oracle.fwd_recurrent(pre["q"], pre["k"], pre["v"], pre["a"], True)
    S0 = torch.as_tensor(S0).float()
    z0 = torch.as_tensor(z0).float()
    inp = si.sequence_inputs(B, H, T, d, d, dtype="bf16", qkv_std=0.125, seed=17)
    gi = cuda(inp)
    o, Z, Sf, zf = tm2.forward(gi["q"], gi["k"], gi["v"], gi["a"], normalize=True, S0=S0.cuda(),
                               z0=z0.cuda(), return_state=True)
    torch.cuda.synchronize()
    o_r, Z_r, Sf_r, zf_r = oracle.fwd_recurrent(inp["q"], inp["k"], inp["v"], inp["a"], True, S0=S0, z0=z0)
    assert err(o.cpu(), o_r) <= 2e-2 and err(Z.cpu(), Z_r) <= 2e-2
    assert err(Sf.cpu(), Sf_r) <= 2e-2 and err(zf.cpu(), zf_r) <= 2e-2


def test_fwd_bf16_d64_antisymmetric_initial_state():
    """An initial state with an antisymmetric part in the key indices (m, n) (no sequence
    produces one, but the boundary accepts any S0, z0) must still give the oracle's outputs
    (the readout (q (x) q)^T S sees only the symmetric part) and its final state (the
    antisymmetric part decays by the product of all chunk decays)."""
    B, H, T, d = 1, 2, 600, 64
    pre = si.sequence_inputs(B, H, 300, d, d, dtype="bf16", qkv_std=0.125, seed=16)
    _, _, S0, z0 = oracle.fwd_recurrent(pre["q"], pre["k"], pre["v"], pre["a"], True)
    S0 = torch.as_tensor(S0).double()
    z0 = torch.as_tensor(z0).double()
    g = torch.Generator().manual_seed(23)
    R = torch.randn(B, H, d, d, d, generator=g, dtype=torch.float64) * S0.abs().mean()
    S0 = (S0.view(B, H, d, d, d) + 0.5 * (R - R.transpose(2, 3))).reshape(B, H, d * d, d).float()
    r = torch.randn(B, H, d, d, generator=g, dtype=torch.float64) * z0.abs().mean()
    z0 = (z0.view(B, H, d, d) + 0.5 * (r - r.transpose(2, 3))).reshape(B, H, d * d).float()
    inp = si.sequence_inputs(B, H, T, d, d, dtype="bf16", qkv_std=0.125, seed=17)
    gi = cuda(inp)
    o, Z, Sf, zf = tm2.forward(gi["q"], gi["k"], gi["v"], gi["a"], normalize=True, S0=S0.cuda(),
                               z0=z0.cuda(), return_state=True)
    torch.cuda.synchronize()
    o_r, Z_r, Sf_r, zf_r = oracle.fwd_recurrent(inp["q"], inp["k"], inp["v"], inp["a"], True, S0=S0, z0=z0)
    assert err(o.cpu(), o_r) <= 2e-2 and err(Z.cpu(), Z_r) <= 2e-2
    assert err(Sf.cpu(), Sf_r) <= 2e-2 and err(zf.cpu(), zf_r) <= 2e-2


def test_fwd_bf16_d64_antisymmetric_state_survives():
    """As above at a = -8 (softplus(-8) = 3.4e-4 per token: the state barely decays over the 600
    tokens), so the antisymmetric part of S0, z0 is still most of the final state's: the forward
    walk keeps only the symmetric part in its (m <= n block-packed) running state and restores
    the decayed antisymmetric part in S_final, z_final."""
    B, H, T, d = 1, 2, 600, 64
    pre = si.sequence_inputs(B, H, 300, d, d, dtype="bf16", qkv_std=0.125, seed=16)
    _, _, S0, z0 = oracle.fwd_recurrent(pre["q"], pre["k"], pre["v"], pre["a"], True)
    S0 = torch.as_tensor(S0).double()
    z0 = torch.as_tensor(z0).double()
    g = torch.Generator().manual_seed(24)
    R = torch.randn(B, H, d, d, d, generator=g, dtype=torch.float64) * 10 * S0.abs().mean()
    S0 = (S0.view(B, H, d, d, d) + 0.5 * (R - R.transpose(2, 3))).reshape(B, H, d * d, d).float()
    r = torch.randn(B, H, d, d, generator=g, dtype=torch.float64) * 10 * z0.abs().mean()
    z0 = (z0.view(B, H, d, d) + 0.5 * (r - r.transpose(2, 3))).reshape(B, H, d * d).float()
    inp = si.sequence_inputs(B, H, T, d, d, dtype="bf16", qkv_std=0.125, seed=18)
    inp["a"] = torch.full_like(inp["a"], -8.0)
    gi = cuda(inp)
    o, Z, Sf, zf = tm2.forward(gi["q"], gi["k"], gi["v"], gi["a"], normalize=True, S0=S0.cuda(),
                               z0=z0.cuda(), return_state=True)
    torch.cuda.synchronize()
    o_r, Z_r, Sf_r, zf_r = oracle.fwd_recurrent(inp["q"], inp["k"], inp["v"], inp["a"], True, S0=S0, z0=z0)
    asym = torch.as_tensor(Sf_r).view(B, H, d, d, d)
    asym = (asym - asym.transpose(2, 3)).abs().max() / torch.as_tensor(Sf_r).abs().max()
    assert asym > 0.1   # the antisymmetric part is a visible share of the final state
    assert err(o.cpu(), o_r) <= 2e-2 and err(Z.cpu(), Z_r) <= 2e-2
    assert err(Sf.cpu(), Sf_r) <= 2e-2 and err(zf.cpu(), zf_r) <= 2e-2


@pytest.mark.parametrize("normalize", [True, False])
def test_fwd_chunk_invariance_bf16_d64(normalize):
    """chunk 64 (CUDA-core path) and chunk 256 (tensor-core path) give the same outputs,
    both within the bf16 bar of the oracle."""
    inp = si.sequence_inputs(2, 2, 1000, 64, 64, dtype="bf16", qkv_std=0.125, seed=19)
    o64, Z64 = run_fwd(inp, normalize, chunk=64)
    o256, Z256 = run_fwd(inp, normalize, chunk=256)
    o_ref, Z_ref = oracle.fwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], normalize)
    assert err(o64.cpu(), o_ref) <= 2e-2 and err(o256.cpu(), o_ref) <= 2e-2
    assert err(Z256.cpu(), Z_ref) <= 2e-2
    assert err(o256.cpu(), o64.cpu()) <= 2e-2


def test_fwd_empty_sequence():
    """T = 0 is a no-op; the final state is the initial state."""
    q = torch.zeros(1, 2, 0, 16, device="cuda")
    a = torch.zeros(1, 2, 0, device="cuda")
    S0 = torch.randn(1, 2, 256, 16, device="cuda")
    o, Z, Sf, zf = tm2.forward(q, q, q, a, S0=S0, return_state=True)
    torch.cuda.synchronize()
    assert o.shape == (1, 2, 0, 16)
    assert torch.equal(Sf, S0) and torch.count_nonzero(zf) == 0


def test_fwd_deterministic():
    inp = si.sequence_inputs(1, 4, 300, 64, 64, dtype="bf16", qkv_std=0.125, seed=3)
    o1, Z1 = run_fwd(inp)
    o2, Z2 = run_fwd(inp)
    assert torch.equal(o1, o2) and torch.equal(Z1, Z2)


def test_fwd_decay_limits():
    """a = -40 (no decay) and a = +40 (decay 0: normalised o_i = v_i) on the GPU."""
    inp = si.sequence_inputs(1, 2, 130, 32, 32, dtype="f32", qkv_std=0.2, seed=5)
    inp["a"] = torch.full_like(inp["a"], 40.0)
    o, _ = run_fwd(inp, True)
    assert err(o.cpu(), inp["v"]) <= 1e-4
    inp["a"] = torch.full_like(inp["a"], -40.0)
    check_fwd(inp, "f32", True)


# ------------------------------------------------------------------------ backward

def run_fwd_bwd(inp, normalize=True, chunk=0):
    g = cuda(inp)
    o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"], normalize=normalize, chunk=chunk)
    dq, dk, dv, da = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], normalize=normalize,
                                  chunk=chunk)
    torch.cuda.synchronize()
    return o, Z, dq, dk, dv, da


def check_bwd(inp, dtype, normalize=True, heads=None):
    o, Z, dq, dk, dv, da = run_fwd_bwd(inp, normalize)
    sel = (slice(None), slice(None)) if heads is None else heads
    q, k, v, a, dO = (inp[n][sel] for n in ("q", "k", "v", "a", "dO"))
    o_ref, Z_ref = oracle.fwd_quadratic(q, k, v, a, normalize)
    refs = oracle.bwd_quadratic(q, k, v, a, dO, normalize)
    errs = {"o": err(o.cpu()[sel], o_ref)}
    scale = float(np.sqrt((refs[2] ** 2).mean()))   # RMS of dv, never degenerate
    for name, x, ref in zip(("dq", "dk", "dv", "da"), (dq, dk, dv, da), refs):
        errs[name] = gerr(x.cpu()[sel], ref, scale)
    for name, e in errs.items():
        assert e <= TOL[dtype], (name, e, errs)
    return errs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64])
@pytest.mark.parametrize("T", [1, 64, 200])
@pytest.mark.parametrize("normalize", [True, False])
def test_bwd_small_ragged(dtype, d, T, normalize):
    inp = si.sequence_inputs(2, 2, T, d, d, dtype=dtype, qkv_std=1 / math.sqrt(d), seed=200 + T + d,
                             with_dO=True)
    check_bwd(inp, dtype, normalize)


@pytest.mark.parametrize("normalize", [True, False])
def test_bwd_chunk_invariance_bf16_d64(normalize):
    """Backward through chunk 64 (CUDA-core path) and chunk 256 (tensor-core path) over
    four chunks with a ragged end: both within the bf16 bar of the oracle."""
    inp = si.sequence_inputs(1, 3, 1000, 64, 64, dtype="bf16", qkv_std=0.125, seed=23, with_dO=True)
    g = cuda(inp)
    refs = oracle.bwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], inp["dO"], normalize)
    for chunk in (64, 256):
        o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"], normalize=normalize, chunk=chunk)
        grads = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], normalize=normalize, chunk=chunk)
        torch.cuda.synchronize()
        for name, x, ref in zip(("dq", "dk", "dv", "da"), grads, refs):
            e = err(x.cpu(), ref)
            assert e <= 2e-2, (chunk, name, e)


@pytest.mark.parametrize("chunk", [64, 256])
def test_bwd_reuse_forward_states(chunk):
    """TM2_REUSE_STATES: the backward reads the chunk states its forward left in the shared
    workspace; the gradients are bitwise those of a backward that recomputes them."""
    inp = si.sequence_inputs(2, 2, 700, 64, 64, dtype="bf16", qkv_std=0.125, seed=29, with_dO=True)
    g = cuda(inp)
    ws = torch.empty(tm2.workspace_bytes(2, 2, 700, 64, 64, chunk), dtype=torch.uint8, device="cuda")
    o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"], chunk=chunk, workspace=ws)
    reused = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], chunk=chunk, workspace=ws,
                          reuse_states=True)
    fresh = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], chunk=chunk)
    torch.cuda.synchronize()
    for x, y in zip(reused, fresh):
        assert torch.equal(x, y)


def test_fwd_bwd_bf16_B2_H16_T8192_sampled_heads():
    """fwd+bwd at B=2, H=16, T=8192, d=dv=64 bf16 on the whole batch; the oracle checks
    two full heads (all 8192 positions, all outputs and gradients)."""
    inp = si.workload_inputs(3)
    o, Z, dq, dk, dv, da = run_fwd_bwd(inp, True)
    for b, h in ((0, 0), (1, 15)):
        sel = (slice(b, b + 1), slice(h, h + 1))
        q, k, v, a, dO = (inp[n][sel] for n in ("q", "k", "v", "a", "dO"))
        o_ref, Z_ref = oracle.fwd_quadratic(q, k, v, a, True)
        refs = oracle.bwd_quadratic(q, k, v, a, dO, True)
        assert err(o.cpu()[sel], o_ref) <= 2e-2
        assert err(Z.cpu()[sel], Z_ref) <= 2e-2
        for name, x, ref in zip(("dq", "dk", "dv", "da"), (dq, dk, dv, da), refs):
            e = err(x.cpu()[sel], ref)
            assert e <= 2e-2, (name, b, h, e)
    assert torch.isfinite(o).all() and torch.isfinite(da).all()


def test_bwd_first_token_decay_gradient_zero():
    """da_0 = 0 (only differences of cumA enter the output) on the GPU too."""
    inp = si.sequence_inputs(1, 4, 256, 64, 64, dtype="f32", qkv_std=0.125, seed=9, with_dO=True)
    *_, da = run_fwd_bwd(inp, True)
    da = da.cpu()
    assert da[..., 0].abs().max() <= 1e-4 * da.abs().max()


# ------------------------------------------------------------------------ decode

def test_decode_matches_forward():
    """T decode steps from a zero state reproduce the forward outputs (App. A)."""
    B, H, T, d = 2, 4, 40, 64
    inp = si.sequence_inputs(B, H, T, d, d, dtype="f32", qkv_std=0.125, seed=11)
    g = cuda(inp)
    o_f, Z_f = tm2.forward(g["q"], g["k"], g["v"], g["a"], normalize=True)
    S = torch.zeros(B, H, d * d, d, device="cuda")
    z = torch.zeros(B, H, d * d, device="cuda")
    for t in range(T):
        o, zeta = tm2.step(g["q"][:, :, t].contiguous(), g["k"][:, :, t].contiguous(),
                           g["v"][:, :, t].contiguous(), g["a"][:, :, t].contiguous(), S, z)
        assert err(o.cpu(), o_f[:, :, t].cpu()) <= 1e-4
        assert err(zeta.cpu(), Z_f[:, :, t].cpu()) <= 1e-4


def test_decode_1000_steps_N256():
    """Decode: 256 sequences x 16 heads, d = dv = 64, fp32 state from S0 ~ N(0, 0.01^2),
    1000 steps on the GPU; the oracle recurrence follows 16 of the sequences (all heads)
    and checks y and zeta at every step and the state at the end.  (o = y / zeta is
    ill-conditioned where zeta is small -- z0 = 0 while S0 is not -- so it is not a
    parity quantity; y and zeta are.)"""
    w = si.WORKLOADS[4]
    N, H, d, dv = w.B, w.H, w.d, w.dv
    S0, z0 = si.decode_initial_state(N, H, d, dv, S0_std=w.S0_std)
    sub = [0, 17, 37, 50, 64, 83, 101, 119, 128, 150, 170, 191, 213, 230, 247, 255]
    S_ref = S0[sub].double().numpy().copy()
    z_ref = z0[sub].double().numpy().copy()
    S = S0.cuda()
    z = z0.cuda()
    del S0
    worst = {"y": 0.0, "zeta": 0.0}
    for t in range(w.steps):
        tok = si.decode_token(t, N, H, d, dv, qkv_std=w.qkv_std)
        gt = cuda(tok)
        y, zeta = tm2.step(gt["q"], gt["k"], gt["v"], gt["a"], S, z, normalize=False)
        sl = {k: v[sub] for k, v in tok.items()}
        y_r, zeta_r = oracle.step(sl["q"], sl["k"], sl["v"], sl["a"], S_ref, z_ref, normalize=False)
        for name, x, ref in (("y", y, y_r), ("zeta", zeta, zeta_r)):
            worst[name] = max(worst[name], err(x[sub].cpu(), ref))
    torch.cuda.synchronize()
    for name, e in worst.items():
        assert e <= 1e-4, (name, e)
    assert err(S[sub].cpu(), S_ref) <= 1e-4
    assert err(z[sub].cpu(), z_ref) <= 1e-4


def test_decode_resume_bitwise():
    """Checkpoint and resume of decode (App. A: the state is all a sequence carries): 500
    steps, a round trip of S and z through host memory, 500 more steps, is bitwise the same
    as 1000 steps straight through."""
    N, H, d = 32, 4, 64
    S0, z0 = si.decode_initial_state(N, H, d, d, S0_std=0.01, seed=13)
    toks = [cuda(si.decode_token(t, N, H, d, d, qkv_std=0.125, seed=13)) for t in range(1000)]
    S1, z1 = S0.cuda(), z0.cuda()
    ys1 = []
    for t in range(1000):
        x = toks[t]
        y, _ = tm2.step(x["q"], x["k"], x["v"], x["a"], S1, z1)
        ys1.append(y)
    S2, z2 = S0.cuda(), z0.cuda()
    ys2 = []
    for t in range(1000):
        if t == 500:
            S_host, z_host = S2.cpu(), z2.cpu()
            del S2, z2
            torch.cuda.synchronize()
            S2, z2 = S_host.cuda(), z_host.cuda()
        x = toks[t]
        y, _ = tm2.step(x["q"], x["k"], x["v"], x["a"], S2, z2)
        ys2.append(y)
    torch.cuda.synchronize()
    assert torch.equal(S1, S2) and torch.equal(z1, z2)
    assert all(torch.equal(a, b) for a, b in zip(ys1, ys2))


def test_decode_bf16_tokens():
    """bf16 token inputs with the fp32 state."""
    N, H, d = 8, 4, 32
    S0, z0 = si.decode_initial_state(N, H, d, d, S0_std=0.01, seed=12)
    S, z = S0.cuda(), z0.cuda()
    S_ref, z_ref = S0.double().numpy().copy(), z0.double().numpy().copy()
    for t in range(20):
        tok = si.decode_token(t, N, H, d, d, dtype="bf16", qkv_std=1 / math.sqrt(d), seed=12)
        gt = cuda(tok)
        o, zeta = tm2.step(gt["q"], gt["k"], gt["v"], gt["a"], S, z, normalize=True)
        o_r, zeta_r = oracle.step(tok["q"], tok["k"], tok["v"], tok["a"], S_ref, z_ref, normalize=True)
        assert err(o.cpu(), o_r) <= 2e-2 and err(zeta.cpu(), zeta_r) <= 2e-2


# ------------------------------------------------------------------------ 2Mamba-E

def run_e(inp):
    g = cuda(inp)
    o, lse = tm2.e_forward(g["q"], g["k"], g["v"], g["a"])
    dq, dk, dv, da = tm2.e_backward(g["q"], g["k"], g["v"], g["a"], o, lse, g["dO"])
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv, da


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1, 64, 190, 1000])
def test_e_small_ragged(dtype, T):
    d = 64
    inp = si.sequence_inputs(2, 2, T, d, d, dtype=dtype, qkv_std=1.0, seed=300 + T, with_dO=True)
    o, lse, dq, dk, dv, da = run_e(inp)
    o_r, lse_r = oracle.e_fwd(inp["q"], inp["k"], inp["v"], inp["a"])
    refs = oracle.e_bwd(inp["q"], inp["k"], inp["v"], inp["a"], inp["dO"])
    tol = TOL[dtype]
    assert err(o.cpu(), o_r) <= tol
    assert err(lse.cpu(), lse_r) <= tol
    for name, x, ref in zip(("dq", "dk", "dv", "da"), (dq, dk, dv, da), refs):
        assert err(x.cpu(), ref) <= tol, name


def test_e_fwd_bwd_bf16_B2_H16_T4096_sampled_heads():
    """2Mamba-E fwd+bwd at B=2, H=16, T=4096, d=dv=64 bf16; two full heads checked."""
    inp = si.workload_inputs(5)
    o, lse, dq, dk, dv, da = run_e(inp)
    for b, h in ((0, 3), (1, 12)):
        sel = (slice(b, b + 1), slice(h, h + 1))
        q, k, v, a, dO = (inp[n][sel] for n in ("q", "k", "v", "a", "dO"))
        o_r, lse_r = oracle.e_fwd(q, k, v, a)
        refs = oracle.e_bwd(q, k, v, a, dO)
        assert err(o.cpu()[sel], o_r) <= 2e-2
        for name, x, ref in zip(("dq", "dk", "dv", "da"), (dq, dk, dv, da), refs):
            e = err(x.cpu()[sel], ref)
            assert e <= 2e-2, (name, e)



# ------------------------------------------------------------------------ gradient output type

def test_grads_in_input_dtype_are_the_rounded_fp32_grads():
    """TM2_GRADS_INPUT_DTYPE: dq, dk, dv come out in bf16, each exactly the round-to-nearest of
    the fp32 gradient the same backward writes without the flag -- on the tensor-core chunked
    path, the CUDA-core chunked path, 2Mamba-E and the quadratic form."""
    inp = si.sequence_inputs(2, 2, 333, 64, 64, dtype="bf16", qkv_std=0.125, seed=801, with_dO=True)
    g = cuda(inp)
    for chunk in (0, 64):
        o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"], chunk=chunk)
        full = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], chunk=chunk)
        low = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], chunk=chunk, lowp_grads=True)
        torch.cuda.synchronize()
        for x, y in zip(full[:3], low[:3]):
            assert y.dtype == torch.bfloat16 and torch.equal(y, x.to(torch.bfloat16))
        assert torch.equal(full[3], low[3])
    ie = si.sequence_inputs(2, 2, 333, 64, 64, dtype="bf16", qkv_std=1.0, seed=802, with_dO=True)
    ge = cuda(ie)
    oe, lse = tm2.e_forward(ge["q"], ge["k"], ge["v"], ge["a"])
    full = tm2.e_backward(ge["q"], ge["k"], ge["v"], ge["a"], oe, lse, ge["dO"])
    low = tm2.e_backward(ge["q"], ge["k"], ge["v"], ge["a"], oe, lse, ge["dO"], lowp_grads=True)
    oq, Zq = tm2.forward_quadratic(g["q"], g["k"], g["v"], g["a"])
    fq = tm2.backward_quadratic(g["q"], g["k"], g["v"], g["a"], oq, Zq, g["dO"])
    lq = tm2.backward_quadratic(g["q"], g["k"], g["v"], g["a"], oq, Zq, g["dO"], lowp_grads=True)
    torch.cuda.synchronize()
    for F, L in ((full, low), (fq, lq)):
        for x, y in zip(F[:3], L[:3]):
            assert y.dtype == torch.bfloat16 and torch.equal(y, x.to(torch.bfloat16))
