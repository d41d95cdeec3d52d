"""GPU parity of the decode-side extensions against the fp64 oracle.

* Symmetric-packed second-order state ("2Mamba2Furious", Sec. 5.1 and Sec. 7: the size of the
  squared hidden state): decode steps on the packed state give the full state's outputs, for a
  zero and for a random (not symmetric) initial state, and the unpacked state equals the
  symmetric part of the oracle's.
* The size-2 input convolution of Mamba-2S (Sec. 3-4; App. A: inference caches the previous raw
  token): fused into the decode step, and as a sequence kernel with its backward.
* 2Mamba-E decoding over a key/value cache (Sec. 6; Sec. 1: 2Mamba-E needs a KV cache): every
  step equals the oracle's 2Mamba-E forward row for that token, including after a prefill and
  across the multi-block split of long caches.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import ssm_sequence_mixer_chunked_b300 as tm2
import synth_inputs as si

pytestmark = pytest.mark.gpu


def cuda(d):
    return {k: v.cuda() for k, v in d.items()}


def sym_part(S, d):
    """Symmetric part in the key indices (m, n) of full states (..., d*d, cols)."""
    S = np.asarray(S, dtype=np.float64)
    lead, cols = S.shape[:-2], S.shape[-1]
    X = S.reshape(lead + (d, d, cols))
    return (0.5 * (X + np.swapaxes(X, -3, -2))).reshape(S.shape)


# ------------------------------------------------------------------------ packed state

@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("init", ["zero", "random"])
def test_packed_decode_matches_full_state(d, init):
    N, H, steps = 12, 4, 60
    S0, z0 = si.decode_initial_state(N, H, d, d, S0_std=0.01 if init == "random" else 0.0, seed=700 + d)
    S_ref, z_ref = S0.double().numpy().copy(), z0.double().numpy().copy()
    Sp, zp = tm2.state_pack(S0.cuda(), z0.cuda())
    for t in range(steps):
        tok = si.decode_token(t, N, H, d, d, qkv_std=1 / math.sqrt(d), seed=700 + d)
        g = cuda(tok)
        y, zeta = tm2.step(g["q"], g["k"], g["v"], g["a"], Sp, zp, normalize=False, packed=True)
        y_r, zeta_r = oracle.step(tok["q"], tok["k"], tok["v"], tok["a"], S_ref, z_ref, normalize=False)
        torch.cuda.synchronize()
        assert si.rel_err(y.cpu(), y_r) <= 1e-4, t
        assert si.rel_err(zeta.cpu(), zeta_r) <= 1e-4, t
    S_full, z_full = tm2.state_unpack(Sp, zp, d=d)
    torch.cuda.synchronize()
    assert si.rel_err(S_full.cpu(), sym_part(S_ref, d)) <= 1e-4
    assert si.rel_err(z_full.cpu(), sym_part(z_ref[..., None], d)[..., 0]) <= 1e-4


def test_packed_decode_1000_steps_workload():
    """The decode workload (256 sequences x 16 heads, d = 64, S0 ~ N(0, 0.01^2), z0 = 0) on the
    packed state for 1000 steps; 8 sequences followed by the oracle at every step."""
    w = si.WORKLOADS[4]
    N, H, d = w.B, w.H, w.d
    S0, z0 = si.decode_initial_state(N, H, d, d, S0_std=w.S0_std)
    sub = [0, 37, 64, 101, 150, 191, 230, 255]
    S_ref = S0[sub].double().numpy().copy()
    z_ref = z0[sub].double().numpy().copy()
    Sp, zp = tm2.state_pack(S0.cuda(), z0.cuda())
    del S0
    worst = {"y": 0.0, "zeta": 0.0}
    for t in range(w.steps):
        tok = si.decode_token(t, N, H, d, d, qkv_std=w.qkv_std)
        g = cuda(tok)
        y, zeta = tm2.step(g["q"], g["k"], g["v"], g["a"], Sp, zp, normalize=False, packed=True)
        sl = {k: v[sub] for k, v in tok.items()}
        y_r, zeta_r = oracle.step(sl["q"], sl["k"], sl["v"], sl["a"], S_ref, z_ref, normalize=False)
        worst["y"] = max(worst["y"], si.rel_err(y[sub].cpu(), y_r))
        worst["zeta"] = max(worst["zeta"], si.rel_err(zeta[sub].cpu(), zeta_r))
    assert worst["y"] <= 1e-4 and worst["zeta"] <= 1e-4, worst
    S_full, _ = tm2.state_unpack(Sp[sub].contiguous(), None, d=d)
    torch.cuda.synchronize()
    assert si.rel_err(S_full.cpu(), sym_part(S_ref, d)) <= 1e-4


# ------------------------------------------------------------------------ input convolution

def conv_params(H, d, seed):
    g = torch.Generator().manual_seed(seed)
    w = [torch.randn(H, d, 2, generator=g, dtype=torch.float64).float() * 0.7 for _ in range(3)]
    b = [torch.randn(H, d, generator=g, dtype=torch.float64).float() * 0.05 for _ in range(3)]
    return w, b


@pytest.mark.parametrize("packed", [False, True])
def test_decode_with_conv_matches_conv_then_step(packed):
    """tm2_step_conv = the oracle convolution over the token stream (previous raw token from the
    cache), then the oracle recurrence on the convolved q, k, v."""
    N, H, d, steps = 6, 4, 64, 40
    w, b = conv_params(H, d, 710)
    toks = [si.decode_token(t, N, H, d, d, dtype="bf16", qkv_std=0.125, seed=711) for t in range(steps)]
    seq = {n: torch.stack([tk[n] for tk in toks], dim=2) for n in ("q", "k", "v")}   # (N,H,T,d)
    conv = {n: oracle.conv2_fwd(seq[n], w[i], b[i]) for i, n in enumerate(("q", "k", "v"))}
    S_ref = np.zeros((N, H, d * d, d))
    z_ref = np.zeros((N, H, d * d))
    rows = d * (d + 1) // 2 if packed else d * d
    S = torch.zeros(N, H, rows, d, device="cuda")
    z = torch.zeros(N, H, rows, device="cuda")
    caches = [torch.zeros(N, H, d, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    wc, bc = [x.cuda() for x in w], [x.cuda() for x in b]
    for t in range(steps):
        g = cuda(toks[t])
        o, zeta = tm2.step_conv(g["q"], g["k"], g["v"], g["a"], wc, bc, caches, S, z, packed=packed)
        o_r, zeta_r = oracle.step(conv["q"][:, :, t], conv["k"][:, :, t], conv["v"][:, :, t], toks[t]["a"],
                                  S_ref, z_ref, normalize=True)
        torch.cuda.synchronize()
        assert si.rel_err(o.cpu(), o_r) <= 1e-4, t
        assert si.rel_err(zeta.cpu(), zeta_r) <= 1e-4, t
    assert torch.equal(caches[0].cpu(), toks[-1]["q"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("C", [16, 64])
def test_conv2_sequence_forward_backward(dtype, C):
    B, H, T = 2, 3, 257
    g = torch.Generator().manual_seed(720 + C)
    x = (torch.randn(B, H, T, C, generator=g) * 0.5).to(si.TORCH_DTYPE[dtype])
    xp = (torch.randn(B, H, C, generator=g) * 0.5).to(si.TORCH_DTYPE[dtype])
    dy = torch.randn(B, H, T, C, generator=g).to(si.TORCH_DTYPE[dtype])
    w = torch.randn(H, C, 2, generator=g) * 0.7
    b = torch.randn(H, C, generator=g) * 0.1
    y = tm2.conv2_forward(x.cuda(), w.cuda(), b.cuda(), xp.cuda())
    dx, dxp, dw, db = tm2.conv2_backward(x.cuda(), w.cuda(), dy.cuda(), xp.cuda())
    torch.cuda.synchronize()
    y_r = oracle.conv2_fwd(x, w, b, xp)
    refs = oracle.conv2_bwd(x, w, dy, xp)
    if dtype == "f32":
        assert si.rel_err(y.cpu(), y_r) <= 1e-6
    else:   # the output is rounded to bf16: within half an ulp (2^-8 relative) of the exact value, plus the
        # fp32 arithmetic's error, which matters only where the two terms cancel
        yr = torch.as_tensor(y_r)
        err = (y.float().cpu().double() - yr).abs()
        assert bool((err <= 2.0 ** -8 * yr.abs() + 1e-6 * yr.pow(2).mean().sqrt()).all())
    for name, got, ref in zip(("dx", "dx_prev", "dw", "db"), (dx, dxp, dw, db), refs):
        assert si.rel_err(got.cpu(), ref) <= 1e-5, name


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv2_weight_gradients_long_sequence(dtype):
    # the weight gradients are reduced by a cluster of 8 blocks per head over token splits:
    # B T = 6002 items per head (splits of 750 and 751), several heads, C = 64
    B, H, T, C = 2, 5, 3001, 64
    g = torch.Generator().manual_seed(733)
    x = (torch.randn(B, H, T, C, generator=g) * 0.5).to(si.TORCH_DTYPE[dtype])
    dy = torch.randn(B, H, T, C, generator=g).to(si.TORCH_DTYPE[dtype])
    w = torch.randn(H, C, 2, generator=g) * 0.7
    dx, dxp, dw, db = tm2.conv2_backward(x.cuda(), w.cuda(), dy.cuda(), None)
    torch.cuda.synchronize()
    refs = oracle.conv2_bwd(x, w, dy, None)
    for name, got, ref in zip(("dx", "dx_prev", "dw", "db"), (dx, dxp, dw, db), refs):
        assert si.rel_err(got.cpu(), ref) <= 1e-5, name
    # the same call again gives the same bits (fixed reduction order)
    dx2, dxp2, dw2, db2 = tm2.conv2_backward(x.cuda(), w.cuda(), dy.cuda(), None)
    assert torch.equal(dw2.cpu(), dw.cpu()) and torch.equal(db2.cpu(), db.cpu())


# ------------------------------------------------------------------------ 2Mamba-E decode

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [16, 64])
def test_e_decode_steps_match_forward_rows(dtype, d):
    """Decode T tokens one at a time from an empty cache: each step's o and lse are the 2Mamba-E
    forward's row for that token."""
    B, H, T = 2, 3, 70
    inp = si.sequence_inputs(B, H, T, d, d, dtype=dtype, qkv_std=1.0, seed=730 + d)
    o_ref, lse_ref = oracle.e_fwd(inp["q"], inp["k"], inp["v"], inp["a"])
    g = cuda(inp)
    L = 96
    Kc = torch.zeros(B, H, L, d, dtype=g["k"].dtype, device="cuda")
    Vc = torch.zeros(B, H, L, d, dtype=g["v"].dtype, device="cuda")
    cc = torch.zeros(B, H, L, 2, device="cuda")
    tol = 1e-4 if dtype == "f32" else 2e-2
    outs, lses = [], []
    for t in range(T):
        o, lse = tm2.e_step(g["q"][:, :, t].contiguous(), g["k"][:, :, t].contiguous(), g["v"][:, :, t].contiguous(),
                            g["a"][:, :, t].contiguous(), Kc, Vc, cc, t)
        outs.append(o)
        lses.append(lse)
    torch.cuda.synchronize()
    assert si.rel_err(torch.stack(outs, 2).cpu(), o_ref) <= tol
    assert si.rel_err(torch.stack(lses, 2).cpu(), lse_ref) <= tol


def test_e_decode_after_prefill_long_cache():
    """Prefill 1500 tokens with tm2e_fill_cache, then decode 40 more (the keys are split over three
    or four blocks per head); every decoded token against the oracle forward over the whole
    sequence, at a = -1 +- 0.3 so the attention reaches far back."""
    B, H, T0, T1, d = 1, 4, 1500, 40, 64
    inp = si.sequence_inputs(B, H, T0 + T1, d, d, dtype="bf16", qkv_std=1.0, seed=740, a_mean=-3.0, a_std=0.3)
    o_ref, lse_ref = oracle.e_fwd(inp["q"], inp["k"], inp["v"], inp["a"])
    g = cuda(inp)
    L = 2048
    Kc = torch.zeros(B, H, L, d, dtype=torch.bfloat16, device="cuda")
    Vc = torch.zeros(B, H, L, d, dtype=torch.bfloat16, device="cuda")
    cc = torch.zeros(B, H, L, 2, device="cuda")
    tm2.e_fill_cache(g["k"][:, :, :T0].contiguous(), g["v"][:, :, :T0].contiguous(), g["a"][:, :, :T0].contiguous(),
                     Kc, Vc, cc)
    outs = []
    for t in range(T0, T0 + T1):
        o, _ = tm2.e_step(g["q"][:, :, t].contiguous(), g["k"][:, :, t].contiguous(), g["v"][:, :, t].contiguous(),
                          g["a"][:, :, t].contiguous(), Kc, Vc, cc, t)
        outs.append(o)
    torch.cuda.synchronize()
    assert si.rel_err(torch.stack(outs, 2).cpu(), o_ref[:, :, T0:]) <= 2e-2
    assert torch.equal(Kc[:, :, :T0 + T1].cpu(), inp["k"])
