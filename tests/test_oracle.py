"""Pins of the fp64 CPU oracle against things other than itself (CPU only).

Each test names what it pins.  Sources: "2Mamba2Furious: Linear in Complexity,
Competitive in Accuracy" -- Sec. 3/5 (softplus A-mask on squared QK scores,
"softmax" normalisation), Sec. 2 (second-order state), Sec. 6 (2Mamba-E =
softmax attention with the A-mask, forgetting-transformer form), App. A
(recurrent inference), App. C (gradients w.r.t. q, k, v and the A-mask).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rnd(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


def small_case(B=2, H=2, T=37, d=4, dv=3, seed=0, a_mean=0.0):
    rng = np.random.default_rng(seed)
    q = rnd((B, H, T, d), rng, 0.5)
    k = rnd((B, H, T, d), rng, 0.5)
    v = rnd((B, H, T, dv), rng)
    a = rnd((B, H, T), rng) + a_mean
    return q, k, v, a


def relmax(x, ref):
    x, ref = np.asarray(x), np.asarray(ref)
    return np.abs(x - ref).max() / max(np.sqrt((ref ** 2).mean()), 1e-300)


# ---------------------------------------------------------------- forward forms

@pytest.mark.parametrize("normalize", [True, False])
def test_quadratic_equals_recurrent(normalize):
    """Sec. 2 / App. A: the O(T^2) form and the d^2 x dv state recurrence are the
    same function (two independent routes through the definition)."""
    q, k, v, a = small_case()
    o1, Z1 = oracle.fwd_quadratic(q, k, v, a, normalize)
    o2, Z2, Sf, zf = oracle.fwd_recurrent(q, k, v, a, normalize)
    assert relmax(o1, o2) < 1e-12
    assert relmax(Z1, Z2) < 1e-12
    assert Sf.shape == (2, 2, 16, 3) and zf.shape == (2, 2, 16)   # state (dh^2, dh)


def test_quadratic_equals_recurrent_with_initial_state():
    """The initial-state term of the quadratic form matches carrying S0, z0 through
    the recurrence."""
    q, k, v, a = small_case(T=23)
    rng = np.random.default_rng(5)
    S0 = rnd((2, 2, 16, 3), rng, 0.3)
    z0 = np.abs(rnd((2, 2, 16), rng, 0.3))
    for normalize in (True, False):
        o1, Z1 = oracle.fwd_quadratic(q, k, v, a, normalize, S0=S0, z0=z0)
        o2, Z2, _, _ = oracle.fwd_recurrent(q, k, v, a, normalize, S0=S0, z0=z0)
        assert relmax(o1, o2) < 1e-12 and relmax(Z1, Z2) < 1e-12


def test_square_identity():
    """(q.k)^2 = <q (x) q, k (x) k>: the identity behind the second-order state."""
    rng = np.random.default_rng(1)
    for _ in range(20):
        q, k = rng.standard_normal(7), rng.standard_normal(7)
        assert abs(np.dot(q, k) ** 2 - np.dot(np.outer(q, q).ravel(), np.outer(k, k).ravel())) < 1e-12


def brute_force(q, k, v, a, normalize):
    """Literal enumeration for one head: decay of step t is sigmoid(-a_t)
    (= exp(-softplus(a_t))), the mask between j <= i is the product of the decays
    of steps j+1..i, and the weight is that mask times the squared inner product."""
    T, d = q.shape
    dv = v.shape[1]
    gam = [1.0 / (1.0 + math.exp(a[t])) for t in range(T)]
    o = np.zeros((T, dv))
    Z = np.zeros(T)
    for i in range(T):
        for j in range(i + 1):
            mask = 1.0
            for t in range(j + 1, i + 1):
                mask *= gam[t]
            s = sum(q[i, m] * k[j, m] for m in range(d))
            w = mask * s * s
            Z[i] += w
            o[i] += w * v[j]
        if normalize:
            o[i] /= Z[i]
    return o, Z


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_brute_force_small_T(normalize, T):
    """Brute force on T <= 8 from the product of per-step decays pins the sign of
    a, the inclusive running sum (a token's own decay does not touch itself) and
    that the square is on the QK product only (Sec. 5)."""
    q, k, v, a = small_case(B=1, H=1, T=T, d=3, dv=2, seed=T)
    ob, Zb = brute_force(q[0, 0], k[0, 0], v[0, 0], a[0, 0], normalize)
    o1, Z1 = oracle.fwd_quadratic(q, k, v, a, normalize)
    o2, Z2, _, _ = oracle.fwd_recurrent(q, k, v, a, normalize)
    for o, Z in ((o1, Z1), (o2, Z2)):
        assert relmax(o[0, 0], ob) < 1e-12
        assert relmax(Z[0, 0], Zb) < 1e-12


def test_exact_rational_example():
    """Worked example in exact rational arithmetic (tests/golden, a = 0 so each
    decay is exactly 1/2)."""
    with open(os.path.join(GOLDEN, "exact_a0_T4_d2.json")) as f:
        g = json.load(f)
    q = np.array(g["q"], float)[None, None]
    k = np.array(g["k"], float)[None, None]
    v = np.array(g["v"], float)[None, None]
    a = np.array(g["a"], float)[None, None]
    for key, normalize in (("o_normalized", True), ("o_unnormalized", False)):
        exp = np.array([[float(Fraction(x)) for x in row] for row in g[key]])
        for o, Z in (oracle.fwd_quadratic(q, k, v, a, normalize),
                     oracle.fwd_recurrent(q, k, v, a, normalize)[:2]):
            assert np.allclose(o[0, 0], exp, rtol=1e-13, atol=1e-13)
            assert np.allclose(Z[0, 0], [float(Fraction(x)) for x in g["Z"]], rtol=1e-13)


def test_no_decay_limit_d1_closed_form():
    """a -> -inf: decay -> 1, the mixer is causal order-2 polynomial-kernel linear
    attention; with d = 1, o_i = q_i^2 cumsum(k^2 v)_i (unnormalised) and
    cumsum(k^2 v)_i / cumsum(k^2)_i (normalised)."""
    rng = np.random.default_rng(3)
    T = 50
    q, k, v = rng.standard_normal((1, 1, T, 1)), rng.standard_normal((1, 1, T, 1)), rng.standard_normal((1, 1, T, 2))
    a = np.full((1, 1, T), -40.0)
    o, Z = oracle.fwd_quadratic(q, k, v, a, False)
    ck = np.cumsum(k[0, 0, :, 0] ** 2)
    ckv = np.cumsum((k[0, 0, :, 0] ** 2)[:, None] * v[0, 0], axis=0)
    assert relmax(o[0, 0], (q[0, 0, :, 0] ** 2)[:, None] * ckv) < 1e-12
    on, _ = oracle.fwd_quadratic(q, k, v, a, True)
    assert relmax(on[0, 0], ckv / ck[:, None]) < 1e-12
    o2, _, _, _ = oracle.fwd_recurrent(q, k, v, a, False)
    assert relmax(o2[0, 0], (q[0, 0, :, 0] ** 2)[:, None] * ckv) < 1e-12


def test_full_decay_limit():
    """a -> +inf: decay -> 0, only the diagonal survives: o_i = (q_i.k_i)^2 v_i,
    and exactly v_i when normalised."""
    q, k, v, a = small_case(B=1, H=2, T=20, d=4, dv=3)
    a = np.full_like(a, 40.0)
    o, _ = oracle.fwd_quadratic(q, k, v, a, False)
    s = np.einsum("bhtd,bhtd->bht", q, k)
    assert relmax(o, s[..., None] ** 2 * v) < 1e-12
    on, _ = oracle.fwd_quadratic(q, k, v, a, True)
    assert relmax(on, v) < 1e-12


def test_normalised_output_invariants():
    """Weights are >= 0 (squared scores times a positive mask), so a normalised
    o_i lies in the convex hull of v_0..v_i; in particular o_0 = v_0."""
    q, k, v, a = small_case(B=2, H=3, T=40, d=5, dv=4, seed=9)
    o, Z = oracle.fwd_quadratic(q, k, v, a, True)
    assert np.all(Z > 0)
    assert np.allclose(o[:, :, 0], v[:, :, 0], rtol=1e-13, atol=1e-13)
    vmin = np.minimum.accumulate(v, axis=2)
    vmax = np.maximum.accumulate(v, axis=2)
    assert np.all(o >= vmin - 1e-12) and np.all(o <= vmax + 1e-12)


def test_decay_matches_log_sigmoid():
    """Sec. 6: the softplus A-mask equals the forgetting transformer's log(sigmoid(.))
    with the sign of the argument flipped: -softplus(a) = log sigmoid(-a)."""
    a = np.linspace(-30, 30, 121)[None]
    cum = oracle.running_log_decay(a)
    step = np.diff(np.concatenate([[0.0], cum[0]]))
    ref = -np.logaddexp(0.0, a[0])          # log sigmoid(-a)
    assert np.abs(step - ref).max() < 1e-12
    assert np.abs(step - np.log(1 / (1 + np.exp(a[0])))).max() < 1e-9


# ---------------------------------------------------------------- decode

def test_decode_steps_equal_forward():
    """App. A: T recurrent steps from a zero state reproduce the forward outputs."""
    q, k, v, a = small_case(B=2, H=2, T=12, d=3, dv=2, seed=4)
    S = np.zeros((2, 2, 9, 2))
    z = np.zeros((2, 2, 9))
    o_ref, Z_ref = oracle.fwd_quadratic(q, k, v, a, True)
    for t in range(12):
        o, zeta = oracle.step(q[:, :, t], k[:, :, t], v[:, :, t], a[:, :, t], S, z, True)
        assert relmax(o, o_ref[:, :, t]) < 1e-12
        assert relmax(zeta, Z_ref[:, :, t]) < 1e-12


def test_decode_from_random_state():
    """From a random S0 (z0 = 0) the steps add exp(cumA_t) (q_t (x) q_t)^T S0 to the
    output: compare with the quadratic form's initial-state term and the final state."""
    q, k, v, a = small_case(B=1, H=2, T=9, d=3, dv=2, seed=6)
    rng = np.random.default_rng(7)
    S0 = rnd((1, 2, 9, 2), rng, 0.1)
    z0 = np.zeros((1, 2, 9))
    S, z = S0.copy(), z0.copy()
    o_ref, _ = oracle.fwd_quadratic(q, k, v, a, False, S0=S0, z0=z0)
    _, _, Sf, zf = oracle.fwd_recurrent(q, k, v, a, False, S0=S0, z0=z0)
    for t in range(9):
        o, _ = oracle.step(q[:, :, t], k[:, :, t], v[:, :, t], a[:, :, t], S, z, False)
        assert relmax(o, o_ref[:, :, t]) < 1e-12
    assert relmax(S, Sf) < 1e-12 and relmax(z, zf) < 1e-12


# ---------------------------------------------------------------- gradients

def _fd_check(fwd, bwd, args, dO, idx_list, h=1e-6):
    grads = bwd(*args, dO)
    for which, idx in idx_list:
        xp = [x.copy() for x in args]
        xm = [x.copy() for x in args]
        xp[which][idx] += h
        xm[which][idx] -= h
        lp = (fwd(*xp) * dO).sum()
        lm = (fwd(*xm) * dO).sum()
        fd = (lp - lm) / (2 * h)
        g = grads[which][idx]
        assert abs(fd - g) <= 1e-7 * max(1.0, abs(g)) + 1e-8, (which, idx, fd, g)


@pytest.mark.parametrize("normalize", [True, False])
def test_gradients_finite_differences(normalize):
    """App. C: the gradients w.r.t. q, k, v and a agree with central differences."""
    q, k, v, a = small_case(B=1, H=1, T=16, d=3, dv=2, seed=11)
    rng = np.random.default_rng(12)
    dO = rng.standard_normal(v.shape)
    fwd = lambda q, k, v, a: oracle.fwd_quadratic(q, k, v, a, normalize)[0]
    bwd = lambda q, k, v, a, dO: oracle.bwd_quadratic(q, k, v, a, dO, normalize)
    idx = []
    for which, shp in enumerate((q.shape, k.shape, v.shape, a.shape)):
        for _ in range(10):
            idx.append((which, tuple(int(rng.integers(0, s)) for s in shp)))
    _fd_check(fwd, bwd, [q, k, v, a], dO, idx)


def test_e_gradients_finite_differences():
    q, k, v, a = small_case(B=1, H=1, T=16, d=3, dv=2, seed=13)
    rng = np.random.default_rng(14)
    dO = rng.standard_normal(v.shape)
    fwd = lambda q, k, v, a: oracle.e_fwd(q, k, v, a, 0.7)[0]
    bwd = lambda q, k, v, a, dO: oracle.e_bwd(q, k, v, a, dO, 0.7)
    idx = []
    for which, shp in enumerate((q.shape, k.shape, v.shape, a.shape)):
        for _ in range(10):
            idx.append((which, tuple(int(rng.integers(0, s)) for s in shp)))
    _fd_check(fwd, bwd, [q, k, v, a], dO, idx)


@pytest.mark.parametrize("normalize", [True, False])
def test_gradients_vs_torch_autograd(normalize):
    """PyTorch fp64 autograd of a directly written dense expression (independent of
    the oracle's hand-written chain rule)."""
    q, k, v, a = small_case(B=2, H=1, T=48, d=6, dv=5, seed=21)
    dO = np.random.default_rng(22).standard_normal(v.shape)
    tq, tk, tv, ta = (torch.tensor(x, requires_grad=True) for x in (q, k, v, a))
    cum = torch.cumsum(-torch.nn.functional.softplus(ta), -1)
    T = q.shape[2]
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    diff = torch.where(causal, cum[..., :, None] - cum[..., None, :], torch.tensor(-math.inf, dtype=torch.float64))
    W = torch.exp(diff) * (tq @ tk.transpose(-1, -2)) ** 2
    o = W @ tv
    if normalize:
        o = o / W.sum(-1, keepdim=True)
    (o * torch.tensor(dO)).sum().backward()
    dq, dk, dv, da = oracle.bwd_quadratic(q, k, v, a, dO, normalize)
    assert relmax(o.detach().numpy(), oracle.fwd_quadratic(q, k, v, a, normalize)[0]) < 1e-12
    for g, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad), (da, ta.grad)):
        assert relmax(g, ref.numpy()) < 1e-10


def test_backward_at_given_forward_values_vs_torch_autograd():
    """The normalised backward as a function of the forward values it is given (the kernel
    boundary's backward takes o and Z as inputs, App. C): with o^g, Z^g held fixed, its
    gradients are those of F = sum_i (dO_i . N_i - (dO_i . o^g_i) Z_i) / Z^g_i, N_i and Z_i the
    weighted sums of the quadratic form, which torch fp64 autograd differentiates directly.
    Pinned at perturbed o^g, Z^g (where it differs from the plain backward) and at the exact
    ones (where it must equal it)."""
    q, k, v, a = small_case(B=1, H=2, T=40, d=5, dv=4, seed=51)
    rng = np.random.default_rng(52)
    dO = rng.standard_normal(v.shape)
    o, Z = oracle.fwd_quadratic(q, k, v, a, True)
    exact = oracle.bwd_quadratic(q, k, v, a, dO, True)
    same = oracle.bwd_quadratic(q, k, v, a, dO, True, o=o, Z=Z)
    for x, y in zip(same, exact):
        assert np.array_equal(x, y)
    og = o + 1e-2 * rng.standard_normal(o.shape)
    Zg = Z * (1 + 1e-2 * rng.standard_normal(Z.shape))
    got = oracle.bwd_quadratic(q, k, v, a, dO, True, o=og, Z=Zg)
    tq, tk, tv, ta = (torch.tensor(x, requires_grad=True) for x in (q, k, v, a))
    cum = torch.cumsum(-torch.nn.functional.softplus(ta), -1)
    T = q.shape[2]
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    diff = torch.where(causal, cum[..., :, None] - cum[..., None, :], torch.tensor(-math.inf, dtype=torch.float64))
    W = torch.exp(diff) * (tq @ tk.transpose(-1, -2)) ** 2
    N, Zs = W @ tv, W.sum(-1)
    tdO, tog, tZg = torch.tensor(dO), torch.tensor(og), torch.tensor(Zg)
    F = (((tdO * N).sum(-1) - (tdO * tog).sum(-1) * Zs) / tZg).sum()
    F.backward()
    for g, ref in zip(got, (tq.grad, tk.grad, tv.grad, ta.grad)):
        assert relmax(g, ref.numpy()) < 1e-10
    assert relmax(got[0], exact[0]) > 1e-4   # the given values do enter


@pytest.mark.parametrize("variant", ["norm", "raw", "e"])
def test_first_token_decay_gradient_is_zero(variant):
    """Shifting a_0 shifts every cumA_t equally, and only differences of cumA enter
    the output, so da_0 = 0 exactly (row-axis and column-axis sums cancel, App. C.1)."""
    q, k, v, a = small_case(B=1, H=2, T=30, d=4, dv=3, seed=31)
    dO = np.random.default_rng(32).standard_normal(v.shape)
    if variant == "e":
        _, _, _, da = oracle.e_bwd(q, k, v, a, dO)
    else:
        _, _, _, da = oracle.bwd_quadratic(q, k, v, a, dO, variant == "norm")
    assert np.abs(da[..., 0]).max() < 1e-10 * np.abs(da).max()
    assert np.abs(da[..., 1:]).max() > 1e-3


def test_unnormalised_decay_gradient_closed_form():
    """For the unnormalised mixer the A-mask gradient has the closed form
    dcumA_t = dO_t . o_t - v_t . dv_t (row-axis sum minus column-axis sum)."""
    q, k, v, a = small_case(B=1, H=1, T=25, d=4, dv=3, seed=41)
    dO = np.random.default_rng(42).standard_normal(v.shape)
    o, _ = oracle.fwd_quadratic(q, k, v, a, False)
    dq, dk, dv, da = oracle.bwd_quadratic(q, k, v, a, dO, False)
    dcum = (dO * o).sum(-1) - (v * dv).sum(-1)
    dl = np.flip(np.cumsum(np.flip(dcum, -1), -1), -1)
    sig = 1 / (1 + np.exp(-a))
    assert relmax(da, -sig * dl) < 1e-11


# ---------------------------------------------------------------- 2Mamba-E

def _sdpa_reference(q, k, v, a, scale, dO):
    tq, tk, tv, ta = (torch.tensor(x, requires_grad=True) for x in (q, k, v, a))
    cum = torch.cumsum(-torch.nn.functional.softplus(ta), -1)
    T = q.shape[2]
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    bias = torch.where(causal, cum[..., :, None] - cum[..., None, :], torch.tensor(-math.inf, dtype=torch.float64))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=bias, scale=scale)
    (o * torch.tensor(dO)).sum().backward()
    return o.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy(), ta.grad.numpy()


def test_e_variant_matches_sdpa_with_decay_bias():
    """Sec. 6: 2Mamba-E is softmax attention whose logits carry the additive A-mask
    cumA_i - cumA_j (the forgetting-transformer form): torch's SDPA with that float
    mask, and its autograd, pin the forward and all four gradients."""
    q, k, v, a = small_case(B=2, H=2, T=33, d=8, dv=6, seed=51)
    q, k = q * 2, k * 2
    dO = np.random.default_rng(52).standard_normal(v.shape)
    scale = 1 / math.sqrt(8)
    o_ref, dq_r, dk_r, dv_r, da_r = _sdpa_reference(q, k, v, a, scale, dO)
    o, lse = oracle.e_fwd(q, k, v, a, scale)
    assert relmax(o, o_ref) < 1e-12
    dq, dk, dv, da = oracle.e_bwd(q, k, v, a, dO, scale)
    for g, ref in ((dq, dq_r), (dk, dk_r), (dv, dv_r), (da, da_r)):
        assert relmax(g, ref) < 1e-10


def test_e_variant_no_decay_is_causal_softmax():
    """a -> -inf removes the A-mask: textbook causal softmax attention."""
    q, k, v, a = small_case(B=1, H=2, T=40, d=8, dv=8, seed=61)
    a = np.full_like(a, -40.0)
    o, lse = oracle.e_fwd(q, k, v, a, 0.5)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), torch.tensor(k), torch.tensor(v), is_causal=True, scale=0.5).numpy()
    assert relmax(o, ref) < 1e-12
    s = 0.5 * np.einsum("bhid,bhjd->bhij", q, k)
    s = np.where(np.tril(np.ones((40, 40), bool)), s, -np.inf)
    assert np.abs(lse - np.log(np.exp(s).sum(-1))).max() < 1e-12


# ---------------------------------------------------------------- first-order mixer (order 1)
# "2Mamba2Furious", Sec. 4 (Mamba-2S: the softplus A-mask on the score q.k itself) and Sec. 2
# (first-order linear attention keeps a (dh, dh) state).

def brute_force_first_order(q, k, v, a, normalize):
    """Literal enumeration for one head: product of per-step decays times the score itself."""
    T, d = q.shape
    dv = v.shape[1]
    gam = [1.0 / (1.0 + math.exp(a[t])) for t in range(T)]
    o = np.zeros((T, dv))
    Z = np.zeros(T)
    for i in range(T):
        for j in range(i + 1):
            mask = 1.0
            for t in range(j + 1, i + 1):
                mask *= gam[t]
            w = mask * sum(q[i, m] * k[j, m] for m in range(d))
            Z[i] += w
            o[i] += w * v[j]
        if normalize:
            o[i] /= Z[i]
    return o, Z


@pytest.mark.parametrize("normalize", [True, False])
def test_first_order_quadratic_equals_recurrent(normalize):
    """The O(T^2) form with order 1 and the (d x dv) state recurrence are the same function."""
    q, k, v, a = small_case(T=29, seed=61)
    o1, Z1 = oracle.fwd_quadratic(q, k, v, a, normalize, order=1)
    o2, Z2 = oracle.fwd1_recurrent(q, k, v, a, normalize)
    assert relmax(o1, o2) < 1e-12 and relmax(Z1, Z2) < 1e-12


@pytest.mark.parametrize("T", [1, 3, 7])
def test_first_order_brute_force_small_T(T):
    q, k, v, a = small_case(B=1, H=1, T=T, d=3, dv=2, seed=70 + T)
    for normalize in (True, False):
        ob, Zb = brute_force_first_order(q[0, 0], k[0, 0], v[0, 0], a[0, 0], normalize)
        o1, Z1 = oracle.fwd_quadratic(q, k, v, a, normalize, order=1)
        assert relmax(o1[0, 0], ob) < 1e-12 and relmax(Z1[0, 0], Zb) < 1e-12


def test_first_order_limits():
    """No decay, d = 1: o_i = q_i cumsum(k v)_i; full decay: o_i = (q_i . k_i) v_i."""
    rng = np.random.default_rng(81)
    T = 40
    q, k, v = rng.standard_normal((1, 1, T, 1)), rng.standard_normal((1, 1, T, 1)), rng.standard_normal((1, 1, T, 2))
    o, _ = oracle.fwd_quadratic(q, k, v, np.full((1, 1, T), -40.0), False, order=1)
    ckv = np.cumsum(k[0, 0, :, 0][:, None] * v[0, 0], axis=0)
    assert relmax(o[0, 0], q[0, 0, :, 0][:, None] * ckv) < 1e-12
    q, k, v, a = small_case(B=1, H=2, T=20, d=4, dv=3, seed=82)
    o, _ = oracle.fwd_quadratic(q, k, v, np.full_like(a, 40.0), False, order=1)
    assert relmax(o, np.einsum("bhtd,bhtd->bht", q, k)[..., None] * v) < 1e-12


@pytest.mark.parametrize("normalize", [True, False])
def test_first_order_gradients(normalize):
    """Order-1 gradients against central differences and torch fp64 autograd of a directly
    written dense expression; da_0 = 0 as for order 2."""
    q, k, v, a = small_case(B=1, H=1, T=16, d=3, dv=2, seed=83)
    rng = np.random.default_rng(84)
    dO = rng.standard_normal(v.shape)
    fwd = lambda q, k, v, a: oracle.fwd_quadratic(q, k, v, a, normalize, order=1)[0]
    bwd = lambda q, k, v, a, dO: oracle.bwd_quadratic(q, k, v, a, dO, normalize, order=1)
    idx = []
    for which, shp in enumerate((q.shape, k.shape, v.shape, a.shape)):
        for _ in range(8):
            idx.append((which, tuple(int(rng.integers(0, s)) for s in shp)))
    _fd_check(fwd, bwd, [q, k, v, a], dO, idx)
    tq, tk, tv, ta = (torch.tensor(x, requires_grad=True) for x in (q, k, v, a))
    cum = torch.cumsum(-torch.nn.functional.softplus(ta), -1)
    T = q.shape[2]
    causal = torch.tril(torch.ones(T, T, dtype=torch.bool))
    diff = torch.where(causal, cum[..., :, None] - cum[..., None, :], torch.tensor(-math.inf, dtype=torch.float64))
    W = torch.exp(diff) * (tq @ tk.transpose(-1, -2))
    o = W @ tv
    if normalize:
        o = o / W.sum(-1, keepdim=True)
    (o * torch.tensor(dO)).sum().backward()
    grads = bwd(q, k, v, a, dO)
    for g, ref in zip(grads, (tq.grad, tk.grad, tv.grad, ta.grad)):
        assert relmax(g, ref.numpy()) < 1e-10
    assert np.abs(grads[3][..., 0]).max() < 1e-10 * np.abs(grads[3]).max()


# ---------------------------------------------------------------- input convolution (window 2)

def test_conv2_against_torch_conv1d_and_autograd():
    """The size-2 causal depthwise convolution (Sec. 3-4) against torch's conv1d in fp64 (groups =
    channels, left padding 1, the kernel reversed: conv1d weight [.., 0] multiplies x_{t-1}) with
    an initial token x_prev prepended, and its gradients against torch autograd."""
    rng = np.random.default_rng(91)
    B, H, T, C = 2, 3, 17, 4
    x = rng.standard_normal((B, H, T, C))
    w = rng.standard_normal((H, C, 2))
    b = rng.standard_normal((H, C))
    xp = rng.standard_normal((B, H, C))
    dy = rng.standard_normal((B, H, T, C))
    y = oracle.conv2_fwd(x, w, b, xp)
    tx, tw, tb, txp = (torch.tensor(z, requires_grad=True) for z in (x, w, b, xp))
    seq = torch.cat([txp[:, :, None], tx], dim=2)                       # (B,H,T+1,C)
    inp = seq.permute(0, 1, 3, 2).reshape(B, H * C, T + 1)
    ker = torch.stack([tw[..., 1], tw[..., 0]], dim=-1).reshape(H * C, 1, 2)
    out = torch.nn.functional.conv1d(inp, ker, bias=tb.reshape(H * C), groups=H * C)   # (B,H*C,T)
    ty = out.reshape(B, H, C, T).permute(0, 1, 3, 2)
    assert relmax(y, ty.detach().numpy()) < 1e-13
    (ty * torch.tensor(dy)).sum().backward()
    dx, dxp, dw, db = oracle.conv2_bwd(x, w, dy, xp)
    for g, ref in ((dx, tx.grad), (dxp, txp.grad), (dw, tw.grad), (db, tb.grad)):
        assert relmax(g, ref.numpy()) < 1e-12


def test_conv2_identity_and_shift():
    """w = (1, 0) is the identity; w = (0, 1) shifts by one token (x_prev first)."""
    rng = np.random.default_rng(92)
    x = rng.standard_normal((1, 2, 9, 3))
    xp = rng.standard_normal((1, 2, 3))
    one = np.zeros((2, 3, 2))
    one[..., 0] = 1.0
    assert np.array_equal(oracle.conv2_fwd(x, one, None, xp), x)
    sh = np.zeros((2, 3, 2))
    sh[..., 1] = 1.0
    ys = oracle.conv2_fwd(x, sh, None, xp)
    assert np.array_equal(ys[:, :, 1:], x[:, :, :-1]) and np.array_equal(ys[:, :, 0], xp)
