"""fp64 CPU oracle for the 2Mamba second-order mixer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or executes anything here, and this
package never imports the product package.

The numerics live in ``tm2_oracle.c`` (plain C, fp64, OpenMP over independent
outputs), which states each formula with its source: "2Mamba2Furious: Linear
in Complexity, Competitive in Accuracy", Sec. 2, 3, 5, 6 and App. A, C.  This
module only marshals numpy arrays to it.

Pins (tests/test_oracle.py): quadratic vs recurrent forms, brute force from the
product of per-step decays at T <= 8, exact rational worked example, the
decay -> 1 and decay -> 0 limits, convex-hull and first-token invariants,
central finite differences of the gradients, PyTorch fp64 autograd of a
directly written expression, and torch's scaled_dot_product_attention for
2Mamba-E.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tm2_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile tm2_oracle.c into liboracle.so (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(_LIB)
        i, d, p = ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        _lib.orc_fwd_quadratic.argtypes = [i] * 5 + [p] * 6 + [i, i, p, p]
        _lib.orc_fwd1_recurrent.argtypes = [i] * 5 + [p] * 4 + [i, p, p]
        _lib.orc_fwd_recurrent.argtypes = [i] * 5 + [p] * 6 + [i, p, p, p, p]
        _lib.orc_step.argtypes = [i] * 4 + [p] * 6 + [i, p, p]
        _lib.orc_bwd_quadratic.argtypes = [i] * 5 + [p] * 5 + [i, i, p, p, p, p, p, p]
        _lib.orc_e_fwd.argtypes = [i] * 5 + [p] * 4 + [d, p, p]
        _lib.orc_e_bwd.argtypes = [i] * 5 + [p] * 5 + [d, p, p, p, p]
        _lib.orc_running_log_decay.argtypes = [p, ctypes.c_long, ctypes.c_long, p]
        _lib.orc_conv2_fwd.argtypes = [i] * 4 + [p] * 5
        _lib.orc_conv2_bwd.argtypes = [i] * 4 + [p] * 8
        _lib.orc_num_threads.restype = i
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def running_log_decay(a):
    """cumA[..., t] = sum_{u<=t} -softplus(a[..., u])."""
    a = _f64(a)
    out = np.empty_like(a)
    T = a.shape[-1]
    _load().orc_running_log_decay(_ptr(a), a.size // max(T, 1), T, _ptr(out))
    return out


def fwd_quadratic(q, k, v, a, normalize=True, S0=None, z0=None, order=2):
    """O(T^2) form. q,k: (B,H,T,d); v: (B,H,T,dv); a: (B,H,T). Returns (o, Z).
    order 2: 2Mamba (squared scores); order 1: the first-order mixer (no initial state)."""
    q, k, v, a, S0, z0 = map(_f64, (q, k, v, a, S0, z0))
    if order not in (1, 2) or (order == 1 and (S0 is not None or z0 is not None)):
        raise ValueError("order 1 or 2; an initial second-order state only with order 2")
    B, H, T, d = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    Z = np.zeros((B, H, T))
    _load().orc_fwd_quadratic(B, H, T, d, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                              _ptr(S0), _ptr(z0), int(normalize), int(order), _ptr(o), _ptr(Z))
    return o, Z


def fwd1_recurrent(q, k, v, a, normalize=True):
    """First-order mixer by its (d x dv) state recurrence. Returns (o, Z)."""
    q, k, v, a = map(_f64, (q, k, v, a))
    B, H, T, d = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    Z = np.zeros((B, H, T))
    _load().orc_fwd1_recurrent(B, H, T, d, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(a), int(normalize),
                               _ptr(o), _ptr(Z))
    return o, Z


def fwd_recurrent(q, k, v, a, normalize=True, S0=None, z0=None):
    """Second-order-state recurrence. Returns (o, Z, S_final (B,H,d*d,dv), z_final (B,H,d*d))."""
    q, k, v, a, S0, z0 = map(_f64, (q, k, v, a, S0, z0))
    B, H, T, d = q.shape
    dv = v.shape[-1]
    o = np.zeros((B, H, T, dv))
    Z = np.zeros((B, H, T))
    Sf = np.zeros((B, H, d * d, dv))
    zf = np.zeros((B, H, d * d))
    _load().orc_fwd_recurrent(B, H, T, d, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(a),
                              _ptr(S0), _ptr(z0), int(normalize), _ptr(o), _ptr(Z),
                              _ptr(Sf), _ptr(zf))
    return o, Z, Sf, zf


def step(q, k, v, a, S, z, normalize=True):
    """One decode step in place on the fp64 arrays S (N,H,d*d,dv), z (N,H,d*d) or None.
    q,k: (N,H,d); v: (N,H,dv); a: (N,H). Returns (o, zeta)."""
    q, k, v, a = map(_f64, (q, k, v, a))
    assert S.dtype == np.float64 and S.flags.c_contiguous
    assert z is None or (z.dtype == np.float64 and z.flags.c_contiguous)
    N, H, d = q.shape
    dv = v.shape[-1]
    o = np.zeros((N, H, dv))
    zeta = np.zeros((N, H))
    _load().orc_step(N, H, d, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(S), _ptr(z),
                     int(normalize), _ptr(o), _ptr(zeta))
    return o, zeta


def bwd_quadratic(q, k, v, a, dO, normalize=True, o=None, Z=None, order=2):
    """Gradients of the quadratic form (no initial state). Returns (dq, dk, dv, da).

    With o and Z given (normalised only), the backward uses them in place of the forward
    values it would recompute: the kernel boundary's backward takes o and Z as inputs, and
    this evaluates it as a function of those inputs (e.g. at a forward output that was
    rounded to fp32)."""
    q, k, v, a, dO, o, Z = map(_f64, (q, k, v, a, dO, o, Z))
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if (o is None) != (Z is None):
        raise ValueError("give both o and Z, or neither")
    if o is not None and (o.shape != (B, H, T, dv) or Z.shape != (B, H, T)):
        raise ValueError("o must be (B,H,T,dv) and Z (B,H,T)")
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    da = np.zeros_like(a)
    if order not in (1, 2):
        raise ValueError("order 1 or 2")
    _load().orc_bwd_quadratic(B, H, T, d, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(dO),
                              int(normalize), int(order), _ptr(o), _ptr(Z), _ptr(dq), _ptr(dk), _ptr(dvv),
                              _ptr(da))
    return dq, dk, dvv, da


def e_fwd(q, k, v, a, scale=None):
    """2Mamba-E forward, two-pass softmax. Returns (o, lse)."""
    q, k, v, a = map(_f64, (q, k, v, a))
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((B, H, T, dv))
    lse = np.zeros((B, H, T))
    _load().orc_e_fwd(B, H, T, d, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(a), float(scale),
                      _ptr(o), _ptr(lse))
    return o, lse


def e_bwd(q, k, v, a, dO, scale=None):
    """2Mamba-E backward. Returns (dq, dk, dv, da)."""
    q, k, v, a, dO = map(_f64, (q, k, v, a, dO))
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dvv = np.zeros_like(v)
    da = np.zeros_like(a)
    _load().orc_e_bwd(B, H, T, d, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(dO),
                      float(scale), _ptr(dq), _ptr(dk), _ptr(dvv), _ptr(da))
    return dq, dk, dvv, da


def conv2_fwd(x, w, b=None, x_prev=None):
    """Size-2 causal depthwise convolution: x (B,H,T,C), w (H,C,2), b (H,C), x_prev (B,H,C)."""
    x, w, b, x_prev = map(_f64, (x, w, b, x_prev))
    B, H, T, C = x.shape
    y = np.zeros_like(x)
    _load().orc_conv2_fwd(B, H, T, C, _ptr(x), _ptr(w), _ptr(b), _ptr(x_prev), _ptr(y))
    return y


def conv2_bwd(x, w, dy, x_prev=None):
    """Gradients of conv2_fwd: returns (dx, dx_prev, dw, db)."""
    x, w, dy, x_prev = map(_f64, (x, w, dy, x_prev))
    B, H, T, C = x.shape
    dx = np.zeros_like(x)
    dxp = np.zeros((B, H, C))
    dw = np.zeros((H, C, 2))
    db = np.zeros((H, C))
    _load().orc_conv2_bwd(B, H, T, C, _ptr(x), _ptr(w), _ptr(x_prev), _ptr(dy), _ptr(dx), _ptr(dxp), _ptr(dw),
                          _ptr(db))
    return dx, dxp, dw, db
