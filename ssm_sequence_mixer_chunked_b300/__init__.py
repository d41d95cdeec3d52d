"""B300-native 2Mamba second-order sequence mixer -- thin Python binding over libtm2.so.

The method ("2Mamba2Furious: Linear in Complexity, Competitive in Accuracy", Sec. 5):
    o_i = sum_{j<=i} exp(cumA_i - cumA_j) (q_i . k_j)^2 v_j  [/ Z_i],
    cumA_t = sum_{u<=t} -softplus(a_u),
its recurrent decode step on the (d^2, dv) state (Sec. 2, App. A), the gradients
(App. C) and the exponentiated-score variant 2Mamba-E (Sec. 6).

Every step of the computation runs in the CUDA kernels of libtm2.so; this module only
checks tensors, allocates outputs and workspace with PyTorch and passes raw pointers
and sizes through the C ABI declared in include/tm2.h.  There is no CPU path: if the
library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = ["forward", "backward", "step", "step_conv", "state_pack", "state_unpack", "e_forward", "e_backward",
           "e_step", "e_fill_cache", "conv2_forward", "conv2_backward", "forward_quadratic",
           "backward_quadratic", "library_path",
           "forward_workspace_bytes", "backward_workspace_bytes", "workspace_bytes", "TM2Error",
           "NORMALIZE", "REUSE_STATES"]

PKG = os.path.dirname(os.path.abspath(__file__))
# TM2_DEBUG=1 selects the bounds-checked build (python -m ssm_sequence_mixer_chunked_b300.build --debug)
_LIB_PATH = os.path.join(PKG, "libtm2_debug.so" if os.environ.get("TM2_DEBUG") == "1" else "libtm2.so")
NORMALIZE = 1
REUSE_STATES = 2
PACKED_STATE = 4
GRADS_INPUT_DTYPE = 8
_DTYPES = {torch.float32: 0, torch.bfloat16: 1}
_lib = None


class TM2Error(RuntimeError):
    pass


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise TM2Error("%s is not built; run `python -m ssm_sequence_mixer_chunked_b300.build%s`"
                       % (_LIB_PATH, " --debug" if _LIB_PATH.endswith("_debug.so") else ""))
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, U, S, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t, ctypes.c_float
    lib.tm2_version.restype = I
    lib.tm2_status_string.restype = ctypes.c_char_p
    lib.tm2_status_string.argtypes = [I]
    for name in ("tm2_forward_workspace", "tm2_backward_workspace"):
        getattr(lib, name).restype = S
        getattr(lib, name).argtypes = [I] * 7 + [U]
    for name in ("tm2e_forward_workspace", "tm2e_backward_workspace"):
        getattr(lib, name).restype = S
        getattr(lib, name).argtypes = [I] * 6
    lib.tm2_forward.restype = I
    lib.tm2_forward.argtypes = [P] * 10 + [I] * 7 + [U, P, S, P]
    lib.tm2_backward.restype = I
    lib.tm2_backward.argtypes = [P] * 11 + [I] * 7 + [U, P, S, P]
    lib.tm2_step.restype = I
    lib.tm2_step.argtypes = [P] * 8 + [I] * 5 + [U, P]
    lib.tm2e_forward.restype = I
    lib.tm2e_forward.argtypes = [P] * 6 + [I] * 5 + [F, I, P, S, P]
    lib.tm2e_backward.restype = I
    lib.tm2e_backward.argtypes = [P] * 11 + [I] * 5 + [F, I, U, P, S, P]
    for name in ("tm2q_forward_workspace", "tm2q_backward_workspace"):
        getattr(lib, name).restype = S
        getattr(lib, name).argtypes = [I] * 7 + [U]
    lib.tm2q_forward.restype = I
    lib.tm2q_forward.argtypes = [P] * 6 + [I] * 7 + [U, P, S, P]
    lib.tm2q_backward.restype = I
    lib.tm2q_backward.argtypes = [P] * 11 + [I] * 7 + [U, P, S, P]
    lib.tm2_step_conv.restype = I
    lib.tm2_step_conv.argtypes = [P] * 17 + [I] * 5 + [U, P]
    for name in ("tm2_state_pack", "tm2_state_unpack"):
        getattr(lib, name).restype = I
        getattr(lib, name).argtypes = [P] * 4 + [I] * 3 + [P]
    lib.tm2e_step_workspace.restype = S
    lib.tm2e_step_workspace.argtypes = [I] * 6
    lib.tm2e_step.restype = I
    lib.tm2e_step.argtypes = [P] * 7 + [I] * 2 + [P] * 2 + [I] * 4 + [F, I, P, S, P]
    lib.tm2e_fill_cache_workspace.restype = S
    lib.tm2e_fill_cache_workspace.argtypes = [I] * 6
    lib.tm2e_fill_cache.restype = I
    lib.tm2e_fill_cache.argtypes = [P] * 6 + [I] * 7 + [P, S, P]
    lib.tm2_conv2_forward.restype = I
    lib.tm2_conv2_forward.argtypes = [P] * 5 + [I] * 5 + [P]
    lib.tm2_conv2_backward.restype = I
    lib.tm2_conv2_backward.argtypes = [P] * 8 + [I] * 5 + [P]
    lib.tm2_poll_status.restype = I
    lib.tm2_last_cuda_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def lib():
    """The loaded ctypes library (raw C ABI)."""
    return _load()


def status_string(st: int) -> str:
    return _load().tm2_status_string(int(st)).decode()


def _check(st: int):
    if st != 0:
        msg = status_string(st)
        if st == -5:
            msg += " (" + _load().tm2_last_cuda_error().decode() + ")"
        raise TM2Error(msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _seq_checks(q, k, v, a):
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a)):
        if not t.is_cuda:
            raise TM2Error("%s must be a CUDA tensor" % name)
        if not t.is_contiguous():
            raise TM2Error("%s must be contiguous" % name)
    if q.dtype not in _DTYPES or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TM2Error("q, k, v must share one dtype in {float32, bfloat16}")
    if a.dtype != torch.float32:
        raise TM2Error("a must be float32")
    B, H, T, d = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or a.shape != (B, H, T):
        raise TM2Error("shape mismatch: q,k (B,H,T,d), v (B,H,T,dv), a (B,H,T)")
    return B, H, T, d, dv, _DTYPES[q.dtype]


def _grad_buffers(q, k, v, a, lowp):
    """dq, dk, dv in fp32 (or the input dtype with lowp), da in fp32: the backward's output types."""
    gt = q.dtype if lowp else torch.float32
    return (torch.empty(q.shape, dtype=gt, device=q.device), torch.empty(k.shape, dtype=gt, device=q.device),
            torch.empty(v.shape, dtype=gt, device=q.device), torch.empty(a.shape, dtype=torch.float32, device=q.device))


def _workspace(nbytes, device, workspace):
    if nbytes == 0:
        return None
    if workspace is not None and workspace.numel() * workspace.element_size() >= nbytes:
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def forward_workspace_bytes(B, H, T, d, dv, chunk=0, dtype=torch.bfloat16, normalize=True):
    return int(_load().tm2_forward_workspace(B, H, T, d, dv, chunk, _DTYPES[dtype],
                                             NORMALIZE if normalize else 0))


def backward_workspace_bytes(B, H, T, d, dv, chunk=0, dtype=torch.bfloat16, normalize=True):
    return int(_load().tm2_backward_workspace(B, H, T, d, dv, chunk, _DTYPES[dtype],
                                              NORMALIZE if normalize else 0))


def workspace_bytes(B, H, T, d, dv, chunk=0, dtype=torch.bfloat16, normalize=True):
    """Bytes of one workspace that serves a forward() and the backward() that reuses its states."""
    return max(forward_workspace_bytes(B, H, T, d, dv, chunk, dtype, normalize),
               backward_workspace_bytes(B, H, T, d, dv, chunk, dtype, normalize))


def forward(q, k, v, a, *, normalize=True, chunk=0, S0=None, z0=None, return_state=False,
            out=None, Z=None, workspace=None, stream=None):
    """2Mamba forward.  Returns (o, Z) or, with return_state, (o, Z, S_final, z_final)."""
    B, H, T, d, dv, dt = _seq_checks(q, k, v, a)
    L = _load()
    flags = NORMALIZE if normalize else 0
    o = torch.empty(v.shape, dtype=torch.float32, device=q.device) if out is None else out
    Z = torch.empty((B, H, T), dtype=torch.float32, device=q.device) if Z is None else Z
    Sf = zf = None
    if return_state:
        Sf = torch.empty((B, H, d * d, dv), dtype=torch.float32, device=q.device)
        zf = torch.empty((B, H, d * d), dtype=torch.float32, device=q.device)
    ws = _workspace(L.tm2_forward_workspace(B, H, T, d, dv, chunk, dt, flags), q.device, workspace)
    nbytes = 0 if ws is None else ws.numel()
    _check(L.tm2_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(S0), _ptr(z0), _ptr(o), _ptr(Z),
                         _ptr(Sf), _ptr(zf), B, H, T, d, dv, chunk, dt, flags, _ptr(ws), nbytes,
                         _stream(stream)))
    return (o, Z, Sf, zf) if return_state else (o, Z)


def backward(q, k, v, a, o, Z, dO, *, normalize=True, chunk=0, workspace=None, stream=None,
             grads=None, reuse_states=False, lowp_grads=False):
    """2Mamba backward.  Returns (dq, dk, dv, da).  With reuse_states=True, `workspace` must
    be the buffer the matching forward() call used (sized with workspace_bytes()); the chunk
    states the forward left there are read instead of recomputed.  lowp_grads: dq, dk, dv in
    the input dtype (rounded from the fp32 values) instead of fp32."""
    B, H, T, d, dv, dt = _seq_checks(q, k, v, a)
    L = _load()
    flags = (NORMALIZE if normalize else 0) | (REUSE_STATES if reuse_states else 0) | \
        (GRADS_INPUT_DTYPE if lowp_grads else 0)
    if reuse_states and (workspace is None or workspace.numel() * workspace.element_size() <
                         L.tm2_backward_workspace(B, H, T, d, dv, chunk, dt, flags)):
        raise TM2Error("reuse_states needs the forward's workspace, sized with workspace_bytes()")
    if grads is None:
        grads = _grad_buffers(q, k, v, a, lowp_grads)
    dq, dk, dvv, da = grads
    ws = _workspace(L.tm2_backward_workspace(B, H, T, d, dv, chunk, dt, flags), q.device, workspace)
    nbytes = 0 if ws is None else ws.numel()
    _check(L.tm2_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(o), _ptr(Z), _ptr(dO), _ptr(dq),
                          _ptr(dk), _ptr(dvv), _ptr(da), B, H, T, d, dv, chunk, dt, flags, _ptr(ws),
                          nbytes, _stream(stream)))
    return dq, dk, dvv, da


def _step_checks(q, k, v, a, S, z, packed):
    N, H, d = q.shape
    dv = v.shape[-1]
    for name, t in (("q", q), ("k", k), ("v", v), ("a", a), ("S", S)) + ((("z", z),) if z is not None else ()):
        if not t.is_cuda or not t.is_contiguous():
            raise TM2Error("%s must be a contiguous CUDA tensor" % name)
    if q.dtype not in _DTYPES or S.dtype != torch.float32 or a.dtype != torch.float32:
        raise TM2Error("q, k, v in {float32, bfloat16}; a, S, z float32")
    rows = d * (d + 1) // 2 if packed else d * d
    if S.shape != (N, H, rows, dv) or (z is not None and z.shape != (N, H, rows)):
        raise TM2Error("S must be (N,H,%d,dv) and z (N,H,%d)" % (rows, rows))
    return N, H, d, dv


def step(q, k, v, a, S, z, *, normalize=True, packed=False, out=None, Z=None, stream=None):
    """One decode step, updating S (N,H,d*d,dv) and z (N,H,d*d) in place -- or, with packed=True,
    the symmetric-packed S (N,H,d(d+1)/2,dv) and z (N,H,d(d+1)/2).  Returns (o, zeta)."""
    N, H, d, dv = _step_checks(q, k, v, a, S, z, packed)
    L = _load()
    o = torch.empty(v.shape, dtype=torch.float32, device=q.device) if out is None else out
    Z = torch.empty((N, H), dtype=torch.float32, device=q.device) if Z is None else Z
    flags = (NORMALIZE if normalize else 0) | (PACKED_STATE if packed else 0)
    _check(L.tm2_step(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(S), _ptr(z), _ptr(o), _ptr(Z), N, H, d,
                      dv, _DTYPES[q.dtype], flags, _stream(stream)))
    return o, Z


def step_conv(q, k, v, a, conv_w, conv_b, caches, S, z, *, normalize=True, packed=False, out=None, Z=None,
              stream=None):
    """Decode step with the size-2 input convolution on q, k, v: conv_w = (wq, wk, wv), each (H,d,2)
    fp32; conv_b = (bq, bk, bv) of (H,d) fp32 or None; caches = (cq, ck, cv), each (N,H,d) in the
    input dtype, updated in place (the raw current token replaces the previous one)."""
    N, H, d, dv = _step_checks(q, k, v, a, S, z, packed)
    L = _load()
    o = torch.empty(v.shape, dtype=torch.float32, device=q.device) if out is None else out
    Z = torch.empty((N, H), dtype=torch.float32, device=q.device) if Z is None else Z
    bq, bk, bv = conv_b if conv_b is not None else (None, None, None)
    flags = (NORMALIZE if normalize else 0) | (PACKED_STATE if packed else 0)
    _check(L.tm2_step_conv(_ptr(q), _ptr(k), _ptr(v), _ptr(a), *(_ptr(t) for t in conv_w), _ptr(bq), _ptr(bk),
                           _ptr(bv), *(_ptr(t) for t in caches), _ptr(S), _ptr(z), _ptr(o), _ptr(Z), N, H, d, dv,
                           _DTYPES[q.dtype], flags, _stream(stream)))
    return o, Z


def state_pack(S, z=None, *, stream=None):
    """Full states (NH..., d*d, dv) -> symmetric-packed (..., d(d+1)/2, dv) (their symmetric part)."""
    d = int(round(S.shape[-2] ** 0.5))
    lead = S.shape[:-2]
    R = d * (d + 1) // 2
    Sp = torch.empty(lead + (R, S.shape[-1]), dtype=torch.float32, device=S.device)
    zp = None if z is None else torch.empty(lead + (R,), dtype=torch.float32, device=S.device)
    nh = S.numel() // (d * d * S.shape[-1])
    _check(_load().tm2_state_pack(_ptr(S), _ptr(z), _ptr(Sp), _ptr(zp), nh, d, S.shape[-1], _stream(stream)))
    return Sp, zp


def state_unpack(Sp, zp=None, *, d, stream=None):
    """Symmetric-packed states back to the full (d*d)-row layout."""
    lead = Sp.shape[:-2]
    S = torch.empty(lead + (d * d, Sp.shape[-1]), dtype=torch.float32, device=Sp.device)
    z = None if zp is None else torch.empty(lead + (d * d,), dtype=torch.float32, device=Sp.device)
    nh = Sp.numel() // (Sp.shape[-2] * Sp.shape[-1])
    _check(_load().tm2_state_unpack(_ptr(Sp), _ptr(zp), _ptr(S), _ptr(z), nh, d, Sp.shape[-1], _stream(stream)))
    return S, z


def e_step(q, k, v, a, K_cache, V_cache, cum_cache, pos, *, scale=None, out=None, lse=None, workspace=None,
           stream=None):
    """2Mamba-E decode step over the KV cache at position pos (caches (N,H,L,d), (N,H,L,dv),
    (N,H,L,2)); appends the token.  Returns (o, lse)."""
    N, H, d = q.shape
    dv = v.shape[-1]
    Lc = K_cache.shape[2]
    L = _load()
    dt = _DTYPES[q.dtype]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty((N, H, dv), dtype=torch.float32, device=q.device) if out is None else out
    lse = torch.empty((N, H), dtype=torch.float32, device=q.device) if lse is None else lse
    ws = _workspace(L.tm2e_step_workspace(N, H, Lc, d, dv, dt), q.device, workspace)
    nbytes = 0 if ws is None else ws.numel()
    _check(L.tm2e_step(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(K_cache), _ptr(V_cache), _ptr(cum_cache), int(pos),
                       Lc, _ptr(o), _ptr(lse), N, H, d, dv, scale, dt, _ptr(ws), nbytes, _stream(stream)))
    return o, lse


def e_fill_cache(k, v, a, K_cache, V_cache, cum_cache, *, workspace=None, stream=None):
    """Writes a prefill's keys, values and A-mask running sums into rows 0..T-1 of the caches."""
    B, H, T, d = k.shape
    dv = v.shape[-1]
    L = _load()
    dt = _DTYPES[k.dtype]
    ws = _workspace(L.tm2e_fill_cache_workspace(B, H, T, d, dv, dt), k.device, workspace)
    nbytes = 0 if ws is None else ws.numel()
    _check(L.tm2e_fill_cache(_ptr(k), _ptr(v), _ptr(a), _ptr(K_cache), _ptr(V_cache), _ptr(cum_cache), B, H, T,
                             K_cache.shape[2], d, dv, dt, _ptr(ws), nbytes, _stream(stream)))


def conv2_forward(x, w, b=None, x_prev=None, *, stream=None):
    """Size-2 causal input convolution of x (B,H,T,C); w (H,C,2), b (H,C) fp32; x_prev (B,H,C)."""
    B, H, T, C = x.shape
    y = torch.empty_like(x)
    _check(_load().tm2_conv2_forward(_ptr(x), _ptr(w), _ptr(b), _ptr(x_prev), _ptr(y), B, H, T, C,
                                     _DTYPES[x.dtype], _stream(stream)))
    return y


def conv2_backward(x, w, dy, x_prev=None, *, stream=None):
    """Gradients of conv2_forward: (dx, dx_prev, dw, db), fp32."""
    B, H, T, C = x.shape
    dx = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    dxp = torch.empty((B, H, C), dtype=torch.float32, device=x.device)
    dw = torch.empty((H, C, 2), dtype=torch.float32, device=x.device)
    db = torch.empty((H, C), dtype=torch.float32, device=x.device)
    _check(_load().tm2_conv2_backward(_ptr(x), _ptr(w), _ptr(x_prev), _ptr(dy), _ptr(dx), _ptr(dxp), _ptr(dw),
                                      _ptr(db), B, H, T, C, _DTYPES[x.dtype], _stream(stream)))
    return dx, dxp, dw, db


def forward_quadratic(q, k, v, a, *, order=2, normalize=True, workspace=None, stream=None, out=None, Z=None):
    """Quadratic (C = T) form of the mixer: order 2 is 2Mamba (the same function as forward()),
    order 1 the first-order mixer with the softplus A-mask.  Returns (o, Z)."""
    B, H, T, d, dv, dt = _seq_checks(q, k, v, a)
    L = _load()
    flags = NORMALIZE if normalize else 0
    o = torch.empty(v.shape, dtype=torch.float32, device=q.device) if out is None else out
    Z = torch.empty((B, H, T), dtype=torch.float32, device=q.device) if Z is None else Z
    ws = _workspace(L.tm2q_forward_workspace(B, H, T, d, dv, order, dt, flags), q.device, workspace)
    nbytes = 0 if ws is None else ws.numel()
    _check(L.tm2q_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(o), _ptr(Z), B, H, T, d, dv, order, dt, flags,
                          _ptr(ws), nbytes, _stream(stream)))
    return o, Z


def backward_quadratic(q, k, v, a, o, Z, dO, *, order=2, normalize=True, workspace=None, stream=None,
                       grads=None, lowp_grads=False):
    """Backward of forward_quadratic.  Returns (dq, dk, dv, da)."""
    B, H, T, d, dv, dt = _seq_checks(q, k, v, a)
    L = _load()
    flags = (NORMALIZE if normalize else 0) | (GRADS_INPUT_DTYPE if lowp_grads else 0)
    if grads is None:
        grads = _grad_buffers(q, k, v, a, lowp_grads)
    dq, dk, dvv, da = grads
    ws = _workspace(L.tm2q_backward_workspace(B, H, T, d, dv, order, dt, flags), q.device, workspace)
    nbytes = 0 if ws is None else ws.numel()
    _check(L.tm2q_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(o), _ptr(Z), _ptr(dO), _ptr(dq), _ptr(dk),
                           _ptr(dvv), _ptr(da), B, H, T, d, dv, order, dt, flags, _ptr(ws), nbytes,
                           _stream(stream)))
    return dq, dk, dvv, da


def e_forward(q, k, v, a, *, scale=None, workspace=None, stream=None, out=None, lse=None):
    """2Mamba-E forward.  Returns (o, lse)."""
    B, H, T, d, dv, dt = _seq_checks(q, k, v, a)
    L = _load()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty(v.shape, dtype=torch.float32, device=q.device) if out is None else out
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device) if lse is None else lse
    ws = _workspace(L.tm2e_forward_workspace(B, H, T, d, dv, dt), q.device, workspace)
    nbytes = 0 if ws is None else ws.numel()
    _check(L.tm2e_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(o), _ptr(lse), B, H, T, d, dv,
                          scale, dt, _ptr(ws), nbytes, _stream(stream)))
    return o, lse


def e_backward(q, k, v, a, o, lse, dO, *, scale=None, workspace=None, stream=None, grads=None, lowp_grads=False):
    """2Mamba-E backward.  Returns (dq, dk, dv, da) (dq, dk, dv fp32, or the input dtype with lowp_grads)."""
    B, H, T, d, dv, dt = _seq_checks(q, k, v, a)
    L = _load()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    flags = GRADS_INPUT_DTYPE if lowp_grads else 0
    if grads is None:
        grads = _grad_buffers(q, k, v, a, lowp_grads)
    dq, dk, dvv, da = grads
    ws = _workspace(L.tm2e_backward_workspace(B, H, T, d, dv, dt), q.device, workspace)
    nbytes = 0 if ws is None else ws.numel()
    _check(L.tm2e_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(o), _ptr(lse), _ptr(dO),
                           _ptr(dq), _ptr(dk), _ptr(dvv), _ptr(da), B, H, T, d, dv, scale, dt, flags,
                           _ptr(ws), nbytes, _stream(stream)))
    return dq, dk, dvv, da


def poll_status() -> int:
    """Reads and clears the device status word (TM2_ERR_TIMEOUT after an expired wait)."""
    return int(_load().tm2_poll_status())
