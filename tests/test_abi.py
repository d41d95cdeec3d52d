"""C-ABI checks that need no GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

import ssm_sequence_mixer_chunked_b300 as tm2
from ssm_sequence_mixer_chunked_b300 import build as tm2_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tm2.h")

OK, INVALID, UNSUPPORTED, ALIGNMENT, WORKSPACE = 0, -1, -2, -3, -4
FAKE = 0x10000000  # a 256-byte aligned address that is never dereferenced (rejected first)


@pytest.fixture(scope="module")
def lib():
    tm2_build.build()
    return tm2.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tm2[eq]?_[a-z0-9_]+)\s*\(", src)))


def test_header_symbols_exported(lib):
    names = declared_functions()
    assert {"tm2_forward", "tm2_backward", "tm2_step", "tm2e_forward", "tm2e_backward", "tm2q_forward",
            "tm2q_backward"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_bounds_checked_build_exports_the_same_symbols():
    # the TM2_DEBUG variant (device index checks, a synchronisation and status read after
    # every launch) is a drop-in: same header, same exports
    path = tm2_build.build(debug=True)
    assert path.endswith("libtm2_debug.so") and os.path.exists(path)
    dbg = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(dbg, n), n
    dbg.tm2_status_string.restype = ctypes.c_char_p
    assert dbg.tm2_status_string(-7).decode().startswith("TM2_ERR_BOUNDS")


def test_version_and_status_strings(lib):
    assert lib.tm2_version() >= 100
    for st in (OK, INVALID, UNSUPPORTED, ALIGNMENT, WORKSPACE, -5, -6, -7, 12345):
        s = tm2.status_string(st)
        assert s.startswith("TM2")


def test_workspace_sizes(lib):
    bf16 = 1
    w = lib.tm2_forward_workspace(2, 16, 8192, 64, 64, 0, bf16, 1)
    # tensor-core path (chunk 256): the state entering each of 32 chunks, 4096 x 64 bf16
    # plus the 4096 fp32 normaliser entries, per (b, h, chunk)
    assert w >= 2 * 16 * 32 * 4096 * (64 * 2 + 4)
    w64 = lib.tm2_forward_workspace(2, 16, 8192, 64, 64, 64, bf16, 1)
    # CUDA-core path (chunk 64): 128 chunk states of 64 * 65 * 64 fp32 per (b, h)
    assert w64 >= 2 * 16 * 128 * 64 * 65 * 64 * 4
    assert lib.tm2_forward_workspace(2, 16, 8192, 64, 64, 256, bf16, 1) == w
    assert lib.tm2_forward_workspace(2, 16, 8192, 64, 64, 256, 0, 1) == 0     # fp32 has no chunk 256
    assert lib.tm2_backward_workspace(2, 16, 8192, 64, 64, 0, bf16, 1) > w
    assert lib.tm2_forward_workspace(2, 16, 8192, 48, 48, 0, bf16, 1) == 0      # unsupported -> 0
    assert lib.tm2_forward_workspace(2, 16, 0, 64, 64, 0, bf16, 1) % 256 == 0
    assert lib.tm2e_forward_workspace(2, 16, 4096, 64, 64, bf16) > 0


def test_reuse_states_flag(lib):
    """TM2_REUSE_STATES (2) is a backward-only flag; the forward rejects it before launching,
    and the backward workspace does not depend on it."""
    bf16 = 1
    assert lib.tm2_backward_workspace(2, 16, 8192, 64, 64, 0, bf16, 3) == \
        lib.tm2_backward_workspace(2, 16, 8192, 64, 64, 0, bf16, 1) > 0
    assert lib.tm2_forward_workspace(2, 16, 8192, 64, 64, 0, bf16, 3) == 0
    assert fwd(lib, flags=3) == INVALID
    assert lib.tm2_backward_workspace(2, 16, 8192, 64, 64, 0, bf16, 4) == 0   # unknown flag


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, a=FAKE, o=FAKE, Z=FAKE, B=1, H=2, T=256, d=16, dv=16,
        chunk=64, dtype=0, flags=1, ws=FAKE, ws_bytes=1 << 40):
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.tm2_forward(P(q), P(k), P(v), P(a), None, None, P(o), P(Z), None, None, B, H, T, d,
                           dv, chunk, dtype, flags, P(ws), ws_bytes, None)


def test_forward_rejects_bad_arguments(lib):
    assert fwd(lib, B=-1) == INVALID
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, flags=8) == INVALID
    assert fwd(lib, d=48, dv=48) == UNSUPPORTED
    assert fwd(lib, d=64, dv=32) == UNSUPPORTED
    assert fwd(lib, chunk=48) == UNSUPPORTED
    assert fwd(lib, dtype=7) == UNSUPPORTED
    assert fwd(lib, k=FAKE + 4) == ALIGNMENT
    assert fwd(lib, ws=None) == WORKSPACE
    assert fwd(lib, ws_bytes=16) == WORKSPACE
    assert fwd(lib, ws=FAKE + 16) == ALIGNMENT


def test_step_and_e_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    f = P(FAKE)
    assert lib.tm2_step(f, f, f, f, f, None, f, None, 4, 2, 64, 64, 0, 1, None) == INVALID  # normalise needs z
    assert lib.tm2_step(f, f, f, f, f, f, f, f, 4, 2, 40, 40, 0, 1, None) == UNSUPPORTED
    assert lib.tm2_step(f, f, f, P(FAKE + 8), f, f, f, f, 4, 2, 64, 64, 0, 1, None) == ALIGNMENT
    assert lib.tm2e_forward(f, f, f, f, f, f, 1, 1, 128, 64, 64, ctypes.c_float(0.0), 1, f, 1 << 30,
                            None) == INVALID
    assert lib.tm2e_forward(f, f, f, f, f, None, 1, 1, 128, 64, 64, ctypes.c_float(0.125), 1, f,
                            1 << 30, None) == INVALID
    assert lib.tm2e_backward(f, f, f, f, f, f, f, f, f, f, f, 1, 1, 128, 64, 64, ctypes.c_float(0.125),
                             1, 0, f, 8, None) == WORKSPACE
    assert lib.tm2e_backward(f, f, f, f, f, f, f, f, f, f, f, 1, 1, 128, 64, 64, ctypes.c_float(0.125),
                             1, 1, f, 1 << 30, None) == INVALID     # no normalisation flag for 2Mamba-E


def test_backward_needs_Z_when_normalised(lib):
    P = ctypes.c_void_p
    f = P(FAKE)
    st = lib.tm2_backward(f, f, f, f, f, None, f, f, f, f, f, 1, 1, 128, 64, 64, 0, 1, 1, f, 1 << 40, None)
    assert st == INVALID


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    x = torch.zeros(1, 1, 4, 16)
    with pytest.raises(tm2.TM2Error):
        tm2.forward(x, x, x, torch.zeros(1, 1, 4))


def test_quadratic_form_rejects_bad_arguments(lib):
    f = ctypes.c_void_p(FAKE)
    args = lambda order, d, flags: (f, f, f, f, f, f, 1, 2, 64, d, d, order, 1, flags, f, 1 << 30, None)
    assert lib.tm2q_forward(*args(3, 64, 1)) == UNSUPPORTED          # order 1 or 2 only
    assert lib.tm2q_forward(*args(2, 48, 1)) == UNSUPPORTED          # head dim
    assert lib.tm2q_forward(*args(2, 64, 4)) == INVALID              # unknown flag
    assert lib.tm2q_forward_workspace(1, 2, 64, 64, 64, 0, 1, 1) == 0
    assert lib.tm2q_forward_workspace(1, 2, 64, 64, 64, 1, 1, 1) > 0
    assert lib.tm2q_backward_workspace(1, 2, 64, 64, 64, 2, 1, 1) > lib.tm2q_forward_workspace(1, 2, 64, 64, 64, 2, 1, 1) - 1
    g = (f, f, f, f, None, None, f, f, f, f, f, 1, 2, 64, 64, 64, 2, 1, 1, f, 1 << 30, None)
    assert lib.tm2q_backward(*g) == INVALID                          # normalised needs o and Z
