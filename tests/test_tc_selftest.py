"""Checks of the tensor-core building blocks on the GPU: TMA 128B-swizzled tiles,
tcgen05.mma (bf16 x bf16 -> fp32 in tensor memory) and tcgen05.ld, against torch's
matmul; and the bounded-wait failure path, which must record TM2_ERR_TIMEOUT in the
status word and leave the context usable (no trap, no hang)."""
import ctypes

import pytest
import torch

import ssm_sequence_mixer_chunked_b300 as tm2

pytestmark = pytest.mark.gpu


MN_MAJOR_B = (4, 5)   # modes whose B operand is given as B^T (K x N, row-major)


def selftest(A, B, N, K, mode, wait_ns=0):
    lib = tm2.lib()
    fn = lib.tm2_selftest_umma
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_ulonglong, ctypes.c_void_p]
    D = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    st = fn(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, mode, wait_ns,
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st, D


@pytest.mark.parametrize("mode", [0, 1, 3, 4, 5])
@pytest.mark.parametrize("N,K", [(16, 64), (64, 64), (64, 256), (80, 128), (128, 192), (256, 128)])
def test_umma_matches_matmul(mode, N, K):
    """Modes: 0 A and B by TMA; 1 A written by the threads into shared memory; 3 A in
    tensor memory; 4 B MN-major (B^T row-major in memory); 5 A in tensor memory and B
    MN-major."""
    g = torch.Generator(device="cpu").manual_seed(N * 1000 + K + mode)
    A = torch.randn(128, K, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    Bin = B.T.contiguous() if mode in MN_MAJOR_B else B
    st, D = selftest(A, Bin, N, K, mode)
    assert st == 0, tm2.status_string(st)
    ref = A.double() @ B.double().T
    err = (D.double() - ref).abs().max().item() / ref.pow(2).mean().sqrt().item()
    assert err < 1e-5, err


def test_bounded_wait_records_timeout_and_context_survives():
    A = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    assert tm2.poll_status() == 0
    st, D = selftest(A, B, 16, 64, 2, wait_ns=1_000_000)
    assert st == 0
    assert tm2.poll_status() == -6          # TM2_ERR_TIMEOUT, then cleared
    assert tm2.poll_status() == 0
    assert torch.isnan(D).all()             # nothing was written
    st, D = selftest(torch.ones(128, 64, dtype=torch.bfloat16, device="cuda"),
                     torch.ones(16, 64, dtype=torch.bfloat16, device="cuda"), 16, 64, 0)
    assert st == 0 and torch.all(D == 64.0)  # the context still computes
