"""Run-to-run bitwise determinism of the GPU path: the same inputs give the same bits.

Nothing in the kernels depends on scheduling order: the forward has no atomics; the backward's
only shared-memory sums add exactly two terms into a zeroed word (a + b = b + a in floating
point) before a barrier orders the next term, and the per-head maxima are integer atomicMax.
The tensor-core 2Mamba forward + backward (with the walks on the library's side streams), the
2Mamba-E forward + backward and the quadratic form are each run twice and compared bit for bit.
"""
import math

import pytest
import torch

import ssm_sequence_mixer_chunked_b300 as tm2
import synth_inputs as si

pytestmark = pytest.mark.gpu


def _same(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x, y), (x - y).abs().max().item()


def _cuda(inp):
    return {k: v.cuda() for k, v in inp.items()}


def test_chunked_fwd_bwd_bitwise():
    g = _cuda(si.sequence_inputs(2, 4, 1000, 64, 64, dtype="bf16", qkv_std=1 / math.sqrt(64), seed=31,
                                 with_dO=True))

    def run():
        o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"])
        grads = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"])
        torch.cuda.synchronize()
        return (o, Z) + tuple(grads)

    _same(run(), run())


def test_softmax_form_fwd_bwd_bitwise():
    g = _cuda(si.sequence_inputs(1, 4, 777, 64, 64, dtype="bf16", qkv_std=1.0, seed=32, with_dO=True))

    def run():
        o, lse = tm2.e_forward(g["q"], g["k"], g["v"], g["a"])
        grads = tm2.e_backward(g["q"], g["k"], g["v"], g["a"], o, lse, g["dO"])
        oq, Zq = tm2.forward_quadratic(g["q"], g["k"], g["v"], g["a"])
        gq = tm2.backward_quadratic(g["q"], g["k"], g["v"], g["a"], oq, Zq, g["dO"])
        torch.cuda.synchronize()
        return (o, lse, oq, Zq) + tuple(grads) + tuple(gq)

    _same(run(), run())
