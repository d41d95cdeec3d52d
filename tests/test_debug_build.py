"""The bounds-checked build (libtm2_debug.so, -DTM2_DEBUG) on the GPU: a child process loads it
(TM2_DEBUG=1) and runs the tensor-core forward + backward of 2Mamba, the 2Mamba-E forward +
backward and a ragged sequence through the C ABI.  Every launch is followed by a
synchronisation and a status read, so an index check that failed would surface as
TM2_ERR_BOUNDS from the call; the results are checked against the fp64 oracle at the bf16 bar.
"""
import os
import subprocess
import sys

import pytest

from ssm_sequence_mixer_chunked_b300 import build as tm2_build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import math, sys
sys.path.insert(0, sys.argv[1])
import torch
import oracle
import ssm_sequence_mixer_chunked_b300 as tm2
import synth_inputs as si
assert tm2.library_path().endswith("libtm2_debug.so"), tm2.library_path()
dev = torch.device("cuda", 0)
worst = 0.0
for T in (512, 333):   # whole chunks, and a ragged tail
    inp = si.sequence_inputs(1, 2, T, 64, 64, dtype="bf16", qkv_std=1 / math.sqrt(64), seed=T, with_dO=True)
    g = {k: v.to(dev) for k, v in inp.items()}
    o, Z = tm2.forward(g["q"], g["k"], g["v"], g["a"])
    grads = tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"])
    torch.cuda.synchronize()
    assert tm2.lib().tm2_poll_status() == 0
    o_ref, _ = oracle.fwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], True)
    refs = oracle.bwd_quadratic(inp["q"], inp["k"], inp["v"], inp["a"], inp["dO"], True)
    worst = max(worst, si.rel_err(o.cpu(), o_ref), *(si.rel_err(x.cpu(), r) for x, r in zip(grads, refs)))
ie = si.sequence_inputs(1, 2, 300, 64, 64, dtype="bf16", qkv_std=1.0, seed=4, with_dO=True)
ge = {k: v.to(dev) for k, v in ie.items()}
oe, lse = tm2.e_forward(ge["q"], ge["k"], ge["v"], ge["a"])
eg = tm2.e_backward(ge["q"], ge["k"], ge["v"], ge["a"], oe, lse, ge["dO"])
torch.cuda.synchronize()
assert tm2.lib().tm2_poll_status() == 0
oe_ref, _ = oracle.e_fwd(ie["q"], ie["k"], ie["v"], ie["a"])
erefs = oracle.e_bwd(ie["q"], ie["k"], ie["v"], ie["a"], ie["dO"])
worst = max(worst, si.rel_err(oe.cpu(), oe_ref), *(si.rel_err(x.cpu(), r) for x, r in zip(eg, erefs)))
print("worst", worst)
assert worst <= 2e-2, worst
"""


def test_bounds_checked_build_runs_clean():
    tm2_build.build(debug=True)
    env = dict(os.environ, TM2_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
