"""CUDA-graph capture of the tensor-core forward and backward (bf16, d = dv = 64).

The library forks its state walks onto side streams of its own and joins them back with
events; captured into a CUDA graph, those become graph edges, so replaying the captured step
must give the eager call's results.  A capture made in a host thread that has not called the
library before (its fork / join events do not exist yet, and making them is not capturable)
runs on the caller's stream alone and must give the same results too.
"""
import threading

import pytest
import torch

import ssm_sequence_mixer_chunked_b300 as tm2
import synth_inputs as si

pytestmark = pytest.mark.gpu


def _inputs():
    inp = si.sequence_inputs(1, 4, 1024, 64, 64, dtype="bf16", qkv_std=0.125, seed=11, with_dO=True)
    return {k: v.cuda() for k, v in inp.items()}


def _buffers(g):
    B, H, T, d = g["q"].shape
    dv = g["v"].shape[-1]
    o = torch.empty(g["v"].shape, dtype=torch.float32, device="cuda")
    Z = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    grads = tuple(torch.empty(g[n].shape, dtype=torch.float32, device="cuda") for n in ("q", "k", "v", "a"))
    ws = torch.empty(tm2.workspace_bytes(B, H, T, d, dv), dtype=torch.uint8, device="cuda")
    return ws, (o, Z) + grads


def _step(g, ws, outs):
    o, Z, dq, dk, dv, da = outs
    tm2.forward(g["q"], g["k"], g["v"], g["a"], out=o, Z=Z, workspace=ws)
    tm2.backward(g["q"], g["k"], g["v"], g["a"], o, Z, g["dO"], workspace=ws, grads=(dq, dk, dv, da),
                 reuse_states=True)


def _eager(g):
    ws, outs = _buffers(g)
    _step(g, ws, outs)
    torch.cuda.synchronize()
    return [x.clone() for x in outs]


def _captured(g):
    ws, outs = _buffers(g)
    for x in outs:
        x.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(g, ws, outs)
    graph.replay()
    torch.cuda.synchronize()
    return [x.clone() for x in outs]


def _compare(got, ref):
    names = ("o", "Z", "dq", "dk", "dv", "da")
    for name, a, b in zip(names, got, ref):
        rms = b.double().pow(2).mean().sqrt().item()
        diff = (a.double() - b.double()).abs().max().item()
        # the backward's shared-memory sums are unordered, so replays agree to fp32 rounding
        assert diff <= 1e-4 * rms + 1e-30, (name, diff, rms)


def test_graph_replay_matches_eager():
    g = _inputs()
    ref = _eager(g)          # this thread's side-stream events now exist: the capture forks
    _compare(_captured(g), ref)


def test_graph_capture_in_a_fresh_thread_runs_on_one_stream():
    g = _inputs()
    ref = _eager(g)
    result = {}

    def body():
        try:
            torch.cuda.set_device(0)
            result["got"] = _captured(g)
        except Exception as e:   # reported below, in the test's own thread
            result["err"] = e

    t = threading.Thread(target=body)
    t.start()
    t.join()
    assert "err" not in result, result.get("err")
    _compare(result["got"], ref)
