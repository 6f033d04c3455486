"""The two-stream schedule of Algorithm 1 (Oases §IV, Fig. 4b and 4d) as it runs
on the GPU, from the per-operator event trace of the block scheduler
(oases_debug_trace_read), at the full 4-layer stack (hidden 2560, ffn 10240,
20 heads, seq 2048, batch 8, w = 4, 2 sub-batches, fine-grained recompute).

Sub-batch b runs on stream b, in Algorithm 1's order, and the streams meet only
where weight gradients are accumulated in sub-batch order.  What the pages'
schedule promises then shows in the trace:
* warm-up: sub-batch 0's backward (the recompute of the last segment) starts
  while sub-batch 1 is still in its forward;
* across segments ("our backward schedule can run across layers"): at every
  segment boundary, sub-batch 0 starts recomputing segment s-1 before
  sub-batch 1 has finished the backward of segment s (its LayerNorm
  backward, which ends segment s);
* cool-down: sub-batch 1 ends the step, after sub-batch 0.
The fraction of the step during which both streams have an operator in flight
is reported (and must be positive).  Stream intervals come from CUDA events on
each sub-batch's stream: an operator's interval is from the moment its stream
reached it to the moment its last kernel finished.
"""
import ctypes
import json

import numpy as np
import pytest
import torch

from synth import SHAPES, block_inputs
from tensor_model_transformer_tp_gb300 import EVENTS, OPS, lib, oases_check_device
from tensor_model_transformer_tp_gb300.device import DeviceBlock

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_model_transformer_tp_gb300 import build_library
    build_library()
    L = lib()
    L.oases_debug_trace_enable.argtypes = [ctypes.c_int]
    L.oases_debug_trace_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.c_int]
    L.oases_debug_trace_read.restype = ctypes.c_int
    return L


def union_length(iv):
    tot, end = 0.0, -np.inf
    for a, b in sorted(iv):
        if b <= end:
            continue
        tot += b - max(a, end)
        end = b
    return tot


def intersect_length(a_iv, b_iv):
    """Length of (union of a) intersected with (union of b)."""
    return union_length(a_iv) + union_length(b_iv) - union_length(a_iv + b_iv)


def traced_step(L, shape):
    inp = block_inputs(shape, seed=0)
    blk = DeviceBlock(shape, inp["layers"])
    x, g = blk.tensor(inp["x"]), blk.tensor(inp["g"])
    blk.step(x, g)                       # warm-up, untraced
    torch.cuda.synchronize()
    L.oases_debug_trace_enable(1)
    try:
        blk.step(x, g)
        torch.cuda.synchronize()
        n = L.oases_debug_trace_read(None, 0)
        buf = (ctypes.c_double * (6 * n))()
        assert L.oases_debug_trace_read(buf, n) == n
    finally:
        L.oases_debug_trace_enable(0)
    oases_check_device(None)
    rec = np.frombuffer(buf, dtype=np.float64).reshape(n, 6)
    return [{"ev": EVENTS[int(r[0])], "op": OPS[int(r[1])], "seg": int(r[2]), "sb": int(r[3]),
             "t0": r[4], "t1": r[5]} for r in rec]


def test_stack_h2560_two_stream_overlap(L):
    shape = SHAPES["stack4_bf16_h2560"]
    steps = traced_step(L, shape)
    nseg = 2 * shape.n_layers
    work = [s for s in steps if s["ev"] != "Sync"]
    by_sb = {b: [s for s in work if s["sb"] == b] for b in (0, 1)}
    iv = {b: [(s["t0"], s["t1"]) for s in by_sb[b]] for b in (0, 1)}
    span = max(s["t1"] for s in work) - min(s["t0"] for s in work)

    # warm-up: sub-batch 0's first backward operator starts before sub-batch 1's forward ends
    fwd_end_1 = max(s["t1"] for s in by_sb[1] if s["ev"] in ("F", "C(F)"))
    bwd_start_0 = min(s["t0"] for s in by_sb[0] if s["ev"] not in ("F", "C(F)"))
    warm = fwd_end_1 - bwd_start_0
    assert warm > 0, (bwd_start_0, fwd_end_1)

    # across segments: sub-batch 0 recomputes segment s-1 before sub-batch 1
    # ends segment s (its LayerNorm backward)
    cross = {}
    for s in range(nseg - 1, 0, -1):
        r0 = min(t["t0"] for t in by_sb[0] if t["ev"] == "R" and t["seg"] == s - 1)
        e1 = max(t["t1"] for t in by_sb[1] if t["ev"] == "B" and t["op"] == "ln" and t["seg"] == s)
        cross[s] = e1 - r0
        assert e1 > r0, (s, r0, e1)

    # cool-down: sub-batch 1 ends the step
    end0, end1 = max(t["t1"] for t in by_sb[0]), max(t["t1"] for t in by_sb[1])
    assert end1 >= end0

    both = intersect_length(iv[0], iv[1])
    frac = both / span
    assert frac > 0
    print(json.dumps({"workload": "stack4_bf16_h2560", "step_us": span,
                      "both_streams_busy_us": both, "overlap_fraction": frac,
                      "warm_up_overlap_us": warm,
                      "cross_segment_overlap_us": {str(k): v for k, v in cross.items()},
                      "cool_down_us": end1 - end0}))
