"""The C-ABI library on the CPU: it builds, loads, exports every declared symbol,
validates arguments, injects failures on the host and schedules the operators
in the order of the oracle's Algorithm 1 executor.  No kernel is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import tensor_model_transformer_tp_gb300 as oz
from synth import BlockShape, block_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    oz.build_library()
    return oz.lib()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            src = re.sub(r"#define[^\n]*", "", src)
            names |= set(re.findall(r"\b(oases_[a-z_0-9]+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert "oases_block_fwd" in names and "oases_stack_step" in names
    for n in names:
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert "sm_103a" in oz.oases_version()
    for st in range(7):
        assert oz.oases_status_str(st)


def _desc(**kw):
    base = dict(kind="ffn", dtype="bf16", batch=2, seq=8, hidden=64, ffn=128, heads=0, w=2,
                sub_batches=2)
    base.update(kw)
    return oz.make_desc(**base)


def test_workspace_bytes(L):
    fine = oz.oases_workspace_bytes(_desc(recompute="fine"))
    assert fine > 0
    # two layers: NONE keeps every segment's activations, FINE one set per kind
    assert oz.oases_workspace_bytes(_desc(recompute="none"), 2) > oz.oases_workspace_bytes(
        _desc(recompute="fine"), 2)
    assert oz.oases_workspace_bytes(_desc(recompute="fine"), 3) > fine
    assert oz.oases_workspace_bytes(_desc(batch=3)) == 0          # batch % sub_batches
    assert oz.oases_workspace_bytes(_desc(ffn=130, w=4)) == 0     # ffn % w


FAKE = 1 << 20  # non-NULL pointer values; nothing is dereferenced before validation fails


def _weights():
    return oz.Weights(*([FAKE] * 12))


def _grads():
    return oz.Grads(*([FAKE] * 12))


def _fwd_status(desc, ws=FAKE, nb=1 << 40):
    return oz.lib().oases_block_fwd(ctypes.byref(desc), ctypes.byref(_weights()), FAKE, FAKE,
                                    ws, nb, None, None)


@pytest.mark.parametrize("bad,status", [
    (dict(batch=-1), 1), (dict(hidden=0), 1), (dict(w=0), 1), (dict(sub_batches=0), 1),
    (dict(batch=3), 1), (dict(ffn=100, w=3), 1), (dict(kind="attn", heads=3), 1),
    (dict(kind="attn", heads=2, hidden=272), 2),          # head dim 136 > 128
    (dict(hidden=60), 2),                                  # bf16 rows not 16-byte multiples
])
def test_invalid_descriptors_rejected(L, bad, status):
    assert _fwd_status(_desc(**bad)) == status


@pytest.mark.parametrize("field,value", [("recompute", 4), ("recompute", -1), ("reduce", 2),
                                         ("reduce", -1), ("kind", 3), ("dtype", 3),
                                         ("dtype", -1)])
def test_out_of_range_codes_rejected(L, field, value):
    d = _desc()
    setattr(d, field, value)
    assert _fwd_status(d) == 1
    assert oz.oases_workspace_bytes(d) == 0


def test_misaligned_device_pointers_rejected(L):
    d = _desc()
    w = _weights()
    w.b1 = FAKE + 8          # 16-byte rule: refused before anything is enqueued
    assert L.oases_block_fwd(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE, FAKE, 1 << 40,
                             None, None) == 1
    assert L.oases_block_fwd(ctypes.byref(d), ctypes.byref(_weights()), FAKE + 4, FAKE, FAKE,
                             1 << 40, None, None) == 1
    g = _grads()
    g.w2 = FAKE + 2
    assert L.oases_block_recompute_bwd(ctypes.byref(d), ctypes.byref(_weights()), FAKE, FAKE, FAKE,
                                       ctypes.byref(g), FAKE, 1 << 40, None, None) == 1


def test_null_and_small_workspace(L):
    d = _desc()
    assert _fwd_status(d, ws=None) == 3
    assert _fwd_status(d, nb=16) == 3
    assert L.oases_block_fwd(ctypes.byref(d), None, FAKE, FAKE, FAKE, 1 << 40, None, None) == 1
    w = _weights()
    w.w1 = None
    assert L.oases_block_fwd(ctypes.byref(d), ctypes.byref(w), FAKE, FAKE, FAKE, 1 << 40,
                             None, None) == 1


def test_host_side_failure_injection(L, monkeypatch):
    d = _desc()
    # C(B) of segment 0, sub-batch 1: a backward operator
    monkeypatch.setenv("OASES_TEST_FAIL_AT", "5:1:0:1")
    st = L.oases_block_recompute_bwd(ctypes.byref(d), ctypes.byref(_weights()), FAKE, FAKE, FAKE,
                                     ctypes.byref(_grads()), FAKE, 1 << 40, None, None)
    assert st == 6
    assert _fwd_status(d) != 6          # the forward has no such operator
    monkeypatch.setenv("OASES_TEST_FAIL_AT", "0:2:0:0")   # F(col) of segment 0
    assert _fwd_status(d) == 6


def _oracle_trace(shape, mode, n_sb):
    inp = block_inputs(shape, seed=0)
    return [tuple(e) for e in oracle.run_step(shape, inp, mode=mode, sub_batches=n_sb)["trace"]]


@pytest.mark.parametrize("kind,n_layers", [("ffn", 1), ("attn", 1), ("layer", 1), ("layer", 2),
                                           ("ffn", 3)])
@pytest.mark.parametrize("mode", ["none", "full", "fine", "selective"])
@pytest.mark.parametrize("n_sb", [1, 2, 4])
def test_schedule_matches_oracle_algorithm1(L, kind, n_layers, mode, n_sb):
    """The library enqueues operators in exactly the oracle's Algorithm 1 order."""
    shape = BlockShape(kind, "f32", batch=4, seq=4, hidden=16, ffn=16, heads=2, w=2,
                       sub_batches=n_sb, n_layers=n_layers)
    desc = oz.desc_from_shape(shape, mode)
    got = oz.oases_schedule_trace(desc, n_layers, 0) + oz.oases_schedule_trace(desc, n_layers, 1)
    assert got == _oracle_trace(shape, mode, n_sb)


def test_schedule_counts_per_mode(L):
    d = {m: _desc(recompute=m) for m in ("none", "full", "fine")}
    for m, cr in (("none", 0), ("full", 2), ("fine", 0)):
        t = oz.oases_schedule_trace(d[m], 1, 1)
        assert sum(e[0] == "C(R)" for e in t) == cr
        assert sum(e[0] == "C(B)" for e in t) == 2
        assert sum(e[0] == "R" for e in t) == {"none": 0, "full": 6, "fine": 4}[m]


def test_selective_workspace_between_fine_and_none(L):
    """SELECTIVE keeps what NONE keeps except each attention segment's output O
    and its LSE, which all attention segments share."""
    d = {m: _desc(kind="layer", heads=2, recompute=m) for m in ("none", "fine", "selective")}
    n = {m: oz.oases_workspace_bytes(d[m], 2) for m in d}
    assert n["fine"] < n["selective"] < n["none"]
    f = {m: oz.oases_workspace_bytes(_desc(recompute=m), 2) for m in ("none", "selective")}
    assert f["none"] == f["selective"]          # FFN only: nothing to recompute


def test_mxfp8_descriptors(L):
    """MX-FP8 blocks store bf16 and add per-stream scratch for the quantised
    operands; shapes whose 32-blocks would straddle a shard's slice, and the
    separate reduction, are refused."""
    bf = oz.oases_workspace_bytes(_desc(dtype="bf16"))
    mx = oz.oases_workspace_bytes(_desc(dtype="mxfp8"))
    assert mx > bf > 0
    assert oz.oases_workspace_bytes(_desc(dtype="mxfp8", ffn=192)) > 0       # ffn / w = 96
    assert oz.oases_workspace_bytes(_desc(dtype="mxfp8", ffn=96)) == 0       # ffn / w = 48
    assert oz.oases_workspace_bytes(_desc(dtype="mxfp8", hidden=48)) == 0    # hidden % 32
    assert oz.oases_workspace_bytes(_desc(dtype="mxfp8", reduce="separate")) == 0
    assert _fwd_status(_desc(dtype="mxfp8", ffn=96)) == 2
