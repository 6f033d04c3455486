"""CUDA path against the CPU oracle, through the C ABI (oases_stack_step,
oases_block_fwd / oases_block_recompute_bwd), on the same seeded inputs.

Tolerance: per output tensor (y, dx and every weight gradient) the relative L2
error ||gpu - oracle|| / ||oracle|| is at most 1e-5 for fp32 workloads and
2e-2 for bf16 workloads (activations stored in bf16, fp32 accumulation).
The causal mask is structural in both implementations.  Properties that must
hold bit for bit on the GPU (recompute modes, sub-batch split, determinism) are
checked with exact equality.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import SHAPES, BlockShape, block_inputs
from tensor_model_transformer_tp_gb300 import OasesError, oases_check_device, oases_last_launch_count
from tensor_model_transformer_tp_gb300.device import DeviceBlock, to_numpy

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_model_transformer_tp_gb300 import build_library
    build_library()


def rel(a, b):
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))


def run_gpu(shape, inp, mode="fine", sub_batches=None, api="stack", reduce="fused"):
    blk = DeviceBlock(shape, inp["layers"], recompute=mode, sub_batches=sub_batches, reduce=reduce)
    x, g = blk.tensor(inp["x"]), blk.tensor(inp["g"])
    if api == "stack":
        y, dx = blk.step(x, g)
    else:
        y = blk.fwd(x)
        dx = blk.recompute_bwd(x, g)
    torch.cuda.synchronize()
    oases_check_device(None)
    return {"y": to_numpy(y), "dx": to_numpy(dx), "grads": blk.grads_numpy(),
            "launches": oases_last_launch_count()}


def compare(shape, got, ref, tol=None):
    tol = TOL[shape.dtype] if tol is None else tol
    errs = {"y": rel(got["y"], ref["y"]), "dx": rel(got["dx"], ref["dx"])}
    for li, (gl, rl) in enumerate(zip(got["grads"], ref["grads"])):
        for k in rl:
            errs["L%d.%s" % (li, k)] = rel(gl[k], rl[k])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, bad
    return errs


def assert_identical(a, b):
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["dx"], b["dx"])
    for ga, gb in zip(a["grads"], b["grads"]):
        for k in ga:
            np.testing.assert_array_equal(ga[k], gb[k])


# ------------------------------------------------------------------ fp32 workload
@pytest.mark.parametrize("mode", ["fine", "full", "none"])
def test_ffn_f32_h256_full_size(mode):
    """FFN block fp32, hidden 256, ffn 1024, seq 128, batch 2, w=2, 2 sub-batches."""
    shape = SHAPES["ffn_f32_h256"]
    inp = block_inputs(shape, seed=0)
    compare(shape, run_gpu(shape, inp, mode), oracle.run_step(shape, inp, mode=mode))


def test_f32_layer_with_ragged_rows_and_affine():
    shape = BlockShape("layer", "f32", batch=2, seq=37, hidden=128, ffn=192, heads=4, w=2)
    inp = block_inputs(shape, seed=1, affine=True)
    compare(shape, run_gpu(shape, inp), oracle.run_step(shape, inp, mode="fine"))


# ------------------------------------------------------------------ bf16 FFN
def test_ffn_bf16_reduced_ragged():
    shape = BlockShape("ffn", "bf16", batch=4, seq=100, hidden=256, ffn=1024, w=4)
    inp = block_inputs(shape, seed=2, affine=True)
    compare(shape, run_gpu(shape, inp), oracle.run_step(shape, inp, mode="fine"))


def test_ffn_bf16_h1024_full_size():
    """FFN bf16 hidden 1024, ffn 4096, seq 512, batch 8, w=4, 2 sub-batches, pre-LN."""
    shape = SHAPES["ffn_bf16_h1024"]
    inp = block_inputs(shape, seed=0)
    got = run_gpu(shape, inp, "fine")
    compare(shape, got, oracle.run_step(shape, inp, mode="fine"))
    assert got["launches"] > 0


def test_ffn_bf16_modes_bit_identical():
    shape = BlockShape("ffn", "bf16", batch=4, seq=96, hidden=256, ffn=512, w=2)
    inp = block_inputs(shape, seed=3, affine=True)
    r = {m: run_gpu(shape, inp, m) for m in ("none", "full", "fine", "selective")}
    assert_identical(r["fine"], r["none"])
    assert_identical(r["full"], r["none"])
    assert_identical(r["selective"], r["none"])


def test_ffn_bf16_sub_batch_split():
    """The split changes the schedule, not the math: y and dx bit-identical,
    weight gradients equal up to fp32 summation order."""
    shape = BlockShape("ffn", "bf16", batch=4, seq=64, hidden=256, ffn=512, w=4)
    inp = block_inputs(shape, seed=4, affine=True)
    r1 = run_gpu(shape, inp, sub_batches=1)
    r2 = run_gpu(shape, inp, sub_batches=2)
    r4 = run_gpu(shape, inp, sub_batches=4)
    for r in (r2, r4):
        np.testing.assert_array_equal(r["y"], r1["y"])
        np.testing.assert_array_equal(r["dx"], r1["dx"])
        for k in r1["grads"][0]:
            assert rel(r["grads"][0][k], r1["grads"][0][k]) <= 1e-5, k


def test_deterministic():
    shape = BlockShape("layer", "bf16", batch=2, seq=64, hidden=256, ffn=512, heads=2, w=2)
    inp = block_inputs(shape, seed=5, affine=True)
    assert_identical(run_gpu(shape, inp), run_gpu(shape, inp))


def test_concurrent_calls_from_two_host_threads():
    """Two host threads, each with its own block, workspace and streams, step
    at the same time; each gets the bits it gets when run alone."""
    import threading
    shape = BlockShape("layer", "bf16", batch=2, seq=64, hidden=256, ffn=512, heads=2, w=2)
    inps = [block_inputs(shape, seed=s, affine=True) for s in (21, 22)]
    alone = [run_gpu(shape, inp) for inp in inps]
    blks = [DeviceBlock(shape, inp["layers"]) for inp in inps]
    io = [(b.tensor(i["x"]), b.tensor(i["g"])) for b, i in zip(blks, inps)]
    torch.cuda.synchronize()
    outs, errs = [None, None], []
    start = threading.Barrier(2)

    def work(k):
        try:
            start.wait(timeout=60)
            for _ in range(4):
                blks[k].zero_grads()
                y, dx = blks[k].step(*io[k])
            torch.cuda.synchronize()
            outs[k] = {"y": to_numpy(y), "dx": to_numpy(dx), "grads": blks[k].grads_numpy()}
        except Exception as e:  # reported below, on the test's thread
            errs.append(e)

    threads = [threading.Thread(target=work, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errs, errs
    oases_check_device(None)
    for k in range(2):
        assert_identical(outs[k], alone[k])


def test_block_api_equals_stack_step():
    shape = BlockShape("layer", "bf16", batch=2, seq=64, hidden=256, ffn=512, heads=2, w=2)
    inp = block_inputs(shape, seed=6, affine=True)
    assert_identical(run_gpu(shape, inp, api="block"), run_gpu(shape, inp, api="stack"))


# ------------------------------------------------------------------ attention / layer
def test_attn_bf16_reduced_ragged():
    shape = BlockShape("attn", "bf16", batch=2, seq=160, hidden=256, heads=2, w=2)
    inp = block_inputs(shape, seed=7, affine=True)
    compare(shape, run_gpu(shape, inp), oracle.run_step(shape, inp, mode="fine"))


def test_attn_bf16_noncausal_no_ln():
    shape = BlockShape("attn", "bf16", batch=2, seq=72, hidden=256, heads=4, w=4, causal=False,
                       pre_ln=False, residual=False)
    inp = block_inputs(shape, seed=8, affine=True)
    compare(shape, run_gpu(shape, inp), oracle.run_step(shape, inp, mode="fine"))


def test_layer_stack_bf16_reduced():
    shape = BlockShape("layer", "bf16", batch=2, seq=96, hidden=256, ffn=768, heads=2, w=2,
                       n_layers=2)
    inp = block_inputs(shape, seed=9, affine=True)
    compare(shape, run_gpu(shape, inp), oracle.run_step(shape, inp, mode="fine"))


# ------------------------------------------------------------------ edge cases
def test_empty_batch():
    shape = BlockShape("layer", "bf16", batch=0, seq=16, hidden=256, ffn=512, heads=2, w=2)
    inp = block_inputs(shape, seed=10)
    got = run_gpu(shape, inp)
    assert got["y"].shape == (0, 256)
    for g in got["grads"][0].values():
        assert np.all(g == 0)


def test_single_token_sequences():
    shape = BlockShape("layer", "bf16", batch=4, seq=1, hidden=128, ffn=256, heads=1, w=1)
    inp = block_inputs(shape, seed=11, affine=True)
    compare(shape, run_gpu(shape, inp), oracle.run_step(shape, inp, mode="fine"))


def test_invalid_shape_raises_before_launch():
    shape = BlockShape("attn", "bf16", batch=2, seq=8, hidden=272, heads=2, w=1)  # head dim 136
    with pytest.raises((OasesError, ValueError)):
        DeviceBlock(shape, block_inputs(shape, seed=0)["layers"])


@pytest.mark.parametrize("shape", [
    BlockShape("ffn", "bf16", batch=2, seq=64, hidden=256, ffn=512, w=2),
    # four sub-batches on two streams: x and dx staged one sub-batch's rows at a time
    BlockShape("layer", "bf16", batch=4, seq=128, hidden=256, ffn=512, heads=2, w=2, sub_batches=4,
               n_layers=2),
])
def test_host_buffers_through_stack_step(shape):
    """x, g, y, dx in pinned host memory: staged through the workspace, bit
    for bit the device-buffer results."""
    inp = block_inputs(shape, seed=12, affine=True)
    dev = run_gpu(shape, inp)
    blk = DeviceBlock(shape, inp["layers"])
    xh = blk.tensor(inp["x"]).cpu().pin_memory()
    gh = blk.tensor(inp["g"]).cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    dxh = torch.empty_like(xh).pin_memory()
    blk.step(xh, gh, yh, dxh)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(yh.double().numpy(), dev["y"])
    np.testing.assert_array_equal(dxh.double().numpy(), dev["dx"])


def test_shutdown_releases_state_and_next_calls_remake_it():
    """oases_shutdown() drops the copy stream, this thread's events and the
    host caches; the next calls (device and host buffers, traced) remake
    them and give the same bits as before."""
    from tensor_model_transformer_tp_gb300 import lib, oases_shutdown
    import ctypes
    shape = BlockShape("layer", "bf16", batch=2, seq=64, hidden=256, ffn=512, heads=2, w=2)
    inp = block_inputs(shape, seed=13, affine=True)
    before = run_gpu(shape, inp)
    blk = DeviceBlock(shape, inp["layers"])
    xh = blk.tensor(inp["x"]).cpu().pin_memory()
    gh = blk.tensor(inp["g"]).cpu().pin_memory()
    yh, dxh = torch.empty_like(xh).pin_memory(), torch.empty_like(xh).pin_memory()
    blk.step(xh, gh, yh, dxh)  # makes the copy stream
    torch.cuda.synchronize()
    L = lib()
    L.oases_debug_trace_enable.argtypes = [ctypes.c_int]
    L.oases_debug_trace_enable(1)
    try:
        blk.zero_grads()
        blk.step(xh, gh, yh, dxh)  # makes the trace events
        torch.cuda.synchronize()
        oases_shutdown()
        oases_shutdown()  # a second call finds nothing to release
        after = run_gpu(shape, inp)
        assert_identical(after, before)
        blk.zero_grads()
        blk.step(xh, gh, yh, dxh)
        torch.cuda.synchronize()
    finally:
        L.oases_debug_trace_enable(0)
    np.testing.assert_array_equal(yh.double().numpy(), before["y"])
    np.testing.assert_array_equal(dxh.double().numpy(), before["dx"])
    for k, v in blk.grads_numpy()[0].items():
        np.testing.assert_array_equal(v, before["grads"][0][k])


# ------------------------------------------------------------------ separate reduction
@pytest.mark.parametrize("mode", ["fine", "full"])
def test_separate_reduce_ffn_f32_h256(mode):
    """Shard partials in HBM + reduction kernel (C(F), C(R), C(B)) at fp32 tolerance."""
    shape = SHAPES["ffn_f32_h256"]
    inp = block_inputs(shape, seed=0)
    compare(shape, run_gpu(shape, inp, mode, reduce="separate"),
            oracle.run_step(shape, inp, mode=mode))


@pytest.mark.parametrize("kind", ["ffn", "attn", "layer"])
def test_separate_reduce_bf16_matches_oracle_and_fused(kind):
    shape = BlockShape(kind, "bf16", batch=2, seq=96, hidden=256, ffn=768, heads=2, w=2,
                       n_layers=2 if kind == "layer" else 1)
    inp = block_inputs(shape, seed=13, affine=True)
    sep = run_gpu(shape, inp, reduce="separate")
    compare(shape, sep, oracle.run_step(shape, inp, mode="fine"))
    fused = run_gpu(shape, inp, reduce="fused")
    assert rel(sep["y"], fused["y"]) < 1e-2 and rel(sep["dx"], fused["dx"]) < 1e-2


def test_separate_reduce_w4_full_recompute():
    shape = BlockShape("ffn", "bf16", batch=4, seq=64, hidden=256, ffn=1024, w=4)
    inp = block_inputs(shape, seed=14, affine=True)
    compare(shape, run_gpu(shape, inp, "full", reduce="separate"),
            oracle.run_step(shape, inp, mode="full"))


@pytest.mark.parametrize("kind", ["ffn", "layer"])
def test_separate_reduce_ragged_sub_batch_rows(kind):
    """200 rows per sub-batch: paired 128-row tiles with a ragged last pair, and
    the shard slabs of the split launch clipped at the sub-batch's last row."""
    shape = BlockShape(kind, "bf16", batch=2, seq=200, hidden=256, ffn=1024, heads=2, w=2)
    inp = block_inputs(shape, seed=15, affine=True)
    compare(shape, run_gpu(shape, inp, reduce="separate"), oracle.run_step(shape, inp, mode="fine"))


# ------------------------------------------------------------------ selective recompute
def test_layer_stack_selective_recompute():
    """SELECTIVE (the attention operation recomputed from kept Q, K, V; both
    layers' attention share one O/LSE buffer): against the oracle, and bit for
    bit equal to keeping everything."""
    shape = BlockShape("layer", "bf16", batch=2, seq=96, hidden=256, ffn=768, heads=2, w=2,
                       n_layers=2)
    inp = block_inputs(shape, seed=16, affine=True)
    sel = run_gpu(shape, inp, "selective")
    compare(shape, sel, oracle.run_step(shape, inp, mode="selective"))
    assert_identical(sel, run_gpu(shape, inp, "none"))
    assert_identical(sel, run_gpu(shape, inp, "fine"))


def test_attn_f32_selective_recompute():
    shape = BlockShape("attn", "f32", batch=2, seq=40, hidden=128, heads=4, w=2)
    inp = block_inputs(shape, seed=17, affine=True)
    compare(shape, run_gpu(shape, inp, "selective"), oracle.run_step(shape, inp, mode="selective"))
