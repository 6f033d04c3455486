"""Full-size workloads through the C ABI.

* Attention block, hidden 2048, 16 heads, seq 1024, batch 4, w=4: the whole
  step against the oracle.
* Transformer layer (hidden 4096, ffn 16384, 32 heads, seq 2048, w=8) and the
  4-layer stack (hidden 2560, ffn 10240, 20 heads, seq 2048, w=4): every
  kernel runs at its full per-sequence shape; one sequence is compared with the
  oracle (the oracle on the full batch would take minutes), and the full batch
  is tied to it by properties that hold at any size: a sequence's rows of y and
  dx do not depend on the other sequences (bit for bit), the weight gradients
  of the batch are the sum of the per-sequence ones, and the sub-batch split
  leaves y and dx bit-identical.
Tolerance: relative L2 per tensor <= 2e-2 against the oracle (bf16).
"""
import numpy as np
import pytest
import torch

import oracle
from synth import SHAPES, block_inputs
from tensor_model_transformer_tp_gb300 import oases_check_device
from tensor_model_transformer_tp_gb300.device import DeviceBlock, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_model_transformer_tp_gb300 import build_library
    build_library()


def rel(a, b):
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (n if n > 0 else 1.0))


def run_gpu(shape, inp, mode="fine"):
    blk = DeviceBlock(shape, inp["layers"], recompute=mode)
    y, dx = blk.step(blk.tensor(inp["x"]), blk.tensor(inp["g"]))
    torch.cuda.synchronize()
    oases_check_device(None)
    out = {"y": to_numpy(y), "dx": to_numpy(dx), "grads": blk.grads_numpy()}
    del blk
    torch.cuda.empty_cache()
    return out


def compare(got, ref, tol=2e-2):
    errs = {"y": rel(got["y"], ref["y"]), "dx": rel(got["dx"], ref["dx"])}
    for li, (gl, rl) in enumerate(zip(got["grads"], ref["grads"])):
        for k in rl:
            errs["L%d.%s" % (li, k)] = rel(gl[k], rl[k])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, bad
    return errs


def one_sequence(inp, shape, b):
    S = shape.seq
    sl = slice(b * S, (b + 1) * S)
    return {"x": inp["x"][sl], "g": inp["g"][sl], "layers": inp["layers"]}


def test_attn_bf16_h2048_full_size():
    shape = SHAPES["attn_bf16_h2048"]
    inp = block_inputs(shape, seed=0)
    compare(run_gpu(shape, inp), oracle.run_step(shape, inp, mode="fine"))


@pytest.mark.parametrize("name", ["layer_bf16_h4096", "stack4_bf16_h2560"])
def test_full_shapes_one_sequence_and_batch_properties(name):
    full = SHAPES[name]
    inp = block_inputs(full, seed=0)
    one = full.replace(batch=1, sub_batches=1)
    seq0 = one_sequence(inp, full, 0)
    got0 = run_gpu(one, seq0)
    compare(got0, oracle.run_step(one, seq0, mode="fine"))

    # the full batch, two sub-batches on two streams
    got = run_gpu(full, inp)
    S = full.seq
    np.testing.assert_array_equal(got["y"][:S], got0["y"])
    np.testing.assert_array_equal(got["dx"][:S], got0["dx"])
    # weight gradients of the batch = sum over sequences
    acc = [{k: v.copy() for k, v in g.items()} for g in got0["grads"]]
    for b in range(1, full.batch):
        gb = run_gpu(one, one_sequence(inp, full, b))
        np.testing.assert_array_equal(got["y"][b * S:(b + 1) * S], gb["y"])
        np.testing.assert_array_equal(got["dx"][b * S:(b + 1) * S], gb["dx"])
        for la, lb in zip(acc, gb["grads"]):
            for k in la:
                la[k] += lb[k]
    for la, lg in zip(acc, got["grads"]):
        for k in la:
            assert rel(lg[k], la[k]) <= 1e-5, k
    assert np.isfinite(got["y"]).all() and np.isfinite(got["dx"]).all()


def test_layer_full_batch_sub_batch_split_and_modes():
    full = SHAPES["layer_bf16_h4096"]
    inp = block_inputs(full, seed=1)
    two = run_gpu(full, inp, "fine")
    one = run_gpu(full.replace(sub_batches=1), inp, "fine")
    np.testing.assert_array_equal(two["y"], one["y"])
    np.testing.assert_array_equal(two["dx"], one["dx"])
    for mode in ("none", "selective"):
        other = run_gpu(full, inp, mode)
        np.testing.assert_array_equal(two["y"], other["y"])
        np.testing.assert_array_equal(two["dx"], other["dx"])
        for gf, gn in zip(two["grads"], other["grads"]):
            for k in gf:
                np.testing.assert_array_equal(gf[k], gn[k])
