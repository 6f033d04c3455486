"""The causal mask, bit for bit, through the C ABI on the tensor-core path.

Causal attention lets token i see tokens j <= i of its own sequence only
(scale 1/sqrt(d), mask j <= i: the attention layer of the block, Oases §IV-A,
with the causal reading of the workloads).  Every other operator of the block
is row-wise.  So, exactly:

* y of tokens < t does not depend on x of tokens >= t: perturbing x there must
  leave those rows of y bit-identical;
* dx of tokens >= t does not depend on g (the loss weights) of tokens < t:
  perturbing g there must leave those rows of dx bit-identical.

A leak of any weight onto a future key (or of a past query's gradient onto a
later key's gradient) changes bits and fails here, where a relative-L2
comparison against the oracle would let a small leak through.  The cases put t
at the start of a 128-query tile, inside the diagonal 128-key block, one before
the end of a tile, and use a sequence length (200) that is not a multiple of
the tile, for the attention block (head dim 128, the tcgen05 kernels) and the
full layer (attention then FFN).
"""
import numpy as np
import pytest
import torch

from synth import BlockShape, block_inputs
from tensor_model_transformer_tp_gb300 import oases_check_device
from tensor_model_transformer_tp_gb300.device import DeviceBlock, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_model_transformer_tp_gb300 import build_library
    build_library()


SHAPES = {
    "attn": BlockShape("attn", "bf16", batch=2, seq=200, hidden=256, heads=2, w=2),
    "layer": BlockShape("layer", "bf16", batch=2, seq=200, hidden=256, ffn=512, heads=2, w=2),
}
CUTS = (1, 60, 127, 128, 150, 199)


def step(blk, x, g):
    blk.zero_grads()
    y, dx = blk.step(blk.tensor(x), blk.tensor(g))
    torch.cuda.synchronize()
    oases_check_device(None)
    return to_numpy(y), to_numpy(dx)


def perturbed(a, shape, rows_of_seq, seed):
    """a with the given token positions of every sequence replaced by fresh
    N(0, 1) values (rounded to bf16 by the device copy)."""
    out = np.array(a, dtype=np.float64, copy=True)
    rng = np.random.default_rng(seed)
    for b in range(shape.batch):
        r = b * shape.seq + rows_of_seq
        out[r] = rng.standard_normal((len(rows_of_seq), shape.hidden))
    return out


def seq_rows(shape, positions):
    return np.concatenate([b * shape.seq + positions for b in range(shape.batch)])


@pytest.mark.parametrize("kind", ["attn", "layer"])
def test_future_inputs_do_not_reach_past_outputs(kind):
    shape = SHAPES[kind]
    inp = block_inputs(shape, seed=31, affine=True)
    blk = DeviceBlock(shape, inp["layers"])
    y0, _ = step(blk, inp["x"], inp["g"])
    for k, t in enumerate(CUTS):
        x1 = perturbed(inp["x"], shape, np.arange(t, shape.seq), seed=100 + k)
        y1, _ = step(blk, x1, inp["g"])
        past, future = seq_rows(shape, np.arange(t)), seq_rows(shape, np.arange(t, shape.seq))
        np.testing.assert_array_equal(y1[past], y0[past], err_msg="cut %d" % t)
        assert not np.array_equal(y1[future], y0[future]), "the perturbation reached nothing"


@pytest.mark.parametrize("kind", ["attn", "layer"])
def test_past_loss_weights_do_not_reach_future_input_gradients(kind):
    shape = SHAPES[kind]
    inp = block_inputs(shape, seed=32, affine=True)
    blk = DeviceBlock(shape, inp["layers"])
    _, dx0 = step(blk, inp["x"], inp["g"])
    for k, t in enumerate(CUTS):
        g1 = perturbed(inp["g"], shape, np.arange(t), seed=200 + k)
        _, dx1 = step(blk, inp["x"], g1)
        past, future = seq_rows(shape, np.arange(t)), seq_rows(shape, np.arange(t, shape.seq))
        np.testing.assert_array_equal(dx1[future], dx0[future], err_msg="cut %d" % t)
        assert not np.array_equal(dx1[past], dx0[past]), "the perturbation reached nothing"
