"""MX-FP8 blocks (dtype "mxfp8": bf16 storage, every GEMM of F_i, F_j and their
backward on E4M3 operands with block-32 UE8M0 scales) through the C ABI,
against the oracle's MX variant (every product oracle.fp8.mx_product_bf16).

Tolerance: relative L2 per output tensor <= 4e-2 for one layer.  Both sides quantise the
same stored bf16 operands, but an operand computed upstream (LayerNorm, GeLU,
attention with bf16 probabilities, earlier GEMMs in fp32 against float64)
differs between them by up to a few bf16 units.  Where such a difference
crosses an E4M3 rounding boundary the element's code moves by one step, 2^-3
relative; the boundaries are 2^-4 apart (relative), so with upstream
differences of about 2^-8 at most one element in 16 can move, which bounds
the rms change of one product's output by sqrt(1/16) * 2^-3 ~ 3.1%, and the
residual path and averaging over a row keep the measured values well below.
In a stack, the first layer's gradients reach it through the later layer's
quantised products as well: up to four products on the gradient path of a
layer, so 3.1% * sqrt(4) ~ 6.2% (6e-2) for the two-layer case.
Bit-for-bit checks: the recompute modes give identical results on the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.fp8 as fp8
from synth import SHAPES, BlockShape, block_inputs
from tensor_model_transformer_tp_gb300 import OasesError, oases_check_device
from tensor_model_transformer_tp_gb300.device import DeviceBlock, to_numpy

pytestmark = pytest.mark.gpu

TOL = 4e-2        # one layer
TOL_STACK = 6e-2  # two layers


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
    return {"y": to_numpy(y), "dx": to_numpy(dx), "grads": blk.grads_numpy()}


def compare(got, ref, tol=TOL):
    errs = {"y": rel(got["y"], ref["y"]), "dx": rel(got["dx"], ref["dx"])}
    for li, (gl, rl) in enumerate(zip(got["grads"], ref["grads"])):
        for k in rl:
            errs["L%d.%s" % (li, k)] = rel(gl[k], rl[k])
    print("max rel-L2 %.3e" % max(errs.values()), {k: round(v, 5) for k, v in errs.items()})
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, bad
    return errs


CASES = {
    "ffn": BlockShape("ffn", "mxfp8", batch=4, seq=128, hidden=256, ffn=1024, w=4),
    "attn_ragged": BlockShape("attn", "mxfp8", batch=2, seq=160, hidden=256, heads=2, w=2),
    "layer_2": BlockShape("layer", "mxfp8", batch=2, seq=96, hidden=256, ffn=768, heads=2, w=2,
                          n_layers=2),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_mxfp8_block_against_the_mx_oracle(name):
    shape = CASES[name]
    inp = block_inputs(shape, seed=17, affine=True)
    compare(run_gpu(shape, inp), oracle.run_step(shape, inp, mode="fine", mm=fp8.mx_product_bf16),
            TOL_STACK if shape.n_layers > 1 else TOL)


def test_mxfp8_ffn_h1024_full_size():
    """The FFN workload's sizes (hidden 1024, ffn 4096, seq 512, batch 8, w = 4,
    two sub-batches) with MX-FP8 GEMMs."""
    shape = SHAPES["ffn_bf16_h1024"].replace(dtype="mxfp8")
    inp = block_inputs(shape, seed=0)
    compare(run_gpu(shape, inp), oracle.run_step(shape, inp, mode="fine", mm=fp8.mx_product_bf16))


def test_mxfp8_recompute_modes_bit_identical():
    shape = BlockShape("layer", "mxfp8", batch=2, seq=64, hidden=256, ffn=512, heads=2, w=2)
    inp = block_inputs(shape, seed=18, affine=True)
    r = {m: run_gpu(shape, inp, m) for m in ("none", "full", "fine", "selective")}
    for m in ("full", "fine", "selective"):
        np.testing.assert_array_equal(r[m]["y"], r["none"]["y"])
        np.testing.assert_array_equal(r[m]["dx"], r["none"]["dx"])
        for ga, gb in zip(r[m]["grads"], r["none"]["grads"]):
            for k in ga:
                np.testing.assert_array_equal(ga[k], gb[k])


def test_mxfp8_rejects_what_it_cannot_run():
    ok = BlockShape("ffn", "mxfp8", batch=2, seq=64, hidden=256, ffn=512, w=2)
    inp = block_inputs(ok, seed=19)
    with pytest.raises((OasesError, ValueError)):    # separate reduction: partials need bf16
        DeviceBlock(ok, inp["layers"], reduce="separate")
    bad = BlockShape("ffn", "mxfp8", batch=2, seq=64, hidden=256, ffn=96, w=2)   # ffn/w = 48
    with pytest.raises((OasesError, ValueError)):
        DeviceBlock(bad, block_inputs(bad, seed=19)["layers"])
