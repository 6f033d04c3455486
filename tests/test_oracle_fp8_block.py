"""Pins of the MX-FP8 variant of the block in the oracle (CPU only).

The variant runs the oracle's own schedule with every matrix product A B^T
replaced by oracle.fp8.mx_product_bf16 (both operands rounded to bf16, the
storage type, then MX-quantised along the contraction and multiplied as
mx_gemm, itself pinned in test_oracle_fp8.py).  Checked against things other
than itself:
* with the exact product the schedule is the one pinned by finite
  differences: bit-identical to the default;
* the sharded schedule (w = 1, 2, 4; scale blocks never straddle a shard's
  slice) equals the unsharded definition with the same product, forward;
* recompute modes NONE / FULL / FINE / SELECTIVE stay bit-identical, and the
  sub-batch split leaves y and dx bit-identical (each 32-block of a
  contraction is the same in both), gradients equal to 1e-12;
* every one of the seven products per FFN segment and sub-batch (two forward,
  one recomputed, four backward) goes through the product, each contracting
  over the axis it must (the batch rows for weight gradients);
* quantisation moves the result, but by no more than E4M3 precision allows;
* the bf16 rounding agrees with torch's conversion.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.fp8 as fp8
from oracle.definition import block_forward_plain
from oracle.schedule import exact_product
from synth import BlockShape, block_inputs

MX = fp8.mx_product_bf16


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


FFN = BlockShape("ffn", "mxfp8", batch=2, seq=32, hidden=64, ffn=256, w=2)
ATT = BlockShape("attn", "mxfp8", batch=2, seq=32, hidden=64, heads=2, w=2)
LAY = BlockShape("layer", "mxfp8", batch=2, seq=32, hidden=64, ffn=128, heads=2, w=2)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-20, 20, 20000),
                        [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)]])
    want = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(fp8.bf16_round(x.astype(np.float32).astype(np.float64)), want)


@pytest.mark.parametrize("shape", [FFN, ATT, LAY], ids=["ffn", "attn", "layer"])
def test_exact_product_is_the_default(shape):
    inp = block_inputs(shape, seed=1, affine=True)
    a = oracle.run_step(shape, inp, mode="fine")
    b = oracle.run_step(shape, inp, mode="fine", mm=exact_product)
    np.testing.assert_array_equal(a["y"], b["y"])
    np.testing.assert_array_equal(a["dx"], b["dx"])


@pytest.mark.parametrize("shape,w", [(FFN, 1), (FFN, 2), (FFN, 4), (ATT, 2), (LAY, 2)])
def test_sharded_mx_forward_equals_unsharded_definition(shape, w):
    inp = block_inputs(shape, seed=2, affine=True)
    got = oracle.run_step(shape, inp, mode="fine", w=w, mm=MX)["y"]
    want = block_forward_plain(shape, inp["x"], inp["layers"], mm=MX)
    assert rel(got, want) <= 1e-12


@pytest.mark.parametrize("shape", [FFN, LAY], ids=["ffn", "layer"])
def test_mx_recompute_modes_bit_identical_and_sub_batch_invariant(shape):
    inp = block_inputs(shape, seed=3, affine=True)
    r = {m: oracle.run_step(shape, inp, mode=m, mm=MX) for m in ("none", "full", "fine", "selective")}
    for m in ("full", "fine", "selective"):
        np.testing.assert_array_equal(r[m]["y"], r["none"]["y"])
        np.testing.assert_array_equal(r[m]["dx"], r["none"]["dx"])
        for ga, gb in zip(r[m]["grads"], r["none"]["grads"]):
            for k in ga:
                np.testing.assert_array_equal(ga[k], gb[k])
    one = oracle.run_step(shape, inp, mode="fine", sub_batches=1, mm=MX)
    np.testing.assert_array_equal(one["y"], r["fine"]["y"])
    np.testing.assert_array_equal(one["dx"], r["fine"]["dx"])
    for ga, gb in zip(one["grads"], r["fine"]["grads"]):
        for k in ga:
            assert rel(ga[k], gb[k]) <= 1e-12, k


def test_every_ffn_product_goes_through_the_hook_with_its_contraction():
    shape = FFN.replace(w=1, sub_batches=2)
    inp = block_inputs(shape, seed=4)
    calls = []

    def spy(A, B):
        calls.append((A.shape, B.shape))
        return MX(A, B)

    oracle.run_step(shape, inp, mode="fine", mm=spy)
    Ms, H, F = shape.rows // 2, shape.hidden, shape.ffn
    want = sorted([((Ms, H), (F, H))] * 2        # column GEMM, forward and recompute
                  + [((Ms, F), (H, F))]          # row GEMM
                  + [((H, Ms), (F, Ms))]         # dW2 = dy^T h: over the rows
                  + [((Ms, H), (F, H))]          # dH = dy W2: over hidden
                  + [((F, Ms), (H, Ms))]         # dW1 = dA^T u: over the rows
                  + [((Ms, F), (H, F))])         # du = dA W1: over ffn
    got = sorted(calls)
    assert got == sorted(want * 2), got          # two sub-batches


@pytest.mark.parametrize("shape", [FFN, LAY], ids=["ffn", "layer"])
def test_quantisation_moves_results_within_e4m3_precision(shape):
    inp = block_inputs(shape, seed=5, affine=True)
    mx = oracle.run_step(shape, inp, mode="fine", mm=MX)
    ex = oracle.run_step(shape, inp, mode="fine")
    # each operand element carries at most 2^-4 relative rounding (3.6% rms
    # for uniform rounding), a product of two such operands about 5%; a
    # weight gradient passes through up to three quantised products
    for key in ("y", "dx"):
        assert 1e-5 < rel(mx[key], ex[key]) < 0.1, key
    for gm, ge in zip(mx["grads"], ex["grads"]):
        for k in ("w1", "w2") if shape.kind == "ffn" else ("w1", "w2", "wqkv", "wo"):
            assert 1e-3 < rel(gm[k], ge[k]) < 0.25, k
