"""Pins of the CPU oracle against facts other than itself (CPU only).

Closed forms, textbook table values, invariants, brute force on tiny inputs
and finite differences, chosen so that a plausible mistake in the oracle (a
dropped term, a wrong sign or index, a transposed operand) fails one of them;
test_oracle_mutations.py plants such mistakes and checks that they are caught.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import ops
from synth import BlockShape, block_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny(kind, **kw):
    base = dict(batch=2, seq=4, hidden=8, ffn=16, heads=2, w=2, sub_batches=2)
    base.update(kw)
    return BlockShape(kind, "f32", **base)


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    n = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (n if n > 0 else 1.0)


# ---------------------------------------------------------------- LayerNorm
def test_layer_norm_closed_form():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 64)) * 3 + 7
    eps = 1e-5
    u, mu, rstd = ops.layer_norm(x, np.ones(64), np.zeros(64), eps)
    var = x.var(axis=1)
    np.testing.assert_allclose(u.mean(axis=1), 0, atol=1e-13)
    np.testing.assert_allclose(u.var(axis=1), var / (var + eps), rtol=1e-12)
    np.testing.assert_allclose(mu, x.mean(axis=1), rtol=1e-14)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(var + eps), rtol=1e-12)
    g, b = rng.normal(size=64), rng.normal(size=64)
    u2 = ops.layer_norm(x, g, b, eps)[0]
    np.testing.assert_allclose(u2, u * g + b, rtol=1e-12, atol=1e-12)


def test_layer_norm_constant_row_maps_to_beta():
    x = np.full((2, 16), 3.25)
    b = np.arange(16.0)
    u = ops.layer_norm(x, np.ones(16), b, 1e-5)[0]
    np.testing.assert_array_equal(u, np.tile(b, (2, 1)))


# -------------------------------------------------------------------- GeLU
def test_gelu_against_normal_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "normal_cdf.txt"))
            if l.strip() and not l.startswith("#")]
    for z, phi in rows:
        z, phi = float(z), float(phi)
        assert abs(ops.gelu(np.float64(z)) - z * phi) <= 1e-14 * max(1, abs(z))
        dens = math.exp(-z * z / 2) / math.sqrt(2 * math.pi)
        assert abs(ops.gelu_grad(np.float64(z)) - (phi + z * dens)) <= 1e-14


def test_gelu_special_values():
    assert ops.gelu(np.float64(0.0)) == 0.0
    assert ops.gelu_grad(np.float64(0.0)) == 0.5
    assert abs(ops.gelu(np.float64(12.0)) - 12.0) < 1e-12     # Phi(12) = 1 to fp64
    assert abs(ops.gelu(np.float64(-12.0))) < 1e-12
    # odd part of gelu is x/2:  gelu(x) - gelu(-x) = x
    z = np.linspace(-4, 4, 41)
    np.testing.assert_allclose(ops.gelu(z) - ops.gelu(-z), z, atol=1e-15)


# --------------------------------------------------------------- attention
def test_attention_single_token_returns_v():
    rng = np.random.default_rng(2)
    q, k, v = (rng.normal(size=(1, 8)) for _ in range(3))
    for causal in (True, False):
        np.testing.assert_array_equal(ops.attention_head(q, k, v, causal)[0], v)


def test_attention_causal_row0_and_mask_exact():
    rng = np.random.default_rng(3)
    q, k, v = (rng.normal(size=(6, 4)) for _ in range(3))
    o, p = ops.attention_head(q, k, v, True)
    np.testing.assert_array_equal(o[0], v[0])
    assert np.all(p[np.triu_indices(6, 1)] == 0.0)          # masked entries exactly zero
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-15)


def test_attention_zero_query_gives_running_mean():
    rng = np.random.default_rng(4)
    k, v = rng.normal(size=(7, 4)), rng.normal(size=(7, 4))
    q = np.zeros((7, 4))
    o = ops.attention_head(q, k, v, True)[0]
    ref = np.cumsum(v, axis=0) / np.arange(1, 8)[:, None]
    np.testing.assert_allclose(o, ref, rtol=1e-14, atol=1e-15)
    o2 = ops.attention_head(q, k, v, False)[0]
    np.testing.assert_allclose(o2, np.tile(v.mean(axis=0), (7, 1)), rtol=1e-14, atol=1e-15)


def test_attention_dominant_key():
    # one key with a huge logit for every query takes all the weight
    k = np.zeros((5, 4))
    k[2] = [40.0, 0, 0, 0]
    q = np.tile([[40.0, 0, 0, 0]], (5, 1))
    v = np.arange(20.0).reshape(5, 4)
    o = ops.attention_head(q, k, v, False)[0]
    np.testing.assert_allclose(o, np.tile(v[2], (5, 1)), atol=1e-12)


# ------------------------------------------- check 1: sum of shards = unsharded
@pytest.mark.parametrize("kind", ["ffn", "attn", "layer"])
@pytest.mark.parametrize("w", [1, 2, 4])
def test_shard_sum_equals_unsharded(kind, w):
    """Oases §IV, Eq. (1): y = sum_k x_k over w shards reproduces the unsharded block."""
    s = tiny(kind, heads=4, w=w)
    inp = block_inputs(s, seed=5, affine=True)
    yd = oracle.block_forward_plain(s, inp["x"], inp["layers"])
    ys = oracle.run_step(s, inp, mode="none")["y"]
    assert rel_l2(ys, yd) <= 1e-13


def test_w1_is_the_textbook_mlp():
    s = tiny("ffn", w=1, pre_ln=False, residual=False)
    inp = block_inputs(s, seed=6, affine=True)
    p = {k: v.astype(np.float64) for k, v in inp["layers"][0].items()}
    x = inp["x"].astype(np.float64)
    # brute force: one output element at a time, scalar loops
    y = oracle.run_step(s, inp, mode="fine", sub_batches=1)["y"]
    for m in (0, 5):
        for i in (0, 7):
            acc = p["b2"][i]
            for j in range(s.ffn):
                a = p["b1"][j] + sum(x[m, t] * p["w1"][j, t] for t in range(s.hidden))
                acc += p["w2"][i, j] * a * 0.5 * (1 + math.erf(a / math.sqrt(2)))
            assert abs(y[m, i] - acc) <= 1e-13 * max(1, abs(acc))


# ------------------------------------ check 2: fine == full == selective == none
@pytest.mark.parametrize("kind", ["ffn", "attn", "layer"])
def test_recompute_modes_bit_identical(kind):
    s = tiny(kind, n_layers=2)
    inp = block_inputs(s, seed=7, affine=True)
    r = {m: oracle.run_step(s, inp, mode=m) for m in ("none", "full", "fine", "selective")}
    for m in ("full", "fine", "selective"):
        np.testing.assert_array_equal(r[m]["y"], r["none"]["y"])
        np.testing.assert_array_equal(r[m]["dx"], r["none"]["dx"])
        for gl, gn in zip(r[m]["grads"], r["none"]["grads"]):
            for k in gn:
                np.testing.assert_array_equal(gl[k], gn[k])


# ------------------------------------------------- check 3: finite differences
def _fd_check(s, seed, h=1e-6, tol=1e-6):
    inp = block_inputs(s, seed=seed, affine=True)
    # weights of N(0, 0.3^2) keep every gradient well above the fp64 rounding
    # noise of a central difference (with 0.02 the grads of a no-LN block are ~1e-6)
    inp["layers"] = [{k: (v * 15 if k.startswith("w") else v) for k, v in p.items()}
                     for p in inp["layers"]]
    res = oracle.run_step(s, inp, mode="fine")
    x64 = inp["x"].astype(np.float64)
    layers = [{k: v.astype(np.float64) for k, v in p.items()} for p in inp["layers"]]
    g = inp["g"].astype(np.float64)

    def loss(xv, lv):
        return oracle.block_loss_plain(s, xv, lv, g)

    def fd(get_arr):
        arr = get_arr()
        out = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = loss(x64, layers)
            arr[idx] = old - h
            lm = loss(x64, layers)
            arr[idx] = old
            out[idx] = (lp - lm) / (2 * h)
        return out

    assert rel_l2(res["dx"], fd(lambda: x64)) <= tol
    for li, p in enumerate(layers):
        for name in p:
            num = fd(lambda: p[name])
            err = rel_l2(res["grads"][li][name], num)
            assert err <= tol, (li, name, err)


@pytest.mark.parametrize("kind", ["ffn", "attn", "layer"])
def test_finite_differences(kind):
    _fd_check(tiny(kind), seed=8)


def test_finite_differences_no_ln_no_residual_noncausal():
    _fd_check(tiny("layer", pre_ln=False, residual=False, causal=False), seed=9)


def test_finite_differences_two_layer_stack():
    _fd_check(tiny("layer", n_layers=2, w=1, batch=1, seq=3, hidden=4, ffn=8, sub_batches=1), seed=10)


# ------------------------------------------------- check 4: sub-batch split
@pytest.mark.parametrize("kind", ["ffn", "attn", "layer"])
def test_sub_batch_split_invariance(kind):
    s = tiny(kind, batch=4)
    inp = block_inputs(s, seed=11, affine=True)
    r1 = oracle.run_step(s, inp, mode="fine", sub_batches=1)
    r2 = oracle.run_step(s, inp, mode="fine", sub_batches=2)
    r4 = oracle.run_step(s, inp, mode="fine", sub_batches=4)
    for r in (r2, r4):
        np.testing.assert_array_equal(r["y"], r1["y"])
        np.testing.assert_array_equal(r["dx"], r1["dx"])
        for gl, g1 in zip(r["grads"], r1["grads"]):
            for k in g1:
                assert rel_l2(gl[k], g1[k]) <= 1e-12, k


# ------------------------------------------------------ invariants
def test_gradients_linear_in_g():
    s = tiny("layer")
    inp = block_inputs(s, seed=12, affine=True)
    g1 = inp["g"].astype(np.float64)
    g2 = np.roll(g1, 3)
    inp, inp2, inps = dict(inp, g=g1), dict(inp, g=g2), dict(inp, g=g1 + g2)
    a, b, c = (oracle.run_step(s, i, mode="fine") for i in (inp, inp2, inps))
    assert rel_l2(a["dx"] + b["dx"], c["dx"]) <= 1e-12
    for ga, gb, gc in zip(a["grads"], b["grads"], c["grads"]):
        for k in ga:
            assert rel_l2(ga[k] + gb[k], gc[k]) <= 1e-12, k


def test_head_permutation_invariance():
    """Relabelling heads consistently (Q, K, V rows and Wo columns) leaves y unchanged."""
    s = tiny("attn", heads=4, w=2)
    inp = block_inputs(s, seed=13, affine=True)
    p = dict(inp["layers"][0])
    H, d = s.hidden, s.head_dim
    perm = [2, 0, 3, 1]
    rows = np.concatenate([np.r_[blk * H + h * d: blk * H + (h + 1) * d]
                           for blk in range(3) for h in perm])
    cols = np.concatenate([np.r_[h * d:(h + 1) * d] for h in perm])
    q = dict(p, wqkv=p["wqkv"][rows], bqkv=p["bqkv"][rows], wo=p["wo"][:, cols])
    y0 = oracle.run_step(s, inp, mode="fine")["y"]
    y1 = oracle.run_step(s, dict(inp, layers=[q]), mode="fine")["y"]
    assert rel_l2(y1, y0) <= 1e-14


# ------------------------------------------------------ schedule / trace
def test_comm_counts_per_mode():
    """Oases §IV-A: three communication operators per segment (C(F), C(R), C(B))
    under the default recompute; fine-grained recomputation drops C(R)."""
    s = tiny("layer", n_layers=2)
    inp = block_inputs(s, seed=14)
    nseg = 4
    for mode, cr in (("none", 0), ("full", 1), ("fine", 0)):
        t = oracle.run_step(s, inp, mode=mode)["trace"]
        assert t.count_event("C(F)") == nseg * s.sub_batches
        assert t.count_event("C(R)") == cr * nseg * s.sub_batches
        assert t.count_event("C(B)") == nseg * s.sub_batches
        nsync = t.count_event("Sync")
        assert nsync == t.count_event("C(F)") + t.count_event("C(B)")


def test_fine_backward_order_and_overlap():
    """Per sub-batch: for each segment in reverse, R(ln), R(col), B(g), B(row),
    B(col), C(B), then B(ln); the other sub-batch runs between a C(B) StartAsync
    and its Sync (Algorithm 1; Fig. 4d)."""
    s = tiny("layer")
    t = oracle.run_step(s, block_inputs(s, seed=15), mode="fine")["trace"]
    bwd = t[[i for i, e in enumerate(t) if e[0] == "R"][0]:]
    sb0 = [e[:3] for e in bwd if e[-1] == 0 and e[0] != "Sync"]
    expect = []
    for seg in (1, 0):
        expect += [("R", "ln", seg), ("R", "col", seg), ("B", "g", seg), ("B", "row", seg),
                   ("B", "col", seg), ("C(B)", "f", seg), ("B", "ln", seg)]
    assert sb0 == expect
    # between sub-batch 0's C(B) and its Sync, sub-batch 1 computes
    i0 = bwd.index(("C(B)", "f", 1, 0))
    j0 = bwd.index(("Sync", "f", 1, 0))
    between = bwd[i0 + 1:j0]
    assert any(e[-1] == 1 and e[0] in ("R", "B") for e in between)


def test_recompute_stores_only_segment_inputs():
    """Oases §IV: only the first input of each recompute sequence is stored."""
    s = tiny("layer", n_layers=2)
    inp = block_inputs(s, seed=16)
    r = {m: oracle.run_step(s, inp, mode=m)["saved_bytes"] for m in ("none", "full", "fine")}
    one = s.rows * s.hidden * 8
    assert r["fine"] == r["full"] == 4 * one      # x_s for 4 segments
    assert r["none"] > r["fine"]


def test_selective_recomputes_only_the_attention_operation():
    """Selective recomputation (§VI, "Megatron SS"): no communication is
    re-run, only the attention operation of attention segments is recomputed,
    once per sub-batch, before that segment's Backward; the forward keeps every
    activation but the attention output (rows x hidden per attention segment)."""
    s = tiny("layer", n_layers=2)
    inp = block_inputs(s, seed=16)
    res = oracle.run_step(s, inp, mode="selective")
    t = res["trace"]
    rec = [e for e in t if e[0] == "R"]
    assert sorted(rec) == sorted(("R", "attn", seg, b) for seg in (0, 2)
                                 for b in range(s.sub_batches))
    assert t.count_event("C(R)") == 0
    for seg in (0, 2):
        for b in range(s.sub_batches):
            assert t.index(("R", "attn", seg, b)) < t.index(("B", "row", seg, b))
    none = oracle.run_step(s, inp, mode="none")["saved_bytes"]
    assert none - res["saved_bytes"] == 2 * s.rows * s.hidden * 8
    f = tiny("ffn")
    fi = block_inputs(f, seed=17)
    assert (oracle.run_step(f, fi, mode="selective")["saved_bytes"] ==
            oracle.run_step(f, fi, mode="none")["saved_bytes"])
    assert oracle.run_step(f, fi, mode="selective")["trace"].count_event("R") == 0


def test_empty_batch():
    s = tiny("ffn", batch=0)
    inp = block_inputs(s, seed=17)
    r = oracle.run_step(s, inp, mode="fine")
    assert r["y"].shape == (0, s.hidden) and r["dx"].shape == (0, s.hidden)
    assert all(np.all(v == 0) for v in r["grads"][0].values() if v.ndim == 2)


def test_attention_two_key_weights_pin_the_scale():
    """Logits are q.k / sqrt(d): with q.k1 = 2 and d = 4 key 1 gets weight e/(e+1)."""
    q = np.array([[2.0, 0, 0, 0], [2.0, 0, 0, 0]])
    k = np.array([[0.0, 0, 0, 0], [1.0, 0, 0, 0]])
    v = np.array([[0.0, 0, 0, 0], [1.0, 0, 0, 0]])
    o = ops.attention_head(q, k, v, False)[0]
    np.testing.assert_allclose(o[:, 0], math.e / (math.e + 1), rtol=1e-15)
    oc = ops.attention_head(q, k, v, True)[0]
    assert oc[0, 0] == 0.0 and abs(oc[1, 0] - math.e / (math.e + 1)) < 1e-15
