"""The seeded input recipe (synth/) and the separation of the oracle from the
CUDA path, checked on the CPU."""
import ast
import os

import numpy as np
import pytest
import torch

from synth import SHAPES, BlockShape, bf16_round, block_inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# The five workloads as specified for the block: kind, storage type, hidden,
# ffn, heads, seq, batch, w shards, sub-batches.
SPEC = {
    "ffn_f32_h256": ("ffn", "f32", 256, 1024, 0, 128, 2, 2, 2),
    "ffn_bf16_h1024": ("ffn", "bf16", 1024, 4096, 0, 512, 8, 4, 2),
    "attn_bf16_h2048": ("attn", "bf16", 2048, 0, 16, 1024, 4, 4, 2),
    "layer_bf16_h4096": ("layer", "bf16", 4096, 16384, 32, 2048, 4, 8, 2),
    "stack4_bf16_h2560": ("layer", "bf16", 2560, 10240, 20, 2048, 8, 4, 2),
}


@pytest.mark.parametrize("name", sorted(SPEC))
def test_workload_sizes(name):
    s = SHAPES[name]
    assert (s.kind, s.dtype, s.hidden, s.ffn, s.heads, s.seq, s.batch, s.w,
            s.sub_batches) == SPEC[name]
    assert s.head_dim in (0, 128)
    s.validate()


def test_special_options_of_the_small_workloads():
    assert not SHAPES["ffn_f32_h256"].pre_ln and not SHAPES["ffn_f32_h256"].residual
    assert SHAPES["stack4_bf16_h2560"].n_layers == 4
    for n in ("ffn_bf16_h1024", "attn_bf16_h2048", "layer_bf16_h4096", "stack4_bf16_h2560"):
        assert SHAPES[n].pre_ln and SHAPES[n].residual and SHAPES[n].causal


def test_distributions_follow_the_recipe():
    s = BlockShape("layer", "f32", batch=4, seq=256, hidden=512, ffn=2048, heads=4, w=2)
    inp = block_inputs(s, seed=0)
    x, g, p = inp["x"], inp["g"], inp["layers"][0]
    for a in (x, g):   # N(0, 1)
        assert abs(a.mean()) < 0.01 and abs(a.std() - 1.0) < 0.01
    for k in ("wqkv", "wo", "w1", "w2"):   # N(0, 0.02^2)
        assert abs(p[k].std() - 0.02) < 0.0005 and abs(p[k].mean()) < 0.0005
    for k in ("bqkv", "bo", "b1", "b2", "ln1_b", "ln2_b"):
        assert not p[k].any()
    assert (p["ln1_g"] == 1).all() and (p["ln2_g"] == 1).all()
    pa = block_inputs(s, seed=0, affine=True)["layers"][0]
    assert abs(pa["ln1_g"].mean() - 1.0) < 0.02 and abs(pa["ln1_g"].std() - 0.1) < 0.02
    assert abs(pa["b1"].std() - 0.02) < 0.002


def test_seeded_and_reproducible():
    s = BlockShape("ffn", "bf16", batch=2, seq=64, hidden=256, ffn=512, w=2)
    a, b, c = block_inputs(s, seed=3), block_inputs(s, seed=3), block_inputs(s, seed=4)
    assert np.array_equal(a["x"], b["x"]) and np.array_equal(a["layers"][0]["w1"],
                                                            b["layers"][0]["w1"])
    assert not np.array_equal(a["x"], c["x"])


def test_bf16_inputs_are_bf16_values():
    s = BlockShape("ffn", "bf16", batch=2, seq=64, hidden=256, ffn=512, w=2)
    inp = block_inputs(s, seed=1)
    for a in [inp["x"], inp["g"]] + list(inp["layers"][0].values()):
        assert not (a.view(np.uint32) & 0xFFFF).any()


def test_bf16_rounding_matches_a_library_conversion():
    rng = np.random.default_rng(0)
    wide = (rng.standard_normal(100000) * 10.0 ** rng.integers(-8, 8, 100000)).astype(np.float32)
    ties = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)  # halfway: to even
    a = np.concatenate([wide, ties])
    assert a.dtype == np.float32
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(bf16_round(a), ref)


def _imports(path):
    tree = ast.parse(open(path).read())
    out = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            out |= {a.name.split(".")[0] for a in node.names}
        elif isinstance(node, ast.ImportFrom) and node.module and node.level == 0:
            out.add(node.module.split(".")[0])
    return out


def _py_files(d):
    for root, _, files in os.walk(os.path.join(ROOT, d)):
        for f in files:
            if f.endswith(".py"):
                yield os.path.join(root, f)


def test_oracle_and_cuda_path_share_no_code():
    pkg = "tensor_model_transformer_tp_gb300"
    for f in _py_files("oracle"):
        bad = _imports(f) & {pkg, "ctypes", "torch"}
        assert not bad, (f, bad)
    for f in list(_py_files(pkg)) + [os.path.join(ROOT, "synth", "inputs.py")]:
        assert "oracle" not in _imports(f), f
    # the C/CUDA sources name nothing under oracle/
    csrc = os.path.join(ROOT, pkg, "csrc")
    for f in os.listdir(csrc):
        assert "oracle" not in open(os.path.join(csrc, f)).read().lower(), f
