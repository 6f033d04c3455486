"""Seeded synthetic workloads for the tensor-parallel transformer block.

Both the CPU oracle (through the tests) and the CUDA path take their inputs from
here, so that the two sides see the same numbers.  Nothing in this module
computes any part of the block: it only draws normal variates from numpy's
PCG64 generator and, for bf16 workloads, rounds them to the nearest bf16 value
(round-to-nearest-even), which is the storage type the CUDA path reads.

Draw order (fixed, so a workload is reproducible from its seed alone):
  x, then for every layer the parameters in the order of ``PARAM_NAMES`` that
  the block kind uses, then the loss weights g.
Weights are N(0, 0.02^2); x and g are N(0, 1).  Biases are 0 and LayerNorm
gamma/beta are 1/0 unless ``affine=True``, in which case biases are
N(0, 0.02^2), gamma ~ N(1, 0.1^2) and beta ~ N(0, 0.1^2) (used to exercise the
bias and LayerNorm-parameter gradients).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import numpy as np

# Parameter names, in draw order and in the order of the C-ABI weight struct.
PARAM_NAMES = ("ln1_g", "ln1_b", "wqkv", "bqkv", "wo", "bo",
               "ln2_g", "ln2_b", "w1", "b1", "w2", "b2")


@dataclasses.dataclass(frozen=True)
class BlockShape:
    """Shape and options of one block workload.

    kind: "ffn" (LN? -> W1 column GEMM + GeLU -> W2 row GEMM -> shard sum),
          "attn" (LN -> QKV column GEMM -> causal attention -> Wo row GEMM -> shard sum),
          "layer" (attn segment then ffn segment).
    n_layers > 1 makes a stack of identical-shape layers.
    """
    kind: str
    dtype: str            # "f32", "bf16" or "mxfp8" (bf16 storage, MX-FP8 GEMM operands)
    batch: int
    seq: int
    hidden: int
    ffn: int = 0
    heads: int = 0
    w: int = 1            # simulated tensor-parallel shards
    sub_batches: int = 2
    pre_ln: bool = True
    residual: bool = True
    causal: bool = True
    n_layers: int = 1
    eps: float = 1e-5

    @property
    def rows(self) -> int:
        return self.batch * self.seq

    @property
    def head_dim(self) -> int:
        return self.hidden // self.heads if self.heads else 0

    def replace(self, **kw) -> "BlockShape":
        return dataclasses.replace(self, **kw)

    def validate(self) -> None:
        assert self.kind in ("ffn", "attn", "layer"), self.kind
        assert self.dtype in ("f32", "bf16", "mxfp8"), self.dtype
        assert self.batch >= 0 and self.seq >= 0 and self.hidden > 0
        assert self.sub_batches >= 1 and self.batch % self.sub_batches == 0
        if self.kind in ("ffn", "layer"):
            assert self.ffn > 0 and self.ffn % self.w == 0
        if self.kind in ("attn", "layer"):
            assert self.heads > 0 and self.hidden % self.heads == 0
            assert self.heads % self.w == 0


# The five workloads: sizes and options as they are specified for this block.
SHAPES: Dict[str, BlockShape] = {
    # FFN block, fp32, no LayerNorm, no residual, bias 0: F_i -> F_j -> C_i exactly.
    "ffn_f32_h256": BlockShape("ffn", "f32", batch=2, seq=128, hidden=256, ffn=1024,
                               w=2, sub_batches=2, pre_ln=False, residual=False),
    # Pre-LN FFN block, bf16 storage with fp32 accumulation.
    "ffn_bf16_h1024": BlockShape("ffn", "bf16", batch=8, seq=512, hidden=1024, ffn=4096,
                                 w=4, sub_batches=2),
    # Pre-LN causal attention block, 16 heads of 128.
    "attn_bf16_h2048": BlockShape("attn", "bf16", batch=4, seq=1024, hidden=2048, heads=16,
                                  w=4, sub_batches=2),
    # Full pre-LN transformer layer (attention segment then FFN segment).
    "layer_bf16_h4096": BlockShape("layer", "bf16", batch=4, seq=2048, hidden=4096, ffn=16384,
                                   heads=32, w=8, sub_batches=2),
    # Four-layer GPT-style stack.
    "stack4_bf16_h2560": BlockShape("layer", "bf16", batch=8, seq=2048, hidden=2560, ffn=10240,
                                    heads=20, w=4, sub_batches=2, n_layers=4),
}


def attn_param_names() -> List[str]:
    return ["ln1_g", "ln1_b", "wqkv", "bqkv", "wo", "bo"]


def ffn_param_names() -> List[str]:
    return ["ln2_g", "ln2_b", "w1", "b1", "w2", "b2"]


def _param_shape(name: str, s: BlockShape):
    H, F = s.hidden, s.ffn
    return {"ln1_g": (H,), "ln1_b": (H,), "wqkv": (3 * H, H), "bqkv": (3 * H,),
            "wo": (H, H), "bo": (H,), "ln2_g": (H,), "ln2_b": (H,),
            "w1": (F, H), "b1": (F,), "w2": (H, F), "b2": (H,)}[name]


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even), kept as float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def block_inputs(s: BlockShape, seed: int = 0, affine: bool = False) -> Dict:
    """Draw x [rows, hidden], per-layer parameters and g [rows, hidden].

    Returns {"x": ndarray, "g": ndarray, "layers": [ {name: ndarray}, ... ]},
    all float32 (bf16-representable when ``s.dtype`` is "bf16" or "mxfp8").
    """
    s.validate()
    rng = np.random.Generator(np.random.PCG64(seed))
    M, H = s.rows, s.hidden

    def normal(shape, std=1.0, mean=0.0):
        v = rng.standard_normal(shape, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if mean != 0.0:
            v += np.float32(mean)
        return v

    x = normal((M, H))
    names = []
    if s.kind in ("attn", "layer"):
        names += attn_param_names()
    if s.kind in ("ffn", "layer"):
        names += ffn_param_names()
    layers = []
    for _ in range(s.n_layers):
        p = {}
        for name in PARAM_NAMES:
            if name not in names:
                continue
            shape = _param_shape(name, s)
            if name.startswith("w"):
                p[name] = normal(shape, 0.02)
            elif name.endswith("_g"):
                p[name] = normal(shape, 0.1, 1.0) if affine else np.ones(shape, np.float32)
            elif name.endswith("_b") and name.startswith("ln"):
                p[name] = normal(shape, 0.1) if affine else np.zeros(shape, np.float32)
            else:  # linear biases
                p[name] = normal(shape, 0.02) if affine else np.zeros(shape, np.float32)
        layers.append(p)
    g = normal((M, H))
    if s.dtype in ("bf16", "mxfp8"):
        x = bf16_round(x)
        g = bf16_round(g)
        layers = [{k: bf16_round(v) for k, v in p.items()} for p in layers]
    return {"x": x, "g": g, "layers": layers}
