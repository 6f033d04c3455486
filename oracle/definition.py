"""The block written as its plain, unsharded definition (oracle; test infrastructure only).

This is what the tensor-parallel computation must reproduce: Oases §IV, Eq. (1)
sums the w shard partials, and because the column split of F_i and the row split
of F_j partition the contraction dimension, that sum equals the unsharded
product exactly in real arithmetic.  No shards, no sub-batches, no schedule here.

FFN segment:  u = LN2(x) (if pre_ln, else u = x);  y = gelu(u W1^T + b1) W2^T + b2 (+ x)
Attention segment:  u = LN1(x);  [Q K V] = u Wqkv^T + bqkv, split into heads
   (Wqkv rows: Q heads 0..n_h-1, then K heads, then V heads, d rows each);
   O_h = softmax(Q_h K_h^T / sqrt(d), causal) V_h per sequence;  y = O Wo^T + bo (+ x)
Layer: attention segment then FFN segment.  Stack: layers in order.
Loss: L = sum(y * g).

Parity: pinned against the sharded schedule executor (sum of shard partials) and
used as the function whose finite differences pin the analytic backward.
"""
from __future__ import annotations

import numpy as np

from .ops import attention_head, gelu, layer_norm


def segment_kinds(shape):
    if shape.kind == "layer":
        return ["attn", "ffn"]
    return [shape.kind]


def _ln(x, g, b, shape):
    if not shape.pre_ln:
        return x
    return layer_norm(x, g, b, shape.eps)[0]


def _exact(A, B):
    return A @ B.T


def ffn_segment_plain(x, p, shape, mm=_exact):
    u = _ln(x, p["ln2_g"], p["ln2_b"], shape)
    h = gelu(mm(u, p["w1"]) + p["b1"])
    y = mm(h, p["w2"]) + p["b2"]
    return y + x if shape.residual else y


def attn_segment_plain(x, p, shape, mm=_exact):
    H, d, S = shape.hidden, shape.head_dim, shape.seq
    u = _ln(x, p["ln1_g"], p["ln1_b"], shape)
    qkv = mm(u, p["wqkv"]) + p["bqkv"]
    o = np.zeros_like(x)
    for b in range(x.shape[0] // S):
        r = slice(b * S, (b + 1) * S)
        for h in range(shape.heads):
            c = slice(h * d, (h + 1) * d)
            q = qkv[r, h * d:(h + 1) * d]
            k = qkv[r, H + h * d:H + (h + 1) * d]
            v = qkv[r, 2 * H + h * d:2 * H + (h + 1) * d]
            o[r, c] = attention_head(q, k, v, shape.causal)[0]
    y = mm(o, p["wo"]) + p["bo"]
    return y + x if shape.residual else y


def block_forward_plain(shape, x, layers, mm=_exact):
    """Forward of the whole block / layer / stack.  x is [rows, hidden].
    mm(A, B) = A B^T is every matrix product (exact unless given)."""
    y = np.asarray(x, dtype=np.float64)
    for p in layers:
        p = {k: np.asarray(v, dtype=np.float64) for k, v in p.items()}
        for kind in segment_kinds(shape):
            y = (ffn_segment_plain(y, p, shape, mm) if kind == "ffn"
                 else attn_segment_plain(y, p, shape, mm))
    return y


def block_loss_plain(shape, x, layers, g):
    """L = sum(y * g)."""
    return float((block_forward_plain(shape, x, layers) * np.asarray(g, np.float64)).sum())
