"""Oases training schedule over w simulated shards (oracle; test infrastructure only).

Follows Oases §IV (Algorithm 1 and Figs. 4a, 4b, 4d) in the pages' order and
notation, at the granularity of one tensor-parallel segment (an FFN or an
attention block).  A segment s contributes five operators to the flattened
operator sequence O:

  ln_s   compute  u = LN(x_s) (identity when the block has no pre-LayerNorm)
  f_s    comm     forward: identity (u is replicated on every shard);
                  backward: AllReduce of the shard input-gradients (C_s(B))
  col_s  compute  column-parallel F_i, per shard k: FFN A_k = u W1_k^T + b1_k,
                  H_k = gelu(A_k); attention QKV_k = u Wqkv_k^T + bqkv_k and
                  O_k = causal softmax attention over the heads of shard k
  row_s  compute  row-parallel F_j, per shard k: P_k = H_k W2_k^T (or O_k Wo_k^T)
  g_s    comm     forward: AllReduce y = sum_k P_k (Oases §IV, Eq. (1)), then the
                  bias once and the residual: y + b (+ x_s) = x_{s+1};
                  backward: identity, dP_k = dy for every k because dy/dP_k = 1

Shard k owns rows [k F/w, (k+1) F/w) of W1 and the same columns of W2, or
heads [k n_h/w, (k+1) n_h/w) of each of Q, K, V and the matching Wo columns.

Schedule (Algorithm 1):
  * the batch is split into n_sb sub-batches (contiguous row slices);
  * forward: per sub-batch run the compute operators' Forward; at a
    communication operator StartAsync it and switch sub-batch; a sub-batch
    Syncs its outstanding communication before it continues;
  * the operators finished after each communication operator are saved as a
    recompute sequence with the communication operators dropped; only the
    first input of each sequence is stored (here x_s);
  * backward: walk the saved sequences in reverse; per sequence Recompute, then
    Backward in reverse operator order; backward communication (C(B)) is
    started asynchronously and the sub-batch is switched, so it overlaps the
    other sub-batch's Recompute and Backward, across sequence boundaries.

Recompute modes:
  "none": no recomputation; the forward keeps every activation.
  "full": the default of Fig. 4a: the sequence is recomputed as the forward
          ran it, including the row GEMM and its AllReduce C(R).
  "fine": Fig. 4d: recomputation starts after the communication operator and
          C(R) is dropped.  Reading: the row operator is not recomputed either,
          since its output reaches only that dropped AllReduce and no Backward
          operation of the sequence reads it.  Backward order per segment pair
          is (R_j, B_j, R_i, B_i, C_i(B)) with j the later segment.
  "selective": the selective recomputation the pages compare against in
          §VI ("Megatron SS"): every activation is kept except the output of
          the attention operation, which is recomputed (operator "attn": the
          causal softmax attention of each shard's heads from the stored Q, K,
          V) before the attention segment's Backward.  FFN segments keep
          everything, as in "none".

Weight gradients are summed (the loss is a sum) and accumulated in sub-batch
order 0, 1, ...

Parity: pinned by tests (sharded sum vs unsharded definition, fine == full ==
none bit for bit, finite differences, sub-batch invariance, trace counts).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np

from .ops import (attention_head, attention_head_backward, gelu, gelu_grad, layer_norm,
                  layer_norm_backward)


@dataclasses.dataclass(frozen=True)
class Op:
    name: str   # "ln", "f", "col", "row", "g"
    seg: int
    kind: str   # "compute" or "comm"


class Trace(list):
    """List of (event, op_name, segment, sub_batch); event in
    F, R, B (compute operations), C(F), C(R), C(B) (StartAsync of a
    communication operation) and Sync."""

    def count_event(self, event: str) -> int:
        return sum(1 for e in self if e[0] == event)


def exact_product(A, B):
    """A B^T in float64: the products of the block as the pages define them."""
    return A @ B.T


class _Segment:
    def __init__(self, index: int, layer: int, kind: str, p: Dict[str, np.ndarray], shape, w: int,
                 mm=exact_product):
        self.s, self.layer, self.kind, self.shape, self.w = index, layer, kind, shape, w
        self.p = p
        # every matrix product of the segment, forward and backward, is
        # mm(A, B) = A B^T, contracting over the columns of both operands
        self.mm = mm
        H = shape.hidden
        if kind == "ffn":
            F = shape.ffn
            fw = F // w
            self.cols = [slice(k * fw, (k + 1) * fw) for k in range(w)]
            self.names = dict(g="ln2_g", b="ln2_b", wc="w1", bc="b1", wr="w2", br="b2")
        else:
            hw = H // w  # hidden columns owned by one shard (n_h / w heads of d)
            self.cols = [slice(k * hw, (k + 1) * hw) for k in range(w)]
            self.qkv_rows = [np.r_[k * hw:(k + 1) * hw, H + k * hw:H + (k + 1) * hw,
                                   2 * H + k * hw:2 * H + (k + 1) * hw] for k in range(w)]
            self.names = dict(g="ln1_g", b="ln1_b", wc="wqkv", bc="bqkv", wr="wo", br="bo")

    # ---- forward operations -------------------------------------------------
    def ln_fwd(self, a):
        x = a[(self.s, "x")]
        if self.shape.pre_ln:
            u, mu, rstd = layer_norm(x, self.p[self.names["g"]], self.p[self.names["b"]],
                                     self.shape.eps)
            a[(self.s, "u")], a[(self.s, "mu")], a[(self.s, "rstd")] = u, mu, rstd
        else:
            a[(self.s, "u")] = x

    def _attn_shard(self, qkv_k):
        """Causal attention over the heads of one shard; qkv_k is [rows, 3 H/w]."""
        S, d = self.shape.seq, self.shape.head_dim
        hw = qkv_k.shape[1] // 3
        o = np.zeros((qkv_k.shape[0], hw))
        for b in range(qkv_k.shape[0] // S):
            r = slice(b * S, (b + 1) * S)
            for j in range(hw // d):
                c = slice(j * d, (j + 1) * d)
                q = qkv_k[r, j * d:(j + 1) * d]
                k = qkv_k[r, hw + j * d:hw + (j + 1) * d]
                v = qkv_k[r, 2 * hw + j * d:2 * hw + (j + 1) * d]
                o[r, c] = attention_head(q, k, v, self.shape.causal)[0]
        return o

    def col_fwd(self, a):
        u = a[(self.s, "u")]
        wc, bc = self.p[self.names["wc"]], self.p[self.names["bc"]]
        if self.kind == "ffn":
            A = [self.mm(u, wc[c]) + bc[c] for c in self.cols]
            a[(self.s, "A")] = A
            a[(self.s, "H")] = [gelu(Ak) for Ak in A]
        else:
            QKV = [self.mm(u, wc[r]) + bc[r] for r in self.qkv_rows]
            a[(self.s, "QKV")] = QKV
            a[(self.s, "H")] = [self._attn_shard(q) for q in QKV]

    def attn_fwd(self, a):
        """The attention operation alone, from the stored Q, K, V of every shard."""
        a[(self.s, "H")] = [self._attn_shard(q) for q in a[(self.s, "QKV")]]

    def row_fwd(self, a):
        wr = self.p[self.names["wr"]]
        a[(self.s, "P")] = [self.mm(Hk, wr[:, c]) for Hk, c in zip(a[(self.s, "H")], self.cols)]

    def g_fwd(self, a) -> np.ndarray:
        """C(F): y = sum_{k=0}^{w-1} P_k, then + bias (+ x_s)."""
        P = a[(self.s, "P")]
        y = P[0].copy()
        for Pk in P[1:]:
            y = y + Pk
        y = y + self.p[self.names["br"]]
        if self.shape.residual:
            y = y + a[(self.s, "x")]
        return y

    # ---- backward operations ------------------------------------------------
    def g_bwd(self, a, grads):
        dy = a[(self.s, "dy")]
        a[(self.s, "dP")] = [dy] * self.w          # Eq. (1): dy/dP_k = 1
        grads[self.names["br"]] += dy.sum(axis=0)
        if self.shape.residual:
            a[(self.s, "dres")] = dy

    def row_bwd(self, a, grads):
        wr = self.p[self.names["wr"]]
        dH = []
        for Hk, dPk, c in zip(a[(self.s, "H")], a[(self.s, "dP")], self.cols):
            grads[self.names["wr"]][:, c] += self.mm(dPk.T, Hk.T)
            dH.append(self.mm(dPk, wr[:, c].T))
        a[(self.s, "dH")] = dH

    def col_bwd(self, a, grads):
        u = a[(self.s, "u")]
        wc = self.p[self.names["wc"]]
        dus = []
        if self.kind == "ffn":
            for Ak, dHk, c in zip(a[(self.s, "A")], a[(self.s, "dH")], self.cols):
                dA = dHk * gelu_grad(Ak)
                grads[self.names["bc"]][c] += dA.sum(axis=0)
                grads[self.names["wc"]][c] += self.mm(dA.T, u.T)
                dus.append(self.mm(dA, wc[c].T))
        else:
            S, d = self.shape.seq, self.shape.head_dim
            for qkv_k, dO, r in zip(a[(self.s, "QKV")], a[(self.s, "dH")], self.qkv_rows):
                hw = qkv_k.shape[1] // 3
                dqkv = np.zeros_like(qkv_k)
                for b in range(qkv_k.shape[0] // S):
                    rr = slice(b * S, (b + 1) * S)
                    for j in range(hw // d):
                        cq = slice(j * d, (j + 1) * d)
                        ck = slice(hw + j * d, hw + (j + 1) * d)
                        cv = slice(2 * hw + j * d, 2 * hw + (j + 1) * d)
                        q, k, v = qkv_k[rr, cq], qkv_k[rr, ck], qkv_k[rr, cv]
                        p = attention_head(q, k, v, self.shape.causal)[1]
                        dq, dk, dv = attention_head_backward(dO[rr, cq], q, k, v, p)
                        dqkv[rr, cq], dqkv[rr, ck], dqkv[rr, cv] = dq, dk, dv
                grads[self.names["bc"]][r] += dqkv.sum(axis=0)
                grads[self.names["wc"]][r] += self.mm(dqkv.T, u.T)
                dus.append(self.mm(dqkv, wc[r].T))
        a[(self.s, "du_k")] = dus

    def f_bwd(self, a):
        """C(B): du = sum_{k=0}^{w-1} du_k (AllReduce of the shard input-gradients)."""
        du_k = a[(self.s, "du_k")]
        du = du_k[0].copy()
        for d in du_k[1:]:
            du = du + d
        a[(self.s, "du")] = du

    def ln_bwd(self, a, grads):
        du = a[(self.s, "du")]
        if self.shape.pre_ln:
            dx, dg, db = layer_norm_backward(du, a[(self.s, "x")], a[(self.s, "mu")],
                                             a[(self.s, "rstd")], self.p[self.names["g"]])
            grads[self.names["g"]] += dg
            grads[self.names["b"]] += db
        else:
            dx = du
        if self.shape.residual:
            dx = dx + a[(self.s, "dres")]
        return dx


def _segments(shape, layers, w, mm=exact_product):
    kinds = ["attn", "ffn"] if shape.kind == "layer" else [shape.kind]
    segs = []
    for li, p in enumerate(layers):
        for kind in kinds:
            segs.append(_Segment(len(segs), li, kind, p, shape, w, mm))
    return segs


def build_operator_sequence(n_segments: int) -> List[Op]:
    """Flattened operator sequence O of Algorithm 1 for n_segments segments."""
    O = []
    for s in range(n_segments):
        O += [Op("ln", s, "compute"), Op("f", s, "comm"), Op("col", s, "compute"),
              Op("row", s, "compute"), Op("g", s, "comm")]
    return O


def recompute_ops(seq: List[Op], mode: str, kind: str = None) -> List[Op]:
    """Operators re-run by the Recompute phase of one saved sequence (kind:
    the segment's "ffn" or "attn", needed by the selective mode)."""
    if mode == "none":
        return []
    if mode == "selective":
        return [Op("attn", seq[0].seg, "compute")] if kind == "attn" else []
    if mode == "full":
        return list(seq)                       # as the forward ran it, incl. C(R)
    # fine: communication dropped; the row operator's output only feeds the
    # dropped AllReduce, so it is not recomputed either.
    return [op for op in seq if op.kind == "compute" and op.name != "row"]


def run_step(shape, inputs, mode: str = "fine", sub_batches: int = None, w: int = None,
             mm=exact_product):
    """One training step (forward, recompute, backward) of the block.

    mm(A, B) = A B^T is every matrix product of the step (default: exact);
    oracle.fp8.mx_product_bf16 gives the MX-FP8 variant of the block's GEMMs.

    inputs: {"x": [rows, hidden], "g": [rows, hidden], "layers": [params...]}.
    Returns dict with y, dx (float64, [rows, hidden]), grads (list per layer of
    {name: float64 array}), trace (Trace) and saved_bytes (activation bytes
    held between the forward and the backward, all sub-batches, excluding y).
    """
    assert mode in ("none", "full", "fine", "selective"), mode
    n_sb = shape.sub_batches if sub_batches is None else sub_batches
    w = shape.w if w is None else w
    layers = [{k: np.asarray(v, dtype=np.float64) for k, v in p.items()} for p in inputs["layers"]]
    x = np.asarray(inputs["x"], dtype=np.float64)
    g = np.asarray(inputs["g"], dtype=np.float64)
    M = x.shape[0]
    assert M % n_sb == 0 and (M // n_sb) % max(shape.seq, 1) == 0
    Mb = M // n_sb
    segs = _segments(shape, layers, w, mm)
    nS = len(segs)
    O = build_operator_sequence(nS)
    grads = [{k: np.zeros_like(v) for k, v in p.items()} for p in layers]
    acts = [{(0, "x"): x[b * Mb:(b + 1) * Mb]} for b in range(n_sb)]
    trace = Trace()

    # ---------------- forward (Algorithm 1: split, Forward, StartAsync/Sync) ----
    runs: List[List[Op]] = [[]]
    for op in O:
        if op.name == "f":
            continue                             # no forward communication
        runs[-1].append(op)
        if op.name == "g":
            runs.append([])
    runs = [r for r in runs if r]
    pending = [None] * n_sb
    for run in runs:
        for b in range(n_sb):
            a = acts[b]
            if pending[b] is not None:
                trace.append(("Sync",) + pending[b] + (b,))
                pending[b] = None
            for op in run:
                seg = segs[op.seg]
                if op.name == "g":
                    y = seg.g_fwd(a)
                    a[(op.seg + 1, "x") if op.seg + 1 < nS else "y"] = y
                    trace.append(("C(F)", "g", op.seg, b))
                    pending[b] = ("g", op.seg)
                else:
                    getattr(seg, op.name + "_fwd")(a)
                    trace.append(("F", op.name, op.seg, b))
    for b in range(n_sb):
        if pending[b] is not None:
            trace.append(("Sync",) + pending[b] + (b,))
            pending[b] = None

    # Saved recompute sequences: one per segment, first input x_s stored.
    seqs = [[op for op in O if op.seg == s] for s in range(nS)]
    if mode == "selective":
        for a in acts:
            for s in range(nS):
                if segs[s].kind == "attn":
                    del a[(s, "H")]              # the attention output, recomputed
    elif mode != "none":
        for a in acts:
            for key in list(a.keys()):
                if not (key == "y" or (isinstance(key, tuple) and key[1] == "x")):
                    del a[key]
    saved = 0
    for a in acts:
        for key, v in a.items():
            if key == "y":
                continue
            vs = v if isinstance(v, list) else [v]
            saved += sum(np.asarray(t).nbytes for t in vs)

    # ---------------- backward (Algorithm 1: reverse, Recompute, Backward) -----
    for b in range(n_sb):
        acts[b][(nS - 1, "dy")] = g[b * Mb:(b + 1) * Mb]
    # Per sub-batch stream of (phase, op); it is cut after every C(B) StartAsync.
    stream: List[Tuple[str, Op]] = []
    for seq in reversed(seqs):
        stream += [("R", op) for op in recompute_ops(seq, mode, segs[seq[0].seg].kind)]
        stream += [("B", op) for op in reversed(seq)]
    bruns: List[List[Tuple[str, Op]]] = [[]]
    for item in stream:
        bruns[-1].append(item)
        if item[0] == "B" and item[1].name == "f":
            bruns.append([])
    bruns = [r for r in bruns if r]
    for run in bruns:
        for b in range(n_sb):
            a = acts[b]
            if pending[b] is not None:
                trace.append(("Sync",) + pending[b] + (b,))
                pending[b] = None
            for phase, op in run:
                seg = segs[op.seg]
                gl = grads[seg.layer]
                if phase == "R":
                    if op.name == "g":
                        seg.g_fwd(a)                 # C(R): recomputed AllReduce, unused
                        trace.append(("C(R)", "g", op.seg, b))
                    elif op.name == "f":
                        pass                         # identity forward, nothing to do
                    else:
                        getattr(seg, op.name + "_fwd")(a)
                        trace.append(("R", op.name, op.seg, b))
                    continue
                if op.name == "g":
                    seg.g_bwd(a, gl)
                    trace.append(("B", "g", op.seg, b))
                elif op.name == "row":
                    seg.row_bwd(a, gl)
                    trace.append(("B", "row", op.seg, b))
                elif op.name == "col":
                    seg.col_bwd(a, gl)
                    trace.append(("B", "col", op.seg, b))
                elif op.name == "f":
                    seg.f_bwd(a)
                    trace.append(("C(B)", "f", op.seg, b))
                    pending[b] = ("f", op.seg)
                else:  # ln
                    dx = seg.ln_bwd(a, gl)
                    trace.append(("B", "ln", op.seg, b))
                    if op.seg > 0:
                        a[(op.seg - 1, "dy")] = dx
                    else:
                        a["dx"] = dx
                    # the segment's activations are no longer needed
                    for key in [k for k in a if isinstance(k, tuple) and k[0] == op.seg]:
                        del a[key]
    for b in range(n_sb):
        if pending[b] is not None:
            trace.append(("Sync",) + pending[b] + (b,))
            pending[b] = None

    y = np.concatenate([a["y"] for a in acts], axis=0)
    dx = np.concatenate([a["dx"] for a in acts], axis=0)
    return {"y": y, "dx": dx, "grads": grads, "trace": trace, "saved_bytes": saved}
