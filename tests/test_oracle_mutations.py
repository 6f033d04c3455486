"""Plant plausible mistakes in the oracle (CPU only) and check that a pin fails.

Each case patches one oracle function with a wrong variant for the duration of
the test, runs the pins that should notice, and requires at least one of them
to fail.  Nothing here touches the CUDA path.
"""
import numpy as np
import pytest

import oracle
import oracle.definition as odef
import oracle.ops as oops
import oracle.schedule as osch
import test_oracle_pins as pins


def _caught(*checks):
    for chk in checks:
        try:
            chk()
        except AssertionError:
            return True
    return False


FD_FFN = lambda: pins._fd_check(pins.tiny("ffn"), seed=8)
FD_ATTN = lambda: pins._fd_check(pins.tiny("attn"), seed=8)
FD_LAYER = lambda: pins._fd_check(pins.tiny("layer"), seed=8)
SHARD = lambda: [pins.test_shard_sum_equals_unsharded(k, w) for k in ("ffn", "attn") for w in (2, 4)]


def test_gelu_grad_missing_density_term(monkeypatch):
    monkeypatch.setattr(osch, "gelu_grad", lambda a: oops.normal_cdf(a))
    assert _caught(FD_FFN)


def test_gelu_without_sqrt2(monkeypatch):
    from scipy.special import erf
    bad = lambda a: a * 0.5 * (1 + erf(a))
    monkeypatch.setattr(oops, "gelu", bad)
    assert _caught(pins.test_gelu_against_normal_table)


def test_layer_norm_unbiased_variance(monkeypatch):
    def bad(x, g, b, eps):
        mean = x.mean(axis=1)
        var = x.var(axis=1, ddof=1)
        rstd = 1 / np.sqrt(var + eps)
        return (x - mean[:, None]) * rstd[:, None] * g + b, mean, rstd
    monkeypatch.setattr(oops, "layer_norm", bad)
    assert _caught(pins.test_layer_norm_closed_form)


def test_layer_norm_backward_dropped_projection(monkeypatch):
    def bad(du, x, mean, rstd, gamma):
        gh = du * gamma
        dx = rstd[:, None] * (gh - gh.mean(axis=1, keepdims=True))
        xhat = (x - mean[:, None]) * rstd[:, None]
        return dx, (du * xhat).sum(0), du.sum(0)
    monkeypatch.setattr(osch, "layer_norm_backward", bad)
    assert _caught(FD_FFN)


def test_attention_missing_scale(monkeypatch):
    def bad(q, k, v, causal):
        S = q.shape[0]
        s = q @ k.T
        if causal:
            s = np.where(np.tril(np.ones((S, S), bool)), s, -np.inf)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        return p @ v, p
    monkeypatch.setattr(oops, "attention_head", bad)
    assert _caught(pins.test_attention_two_key_weights_pin_the_scale)


def test_attention_mask_off_by_one(monkeypatch):
    def bad(q, k, v, causal):
        S, d = q.shape
        s = q @ k.T / np.sqrt(d)
        if causal:
            s = np.where(np.tril(np.ones((S, S), bool), -1), s, -1e30)   # hides the diagonal
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        return p @ v, p
    monkeypatch.setattr(oops, "attention_head", bad)
    assert _caught(pins.test_attention_causal_row0_and_mask_exact,
                   pins.test_attention_zero_query_gives_running_mean)


def test_attention_backward_swapped_dq_dk(monkeypatch):
    orig = oops.attention_head_backward
    monkeypatch.setattr(osch, "attention_head_backward",
                        lambda *a: (lambda r: (r[1], r[0], r[2]))(orig(*a)))
    assert _caught(FD_ATTN)


def test_allreduce_backward_averaged_instead_of_identity(monkeypatch):
    """Eq. (1) gives dP_k = dy; dividing by w is a plausible slip."""
    orig = osch._Segment.g_bwd

    def bad(self, a, grads):
        orig(self, a, grads)
        a[(self.s, "dP")] = [d / self.w for d in a[(self.s, "dP")]]
    monkeypatch.setattr(osch._Segment, "g_bwd", bad)
    assert _caught(FD_FFN)


def test_input_grad_allreduce_drops_a_shard(monkeypatch):
    def bad(self, a):
        du_k = a[(self.s, "du_k")]
        a[(self.s, "du")] = sum(du_k[:-1]) if len(du_k) > 1 else du_k[0]
    monkeypatch.setattr(osch._Segment, "f_bwd", bad)
    assert _caught(FD_FFN)


def test_forward_allreduce_drops_a_shard(monkeypatch):
    orig = osch._Segment.g_fwd

    def bad(self, a):
        P = a[(self.s, "P")]
        a[(self.s, "P")] = P[:-1] if len(P) > 1 else P
        try:
            return orig(self, a)
        finally:
            a[(self.s, "P")] = P
    monkeypatch.setattr(osch._Segment, "g_fwd", bad)
    assert _caught(SHARD)


def test_residual_gradient_dropped(monkeypatch):
    orig = osch._Segment.g_bwd

    def bad(self, a, grads):
        orig(self, a, grads)
        a[(self.s, "dres")] = 0 * a[(self.s, "dy")]
    monkeypatch.setattr(osch._Segment, "g_bwd", bad)
    assert _caught(FD_LAYER)


def test_bias_added_per_shard(monkeypatch):
    """The row-parallel bias is added once after the sum, not once per shard."""
    orig = osch._Segment.g_fwd

    def bad(self, a):
        return orig(self, a) + (self.w - 1) * self.p[self.names["br"]]
    monkeypatch.setattr(osch._Segment, "g_fwd", bad)
    assert _caught(SHARD)


def test_wrong_qkv_head_rows(monkeypatch):
    """Shard k must take the K and V rows of its own heads."""
    orig = osch._Segment.__init__

    def bad(self, *a, **k):
        orig(self, *a, **k)
        if self.kind == "attn" and self.w > 1:
            H = self.shape.hidden
            hw = H // self.w
            self.qkv_rows = [np.r_[kk * hw:(kk + 1) * hw, H + ((kk + 1) % self.w) * hw:
                                   H + ((kk + 1) % self.w + 1) * hw,
                                   2 * H + kk * hw:2 * H + (kk + 1) * hw] for kk in range(self.w)]
    monkeypatch.setattr(osch._Segment, "__init__", bad)
    assert _caught(SHARD)


def test_row_gemm_uses_neighbour_shard_columns(monkeypatch):
    """Shard k must contract with its own K-slice of W2 / Wo."""
    def bad(self, a):
        wr = self.p[self.names["wr"]]
        n = len(self.cols)
        a[(self.s, "P")] = [Hk @ wr[:, self.cols[(k + 1) % n]].T
                            for k, Hk in enumerate(a[(self.s, "H")])]
    monkeypatch.setattr(osch._Segment, "row_fwd", bad)
    assert _caught(SHARD)


def test_selective_recompute_of_attention_drops_the_mask(monkeypatch):
    """A selective recompute that re-runs the attention operation without the
    causal mask: the mode no longer matches "none"."""
    def bad(self, a):
        shape = self.shape
        self.shape = shape.replace(causal=False)
        try:
            a[(self.s, "H")] = [self._attn_shard(q) for q in a[(self.s, "QKV")]]
        finally:
            self.shape = shape
    monkeypatch.setattr(osch._Segment, "attn_fwd", bad)
    assert _caught(lambda: pins.test_recompute_modes_bit_identical("attn"))


def test_gelu_tanh_approximation(monkeypatch):
    """The tanh form of GeLU is a different function (off by up to ~1e-3)."""
    def bad(a):
        return 0.5 * a * (1 + np.tanh(np.sqrt(2 / np.pi) * (a + 0.044715 * a ** 3)))
    monkeypatch.setattr(oops, "gelu", bad)
    assert _caught(pins.test_gelu_against_normal_table)


def test_layer_norm_gamma_gradient_without_normalisation(monkeypatch):
    """dgamma must use xhat = (x - mean) * rstd, not the centred x alone."""
    orig = oops.layer_norm_backward

    def bad(du, x, mean, rstd, gamma):
        dx, _, db = orig(du, x, mean, rstd, gamma)
        return dx, (du * (x - mean[:, None])).sum(0), db
    monkeypatch.setattr(osch, "layer_norm_backward", bad)
    assert _caught(FD_FFN)


def test_attention_backward_without_the_row_term(monkeypatch):
    """dS = P * (dP - rowsum(dP * P)); dropping the row term breaks dQ and dK."""
    import math

    def bad(do, q, k, v, p):
        scale = 1.0 / math.sqrt(q.shape[1])
        dv = p.T @ do
        ds = p * (do @ v.T)
        return (ds @ k) * scale, (ds.T @ q) * scale, dv
    monkeypatch.setattr(osch, "attention_head_backward", bad)
    assert _caught(FD_ATTN)


def test_weight_gradient_overwritten_per_sub_batch(monkeypatch):
    """Gradients of the sub-batches are summed; keeping only the last one is a
    plausible slip (two sub-batches in every tiny shape)."""
    def bad(self, a, grads):
        wr = self.p[self.names["wr"]]
        dH = []
        for Hk, dPk, c in zip(a[(self.s, "H")], a[(self.s, "dP")], self.cols):
            grads[self.names["wr"]][:, c] = dPk.T @ Hk
            dH.append(dPk @ wr[:, c])
        a[(self.s, "dH")] = dH
    monkeypatch.setattr(osch._Segment, "row_bwd", bad)
    assert _caught(FD_FFN, lambda: pins.test_sub_batch_split_invariance("ffn"))


# ---- FP8 E4M3 / MX oracle (oracle/fp8.py) ----
import oracle.fp8 as ofp8
import test_oracle_fp8 as fp8pins


def test_fp8_ties_away_from_zero(monkeypatch):
    orig_pos = ofp8._POS

    def bad(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.minimum(np.abs(x), ofp8.E4M3_MAX)
        hi = np.clip(np.searchsorted(orig_pos, a, side="left"), 0, len(orig_pos) - 1)
        lo = np.maximum(hi - 1, 0)
        code = np.where(orig_pos[hi] - a <= a - orig_pos[lo], hi, lo).astype(np.int64)
        code = np.where(np.signbit(x), code | 0x80, code)
        return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)
    monkeypatch.setattr(ofp8, "e4m3_encode", bad)
    assert _caught(fp8pins.test_ties_go_to_the_even_code)


def test_fp8_overflow_to_nan_instead_of_saturating(monkeypatch):
    orig = ofp8.e4m3_encode

    def bad(x):
        x = np.asarray(x, dtype=np.float64)
        return np.where(np.abs(x) > ofp8.E4M3_MAX, 0x7F, orig(x)).astype(np.uint8)
    monkeypatch.setattr(ofp8, "e4m3_encode", bad)
    assert _caught(fp8pins.test_saturation_and_underflow)


def test_fp8_mx_scale_exponent_off_by_one(monkeypatch):
    monkeypatch.setattr(ofp8, "EMAX_ELEM", 7)
    assert _caught(lambda: fp8pins.test_mx_scale_is_the_block_exponent_minus_8(0))


def test_fp8_mx_gemm_drops_the_b_scale(monkeypatch):
    def bad(A, B, block=32):
        PA, XA = ofp8.mx_quantize(A, block)
        PB, _ = ofp8.mx_quantize(B, block)
        D = np.zeros((A.shape[0], B.shape[0]))
        for b in range((A.shape[1] + block - 1) // block):
            s = slice(b * block, (b + 1) * block)
            D += XA[:, b:b + 1] * (PA[:, s] @ PB[:, s].T)
        return D
    monkeypatch.setattr(ofp8, "mx_gemm", bad)
    assert _caught(fp8pins.test_mx_gemm_exact_on_representable_inputs)
