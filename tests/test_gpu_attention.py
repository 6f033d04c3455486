"""Attention kernels (oases_debug_attention): tensor-core forward against the
CUDA-core forward and against float64 numpy; backward against float64 numpy.
Sequences are ragged against the 128-row tiles."""
import ctypes

import numpy as np
import pytest
import torch

import tensor_model_transformer_tp_gb300 as oz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oz.build_library()
    L = oz.lib()
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    L.oases_debug_attention.argtypes = [vp, vp, vp, vp, vp, vp] + [i32] * 8 + [vp]
    L.oases_debug_attention.restype = i32
    return L


def ref_attention(qkv, B, S, nh, d, causal, d_o=None):
    H = nh * d
    q = qkv[:, :H].reshape(B, S, nh, d).transpose(0, 2, 1, 3)
    k = qkv[:, H:2 * H].reshape(B, S, nh, d).transpose(0, 2, 1, 3)
    v = qkv[:, 2 * H:].reshape(B, S, nh, d).transpose(0, 2, 1, 3)
    s = q @ k.transpose(0, 1, 3, 2) / np.sqrt(d)
    if causal:
        s = np.where(np.tril(np.ones((S, S), bool)), s, -np.inf)
    mx = s.max(-1, keepdims=True)
    p = np.exp(s - mx)
    l = p.sum(-1, keepdims=True)
    lse = (mx + np.log(l))[..., 0]            # [B, nh, S]
    p = p / l
    o = p @ v
    out = {"o": o.transpose(0, 2, 1, 3).reshape(B * S, H),
           "lse": lse.transpose(1, 0, 2).reshape(nh, B * S)}
    if d_o is not None:
        do = d_o.reshape(B, S, nh, d).transpose(0, 2, 1, 3)
        dv = p.transpose(0, 1, 3, 2) @ do
        dp = do @ v.transpose(0, 1, 3, 2)
        ds = p * (dp - (dp * p).sum(-1, keepdims=True))
        dq = ds @ k / np.sqrt(d)
        dk = ds.transpose(0, 1, 3, 2) @ q / np.sqrt(d)
        g = lambda t: t.transpose(0, 2, 1, 3).reshape(B * S, H)
        out["dqkv"] = np.concatenate([g(dq), g(dk), g(dv)], axis=1)
    return out


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def run(L, qkv, B, S, nh, d, causal, path, d_o=None):
    M, H = B * S, nh * d
    o = torch.zeros(M, H, dtype=qkv.dtype, device="cuda")
    lse = torch.zeros(nh, M, dtype=torch.float32, device="cuda")
    dt = 1 if qkv.dtype == torch.bfloat16 else 0
    st = L.oases_debug_attention(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), None, None, None,
                                 B, S, nh, d, int(causal), dt, 0, path, None)
    assert st == 0, st
    res = {"o": o, "lse": lse}
    if d_o is not None:
        delta = torch.zeros(nh, M, dtype=torch.float32, device="cuda")
        dqkv = torch.zeros(M, 3 * H, dtype=qkv.dtype, device="cuda")
        st = L.oases_debug_attention(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     d_o.data_ptr(), delta.data_ptr(), dqkv.data_ptr(), B, S, nh,
                                     d, int(causal), dt, 1, path, None)
        assert st == 0, st
        res["dqkv"] = dqkv
    torch.cuda.synchronize()
    oz.oases_check_device(None)
    return {k: v.double().cpu().numpy() for k, v in res.items()}


@pytest.mark.parametrize("B,S,nh,causal", [(1, 128, 1, True), (2, 200, 2, True), (1, 77, 3, True),
                                           (2, 256, 2, False), (1, 1, 1, True), (1, 300, 1, False)])
def test_tc_forward(L, B, S, nh, causal):
    d = 128
    g = torch.Generator().manual_seed(S + nh)
    qkv = (torch.randn(B * S, 3 * nh * d, generator=g) * 1.5).bfloat16()
    ref = ref_attention(qkv.double().numpy(), B, S, nh, d, causal)
    tc = run(L, qkv.cuda(), B, S, nh, d, causal, path=2)
    simt = run(L, qkv.cuda(), B, S, nh, d, causal, path=1)
    assert rel(tc["o"], ref["o"]) < 1e-2
    assert rel(tc["lse"], ref["lse"]) < 1e-3
    assert rel(tc["o"], simt["o"]) < 1e-2
    assert np.all(np.isfinite(tc["o"]))


@pytest.mark.parametrize("B,S,nh,causal", [(2, 200, 2, True), (1, 128, 1, False), (1, 77, 3, True),
                                           (2, 300, 1, False), (1, 1, 1, True), (1, 320, 2, True)])
def test_backward(L, B, S, nh, causal):
    d = 128
    g = torch.Generator().manual_seed(11 + S)
    qkv = torch.randn(B * S, 3 * nh * d, generator=g).bfloat16()
    d_o = torch.randn(B * S, nh * d, generator=g).bfloat16()
    ref = ref_attention(qkv.double().numpy(), B, S, nh, d, causal, d_o.double().numpy())
    got = run(L, qkv.cuda(), B, S, nh, d, causal, path=0, d_o=d_o.cuda())
    H = nh * d
    scale = np.linalg.norm(ref["dqkv"])
    for part, sl in (("dq", slice(0, H)), ("dk", slice(H, 2 * H)), ("dv", slice(2 * H, 3 * H))):
        a, b = got["dqkv"][:, sl], ref["dqkv"][:, sl]
        if np.linalg.norm(b) < 1e-9 * scale:
            # exactly zero in exact arithmetic (one-token sequences: dS = P (dP - delta) = 0)
            assert np.linalg.norm(a) <= 1e-4 * scale, part
        else:
            assert rel(a, b) < 2e-2, part


def test_tc_backward_matches_cuda_core_backward(L):
    B, S, nh, d = 2, 192, 2, 128
    g = torch.Generator().manual_seed(5)
    qkv = torch.randn(B * S, 3 * nh * d, generator=g).bfloat16().cuda()
    d_o = torch.randn(B * S, nh * d, generator=g).bfloat16().cuda()
    tc = run(L, qkv, B, S, nh, d, True, path=0, d_o=d_o)
    simt = run(L, qkv, B, S, nh, d, True, path=1, d_o=d_o)
    assert rel(tc["dqkv"], simt["dqkv"]) < 1e-2


def test_results_do_not_depend_on_the_item_order(L):
    """The persistent kernels hand out work items by a schedule: the forward
    by the host's longest-first order up to 2048 items (a snake order over
    rounds of CTAs beyond), the dQ kernel by the snake order.  16 sequences x
    20 heads (2560 forward items, 5120 dQ items) against the same sequences
    as two calls of 8 (1280 forward items each, the host's order): every
    output bit-identical, since no item's arithmetic depends on which CTA
    runs it or when."""
    B, S, nh, d = 16, 2048, 20, 128
    H = nh * d

    def call(qkv, d_o, b):
        M = b * S
        o = torch.zeros(M, H, dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros(nh, M, dtype=torch.float32, device="cuda")
        delta = torch.zeros(nh, M, dtype=torch.float32, device="cuda")
        dqkv = torch.zeros(M, 3 * H, dtype=torch.bfloat16, device="cuda")
        assert L.oases_debug_attention(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), None, None, None,
                                       b, S, nh, d, 1, 1, 0, 2, None) == 0
        assert L.oases_debug_attention(qkv.data_ptr(), o.data_ptr(), lse.data_ptr(), d_o.data_ptr(),
                                       delta.data_ptr(), dqkv.data_ptr(), b, S, nh, d, 1, 1, 1, 2,
                                       None) == 0
        torch.cuda.synchronize()
        oz.oases_check_device(None)
        return o, lse, dqkv

    g = torch.Generator(device="cuda").manual_seed(7)
    qkv = (torch.randn(B * S, 3 * H, generator=g, device="cuda") * 1.5).bfloat16()
    d_o = torch.randn(B * S, H, generator=g, device="cuda").bfloat16()
    o, lse, dqkv = call(qkv, d_o, B)
    half = B * S // 2
    for k, r in enumerate((0, half)):
        o2, lse2, dqkv2 = call(qkv[r:r + half].contiguous(), d_o[r:r + half].contiguous(), B // 2)
        assert torch.equal(o[r:r + half], o2)
        assert torch.equal(lse[:, r:r + half], lse2)
        assert torch.equal(dqkv[r:r + half], dqkv2)
    assert bool(torch.isfinite(dqkv.float()).all())
