"""Kernel-level entry points (include/oases_debug.h) other than the GEMM,
against float64 numpy on the same inputs."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tensor_model_transformer_tp_gb300 as oz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oz.build_library()
    L = oz.lib()
    L.oases_debug_bias_grad_scratch_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    L.oases_debug_bias_grad_scratch_bytes.restype = ctypes.c_size_t
    L.oases_debug_bias_grad.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_size_t, ctypes.c_void_p]
    L.oases_debug_bias_grad.restype = ctypes.c_int
    return L


# (2200000, 8) and (2100000, 3): more partial rows of 32 (68750, 65625) than one
# grid dimension holds (65535), on the vector and the scalar kernel
@pytest.mark.parametrize("M,N,ld,dtype", [(1, 1, 1, "f32"), (33, 70, 75, "f32"), (2048, 4096, 4096, "bf16"),
                                          (100, 1030, 1030, "bf16"), (0, 16, 16, "bf16"),
                                          (2200000, 8, 8, "bf16"), (2100000, 3, 3, "f32"),
                                          (1000, 12, 12, "f32"), (64, 40, 40, "bf16")])
def test_bias_grad(L, M, N, ld, dtype):
    g = torch.Generator().manual_seed(M + N)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = torch.randn(M, ld, generator=g).to(tdt)
    out0 = torch.randn(N, generator=g)
    out = out0.cuda()
    nb = L.oases_debug_bias_grad_scratch_bytes(M, N)
    scratch = torch.empty(max(nb, 4), dtype=torch.uint8, device="cuda")
    xd = x.cuda()
    st = L.oases_debug_bias_grad(xd.data_ptr() if M else None, ld, M, N, 1 if dtype == "bf16" else 0,
                                 out.data_ptr(), scratch.data_ptr(), nb, None)
    assert st == 0
    torch.cuda.synchronize()
    ref = out0.double().numpy() + x.double().numpy()[:, :N].sum(axis=0)
    np.testing.assert_allclose(out.double().cpu().numpy(), ref, rtol=1e-5, atol=1e-4)
    # scratch too small is refused before any launch
    if nb > 4:
        assert L.oases_debug_bias_grad(xd.data_ptr(), ld, M, N, 1 if dtype == "bf16" else 0,
                                       out.data_ptr(), scratch.data_ptr(), nb - 4, None) == 3


# ---- LayerNorm forward / backward and the shard sum, against the oracle ----

def _bind(L):
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    L.oases_debug_layer_norm.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, f32, i32, vp]
    L.oases_debug_layer_norm.restype = i32
    L.oases_debug_layer_norm_bwd_scratch_bytes.argtypes = [i32, i32]
    L.oases_debug_layer_norm_bwd_scratch_bytes.restype = sz
    L.oases_debug_layer_norm_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, sz, vp]
    L.oases_debug_layer_norm_bwd.restype = i32
    L.oases_debug_shard_sum.argtypes = [vp, i64, i32, vp, vp, vp, i32, i32, i32, vp]
    L.oases_debug_shard_sum.restype = i32
    return L


def _p(t):
    return t.data_ptr() if t is not None and t.numel() else None


def _np(t):
    return t.detach().double().cpu().numpy()


def _close(got, ref, dtype, scale=1.0):
    """bf16 outputs: within one bf16 rounding (2^-8 relative, with a floor at
    the data's scale) element by element, and rel-L2 <= 2e-2; fp32: 1e-5."""
    if dtype == "bf16":
        np.testing.assert_allclose(got, ref, rtol=2.0 ** -7, atol=2.0 ** -9 * scale)
        tol = 2e-2
    else:
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6 * scale)
        tol = 1e-5
    if ref.size:
        assert np.linalg.norm(got - ref) <= tol * max(np.linalg.norm(ref), 1e-30)


LN_CASES = [(1, 256, "bf16"), (37, 1024, "bf16"), (129, 2560, "bf16"), (50, 296, "bf16"),
            (33, 200, "f32"), (2048, 1024, "bf16"), (0, 256, "bf16")]


@pytest.mark.parametrize("M,H,dtype", LN_CASES)
def test_layer_norm_forward(L, M, H, dtype):
    L = _bind(L)
    g = torch.Generator().manual_seed(7 * M + H)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = (torch.randn(M, H, generator=g) * 3 + 0.5).to(tdt)
    gamma = (1 + 0.1 * torch.randn(H, generator=g)).to(tdt)
    beta = (0.1 * torch.randn(H, generator=g)).to(tdt)
    xd, gd, bd = x.cuda(), gamma.cuda(), beta.cuda()
    u = torch.empty_like(xd)
    mean = torch.empty(M, device="cuda")
    rstd = torch.empty(M, device="cuda")
    st = L.oases_debug_layer_norm(_p(xd), _p(gd), _p(bd), _p(u), _p(mean), _p(rstd), M, H, 1e-5,
                                  1 if dtype == "bf16" else 0, None)
    assert st == 0
    torch.cuda.synchronize()
    if M == 0:
        return
    ru, rmean, rrstd = oracle.ops.layer_norm(_np(x), _np(gamma), _np(beta), 1e-5)
    np.testing.assert_allclose(_np(mean), rmean, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(_np(rstd), rrstd, rtol=1e-5)
    _close(_np(u), ru, dtype)


# 4-column chunks per thread 1 (H <= 1024), 2, 3 and 4 (H <= 4096), H % 4 != 0
# (scalar kernels), H > 4096 (two-phase kernel), ragged row blocks, M = 0
LN_BWD_CASES = [(37, 1024, "bf16", True), (9, 256, "f32", False), (50, 302, "bf16", True),
                (1, 2560, "bf16", False), (4096, 4096, "bf16", True), (0, 256, "f32", True),
                (13, 1028, "bf16", True), (19, 4096, "f32", True), (5, 5120, "bf16", True)]


@pytest.mark.parametrize("M,H,dtype,resid", LN_BWD_CASES)
def test_layer_norm_backward(L, M, H, dtype, resid):
    L = _bind(L)
    g = torch.Generator().manual_seed(11 * M + H)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = (torch.randn(M, H, generator=g) * 2 - 0.3).to(tdt)
    gamma = (1 + 0.1 * torch.randn(H, generator=g)).to(tdt)
    du = torch.randn(M, H, generator=g)
    dres = torch.randn(M, H, generator=g).to(tdt) if resid else None
    dg0, db0 = torch.randn(H, generator=g), torch.randn(H, generator=g)
    # the forward's statistics, from the oracle (fp64) rounded to fp32 as the kernel takes them
    _, mean64, rstd64 = oracle.ops.layer_norm(_np(x), np.ones(H), np.zeros(H), 1e-5) if M else (0, np.zeros(0), np.zeros(0))
    mean = torch.from_numpy(mean64).float()
    rstd = torch.from_numpy(rstd64).float()
    dev = [t.cuda() if t is not None else None for t in (x, gamma, du, dres, mean, rstd)]
    xd, gd, dud, dresd, md, rd = dev
    dx = torch.empty_like(xd)
    nb = L.oases_debug_layer_norm_bwd_scratch_bytes(M, H)
    scratch = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")

    def run(dgamma, dbeta):
        return L.oases_debug_layer_norm_bwd(_p(dud), _p(xd), _p(md), _p(rd), _p(gd), _p(dresd), _p(dx),
                                            _p(dgamma), _p(dbeta), M, H, 1 if dtype == "bf16" else 0,
                                            _p(scratch), nb, None)

    dgamma, dbeta = dg0.cuda(), db0.cuda()
    assert run(dgamma, dbeta) == 0
    torch.cuda.synchronize()
    if M == 0:
        assert torch.equal(dgamma.cpu(), dg0) and torch.equal(dbeta.cpu(), db0)
        return
    rdx, rdg, rdb = oracle.ops.layer_norm_backward(_np(du), _np(x), _np(mean), _np(rstd), _np(gamma))
    if resid:
        rdx = rdx + _np(dres)
    _close(_np(dx), rdx, dtype, scale=float(np.abs(rdx).max()))
    s = float(np.sqrt(M))
    np.testing.assert_allclose(_np(dgamma), _np(dg0) + rdg, rtol=1e-4, atol=1e-4 * s)
    np.testing.assert_allclose(_np(dbeta), _np(db0) + rdb, rtol=1e-4, atol=1e-4 * s)
    # the parameter-gradient sums take a fixed order: bit-identical on a second call
    dgamma2, dbeta2 = dg0.cuda(), db0.cuda()
    assert run(dgamma2, dbeta2) == 0
    torch.cuda.synchronize()
    assert torch.equal(dgamma, dgamma2) and torch.equal(dbeta, dbeta2)
    # too small a scratch is refused before anything is enqueued
    assert L.oases_debug_layer_norm_bwd(_p(dud), _p(xd), _p(md), _p(rd), _p(gd), _p(dresd), _p(dx),
                                        _p(dgamma), _p(dbeta), M, H, 1 if dtype == "bf16" else 0,
                                        _p(scratch), nb - 16, None) == 3


@pytest.mark.parametrize("M,N,w,dtype,bias,resid", [
    (2048, 1024, 4, "bf16", True, True), (37, 100, 8, "bf16", True, False),
    (5, 7, 3, "bf16", False, True), (33, 64, 1, "f32", True, True), (17, 30, 2, "f32", False, False),
    (0, 64, 4, "bf16", True, True)])
def test_shard_sum(L, M, N, w, dtype, bias, resid):
    L = _bind(L)
    g = torch.Generator().manual_seed(M * N + w)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    pstride = M * N + 12  # slabs need not be packed
    part = torch.randn(w * pstride, generator=g)
    b = torch.randn(N, generator=g).to(tdt) if bias else None
    r = torch.randn(M, N, generator=g).to(tdt) if resid else None
    partd = part.cuda()
    bd = b.cuda() if bias else None
    rd = r.cuda() if resid else None
    out = torch.zeros(M, N, dtype=tdt, device="cuda")
    st = L.oases_debug_shard_sum(_p(partd), pstride, w, _p(bd), _p(rd), _p(out), M, N,
                                 1 if dtype == "bf16" else 0, None)
    assert st == 0
    torch.cuda.synchronize()
    if M == 0:
        return
    p64 = part.double().numpy()
    ref = sum(p64[k * pstride:k * pstride + M * N].reshape(M, N) for k in range(w))
    if bias:
        ref = ref + _np(b)[None, :]
    if resid:
        ref = ref + _np(r)
    _close(_np(out), ref, dtype, scale=float(np.abs(ref).max()))


def test_kernel_entries_refuse_misaligned_pointers(L):
    L = _bind(L)
    buf = torch.zeros(4096, device="cuda")
    base = buf.data_ptr()
    # an 8-byte offset breaks the 16-byte rule: refused before any launch
    assert L.oases_debug_layer_norm(base + 8, base, base, base + 1024, base + 2048, base + 3072,
                                    2, 256, 1e-5, 1, None) == 1
    assert L.oases_debug_shard_sum(base + 4, 64, 1, None, None, base + 8192, 4, 16, 0, None) == 1
