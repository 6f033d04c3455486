"""Kernel-level entry points (include/oases_debug.h) other than the GEMM,
against float64 numpy on the same inputs."""
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
    L.oases_debug_bias_grad_scratch_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    L.oases_debug_bias_grad_scratch_bytes.restype = ctypes.c_size_t
    L.oases_debug_bias_grad.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_size_t, ctypes.c_void_p]
    L.oases_debug_bias_grad.restype = ctypes.c_int
    return L


@pytest.mark.parametrize("M,N,ld,dtype", [(1, 1, 1, "f32"), (33, 70, 75, "f32"), (2048, 4096, 4096, "bf16"),
                                          (100, 1030, 1030, "bf16"), (0, 16, 16, "bf16")])
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
