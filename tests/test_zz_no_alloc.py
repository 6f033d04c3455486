"""oases_bias_grad_noalloc: the bias-gradient sum for callers that cannot
allocate device memory (a plugin in a framework that owns all device memory, a
real-time loop that cannot afford cudaMalloc's implicit synchronisation).  Its
scratch is a static device array inside the library.

This file is collected last on purpose.  It checks, through the C ABI, that
the entry point gives the same result as oases_debug_bias_grad (which takes
caller-owned scratch) on two calls in a row, that both agree with the column
sums taken in float64 on the host, that a narrow input with more partial rows
than a grid dimension allows is still summed, and that a size whose partial
rows do not fit the static array is refused.  It passes alone in a fresh
process and after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import tensor_model_transformer_tp_gb300 as oz

pytestmark = pytest.mark.gpu

NOALLOC_FLOATS = 1 << 20


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oz.build_library()
    L = oz.lib()
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.oases_debug_bias_grad_scratch_bytes.argtypes = [i32, i32]
    L.oases_debug_bias_grad_scratch_bytes.restype = ctypes.c_size_t
    L.oases_debug_bias_grad.argtypes = [vp, i64, i32, i32, i32, vp, vp, ctypes.c_size_t, vp]
    L.oases_debug_bias_grad.restype = i32
    L.oases_bias_grad_noalloc.argtypes = [vp, i64, i32, i32, i32, vp, vp]
    L.oases_bias_grad_noalloc.restype = i32
    return L


def test_noalloc_matches_scratch_entry_point_twice(L):
    M, N = 2048, 512           # ceil(2048/32) * 512 = 32768 partial floats
    gen = torch.Generator().manual_seed(7)
    stream = torch.cuda.current_stream().cuda_stream
    init = torch.randn(N, generator=gen)
    out_ref = init.clone().cuda()
    out_new = init.clone().cuda()
    nb = L.oases_debug_bias_grad_scratch_bytes(M, N)
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    expect = None
    for call in range(2):     # the second call sees the array the first one left
        x = torch.randn(M, N, generator=gen).to(torch.bfloat16).cuda()
        assert L.oases_debug_bias_grad(x.data_ptr(), N, M, N, 1, out_ref.data_ptr(),
                                       scratch.data_ptr(), nb, stream) == 0
        assert L.oases_bias_grad_noalloc(x.data_ptr(), N, M, N, 1, out_new.data_ptr(),
                                         stream) == 0
        torch.cuda.synchronize()
        a = out_new.double().cpu().numpy()
        b = out_ref.double().cpu().numpy()
        np.testing.assert_allclose(a, b, rtol=1e-6, atol=0), call
        np.testing.assert_array_equal(a, b)   # same kernels, same summation order
        # the plain definition: out += sum over rows, in float64 on the host
        expect = expect + x.double().cpu().numpy().sum(axis=0) if call else \
            init.double().numpy() + x.double().cpu().numpy().sum(axis=0)
        scale = np.abs(x.double().cpu().numpy()).sum(axis=0) + np.abs(expect)
        assert np.all(np.abs(a - expect) <= 1e-5 * scale), call


def test_noalloc_narrow_input_with_many_partial_rows(L):
    """N = 4 columns, 2.2 million rows: 68750 partial rows of 32, more than one
    grid dimension holds (65535), within the static array (275000 floats)."""
    M, N = 2200000, 4
    gen = torch.Generator().manual_seed(8)
    xh = torch.randn(M, N, generator=gen).to(torch.bfloat16)
    x = xh.cuda()
    out = torch.zeros(N, device="cuda")
    assert L.oases_bias_grad_noalloc(x.data_ptr(), N, M, N, 1, out.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    expect = xh.double().numpy().sum(axis=0)
    scale = np.abs(xh.double().numpy()).sum(axis=0)
    assert np.all(np.abs(out.double().cpu().numpy() - expect) <= 1e-5 * scale)


def test_noalloc_rejects_sizes_beyond_the_array(L):
    N = 4096
    M = 32 * (NOALLOC_FLOATS // N) + 1    # one 32-row partial row too many
    out = torch.zeros(N, device="cuda")
    x = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    st = L.oases_bias_grad_noalloc(x.data_ptr(), N, M, N, 1, out.data_ptr(), None)
    assert st == 2
    assert "scratch floats" in oz.lib().oases_last_error().decode()
    assert torch.count_nonzero(out).item() == 0
