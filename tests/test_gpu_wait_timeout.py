"""Failure detection on the GPU without a fault: a bounded wait that runs out.

oases_debug_wait_probe launches one thread that waits, with the bounded
mbarrier wait every tensor-core kernel of the library uses, on a barrier that
nothing arrives on.  The wait must give up after its limit (a few
milliseconds here), record its site, and leave the CUDA context usable: the
next oases_check_device reports OASES_ERR_TIMEOUT once, the error word is
cleared by reading it, and a kernel launched afterwards computes correctly.
"""
import ctypes
import time

import pytest
import torch

import tensor_model_transformer_tp_gb300 as oz

pytestmark = pytest.mark.gpu

OASES_ERR_INVALID_ARG, OASES_ERR_TIMEOUT = 1, 5


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oz.build_library()
    L = oz.lib()
    L.oases_debug_wait_probe.argtypes = [ctypes.c_uint64, ctypes.c_void_p]
    L.oases_debug_wait_probe.restype = ctypes.c_int
    L.oases_check_device.argtypes = [ctypes.c_void_p]
    L.oases_check_device.restype = ctypes.c_int
    L.oases_debug_attention_error_word.restype = ctypes.c_int
    return L


def test_wait_runs_out_and_the_context_stays_usable(L):
    assert L.oases_check_device(None) == 0           # nothing pending before
    t0 = time.perf_counter()
    assert L.oases_debug_wait_probe(1 << 22, None) == 0
    assert L.oases_check_device(None) == OASES_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0            # the wait gave up by itself
    assert L.oases_check_device(None) == 0           # reported once, then cleared
    # the same through the error word: site 999
    assert L.oases_debug_wait_probe(1 << 20, None) == 0
    torch.cuda.synchronize()
    assert L.oases_debug_attention_error_word() == 999
    assert L.oases_debug_attention_error_word() == 0
    # the context still computes
    a = torch.randn(256, 256, device="cuda")
    assert torch.allclose(a @ torch.eye(256, device="cuda"), a)
    assert L.oases_check_device(None) == 0


def test_out_of_range_limit_is_refused_before_launch(L):
    assert L.oases_debug_wait_probe(0, None) == OASES_ERR_INVALID_ARG
    assert L.oases_debug_wait_probe((1 << 32) + 1, None) == OASES_ERR_INVALID_ARG
    assert L.oases_check_device(None) == 0
