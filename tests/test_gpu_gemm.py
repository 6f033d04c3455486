"""The GEMM kernels of the block (CUDA-core and tcgen05 tensor-core paths),
every operand layout and epilogue, through oases_debug_gemm, against a float64
product of the same rounded inputs.  Sizes span several tiles with ragged M,
N and K tails."""
import ctypes

import numpy as np
import pytest
import torch

import tensor_model_transformer_tp_gb300 as oz

pytestmark = pytest.mark.gpu

EPI = {"store": 0, "bias": 1, "bias_gelu": 2, "bias_resid": 3, "mul": 4, "accum": 5}


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oz.build_library()
    L = oz.lib()
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    L.oases_debug_gemm.argtypes = [i32, i32, i32, i32, vp, i64, i32, vp, i64, i32, i32, vp, i64,
                                   i32, vp, vp, vp, i64, i32, vp]
    L.oases_debug_gemm.restype = i32
    return L


def _gelu(a):
    from scipy.special import erf
    return 0.5 * a * (1 + erf(a / np.sqrt(2)))


def _gelu_grad(a):
    from scipy.special import erf
    return 0.5 * (1 + erf(a / np.sqrt(2))) + a * np.exp(-0.5 * a * a) / np.sqrt(2 * np.pi)


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def run_case(L, M, N, K, a_k, b_k, epi, dtype, path, seed=0):
    g = torch.Generator().manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    A = torch.randn(M, K, generator=g).to(tdt)
    B = torch.randn(N, K, generator=g).to(tdt)
    bias = torch.randn(N, generator=g).to(tdt)
    aux = torch.randn(M, N, generator=g).to(tdt)
    A_dev = (A if a_k else A.t().contiguous()).cuda()
    B_dev = (B if b_k else B.t().contiguous()).cuda()
    lda = K if a_k else M
    ldb = K if b_k else N
    c_t = torch.float32 if epi == "accum" else tdt
    C0 = torch.randn(M, N, generator=g).to(c_t)
    C = C0.clone().cuda()
    C2 = torch.zeros(M, N, dtype=c_t).cuda() if epi == "bias_gelu" else None
    auxd, biasd = aux.cuda(), bias.cuda()
    st = L.oases_debug_gemm(M, N, K, 1 if dtype == "bf16" else 0, A_dev.data_ptr(), lda, int(a_k),
                            B_dev.data_ptr(), ldb, int(b_k), EPI[epi], C.data_ptr(), N,
                            0 if c_t == torch.float32 else 1,
                            C2.data_ptr() if C2 is not None else None, biasd.data_ptr(),
                            auxd.data_ptr(), N, path, None)
    if st == 2:
        return None
    assert st == 0, st
    torch.cuda.synchronize()
    D = A.double().numpy() @ B.double().numpy().T
    b64, aux64 = bias.double().numpy(), aux.double().numpy()
    ref2 = None
    if epi == "store":
        ref = D
    elif epi == "bias":
        ref = D + b64
    elif epi == "bias_gelu":
        ref2 = _gelu_grad(D + b64)
        ref = _gelu(D + b64)
    elif epi == "bias_resid":
        ref = D + b64 + aux64
    elif epi == "mul":
        ref = D * aux64
    else:
        ref = C0.double().numpy() + D
    out = C.double().cpu().numpy()
    tol = 1e-2 if dtype == "bf16" else 1e-5
    assert rel(out, ref) <= tol, (epi, rel(out, ref))
    if ref2 is not None:
        assert rel(C2.double().cpu().numpy(), ref2) <= tol
    return rel(out, ref)


@pytest.mark.parametrize("a_k,b_k", [(True, True), (True, False), (False, True), (False, False)])
@pytest.mark.parametrize("epi", list(EPI))
def test_tensor_core_gemm_layouts_and_epilogues(L, a_k, b_k, epi):
    # 3 x 3..5 tiles with ragged tails in M, N and K (TMA needs 16-byte row pitches)
    r = run_case(L, 304, 520, 200, a_k, b_k, epi, "bf16", path=2)
    assert r is not None, "tensor-core path refused a supported case"


# 4736 rows = 19 pair row blocks.  K = 192: A is small, tiles run row block
# fastest over all 19 (x 9 column blocks = 171 tiles, several per CTA pair).
# K = 5376: A is 51 MB, tiles run in row-block groups of 8, 8 and 3 (x 7
# column blocks, the last one 8 columns wide).
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (8, 8, 8), (264, 136, 1000), (2048, 1024, 512),
                                   (4736, 2304, 192), (4736, 1544, 5376)])
def test_tensor_core_gemm_shapes(L, M, N, K):
    assert run_case(L, M, N, K, True, True, "bias", "bf16", path=2) is not None
    assert run_case(L, M, N, K, False, False, "accum", "bf16", path=2) is not None


@pytest.mark.parametrize("epi", list(EPI))
def test_simt_gemm_fp32(L, epi):
    run_case(L, 130, 70, 33, False, True, epi, "f32", path=1)
    run_case(L, 65, 129, 300, True, False, epi, "f32", path=1)


def test_tensor_core_matches_simt_bf16(L):
    """Same bf16 operands: both kernels agree to fp32 accumulation-order noise."""
    g = torch.Generator().manual_seed(3)
    M, N, K = 256, 384, 320
    A = torch.randn(M, K, generator=g).bfloat16().cuda()
    B = torch.randn(N, K, generator=g).bfloat16().cuda()
    outs = []
    for path in (1, 2):
        C = torch.zeros(M, N, dtype=torch.float32, device="cuda")
        assert L.oases_debug_gemm(M, N, K, 1, A.data_ptr(), K, 1, B.data_ptr(), K, 1, 0,
                                  C.data_ptr(), N, 0, None, None, None, 0, path, None) == 0
        outs.append(C)
    torch.cuda.synchronize()
    assert rel(outs[1].double().cpu().numpy(), outs[0].double().cpu().numpy()) < 1e-5


def test_no_timeout_recorded(L):
    oz.oases_check_device(None)


def test_gelu_accuracy_against_float64(L):
    """GeLU and GeLU' of the epilogue (erf via Abramowitz & Stegun 7.1.26,
    |error| <= 1.5e-7) against float64, through an fp32 K=1 product C = a * 1."""
    from scipy.special import erf
    a = np.concatenate([np.linspace(-9, 9, 4001), np.random.default_rng(0).normal(0, 2, 4000)])
    M = a.size
    A = torch.tensor(a, dtype=torch.float32).reshape(M, 1).cuda()
    B = torch.ones(1, 1, dtype=torch.float32, device="cuda")
    bias = torch.zeros(1, dtype=torch.float32, device="cuda")
    a32 = A.double().cpu().numpy()[:, 0]
    cdf = 0.5 * (1 + erf(a32 / np.sqrt(2)))
    pdf = np.exp(-0.5 * a32 * a32) / np.sqrt(2 * np.pi)
    C = torch.zeros(M, 1, dtype=torch.float32, device="cuda")
    D = torch.zeros(M, 1, dtype=torch.float32, device="cuda")
    # C = gelu(a), D = gelu'(a) from one bias + GeLU epilogue with its derivative output
    assert L.oases_debug_gemm(M, 1, 1, 0, A.data_ptr(), 1, 1, B.data_ptr(), 1, 1, 2, C.data_ptr(), 1,
                              0, D.data_ptr(), bias.data_ptr(), None, 0, 1, None) == 0
    torch.cuda.synchronize()
    g = C.double().cpu().numpy()[:, 0]
    d = D.double().cpu().numpy()[:, 0]
    assert np.max(np.abs(g - a32 * cdf)) <= 1e-6 * np.maximum(1, np.abs(a32)).max()
    assert np.max(np.abs(g - a32 * cdf) / np.maximum(1, np.abs(a32))) <= 3e-7
    assert np.max(np.abs(d - (cdf + a32 * pdf)) / np.maximum(1, np.abs(a32))) <= 4e-7
