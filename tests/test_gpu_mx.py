"""The MX-FP8 GEMM variant (E4M3 elements, UE8M0 block-32 scales) through the
C ABI (oases_mx.h), against the oracle of the format (oracle/fp8.py, which
restates the OCP MX v1.0 and E4M3 definitions).

* Quantisation is integer work: the E4M3 codes and the scale bytes of the
  CUDA quantiser must equal the oracle's bit for bit, row-wise and transposed,
  on ragged sizes, with all-zero blocks, tiny values and values that saturate.
* The GEMM: the MX product of the oracle is exact (float64); the kernel sums
  the same products in fp32.  Each output element must lie within the bound on
  fp32 summation of K terms in any order, |D - D_exact| <= g_K * sum |terms|
  with g_K = K u / (1 - K u), u = 2^-24 (Higham, Accuracy and Stability of
  Numerical Algorithms, §3.1), where sum |terms| is taken over the products
  X_A X_B P_A P_B.  Epilogues are checked against the plain definition applied
  to the oracle's product, within their own rounding (bf16 outputs: 2^-8
  relative, as the bf16 GEMM tests).
* Structured probes pin which scale the hardware applies to which row and K
  block: with all elements 1.0 and K = 128, the output is a sum of the four
  block scales of the row (and of the column), so a wrong tile layout shows up
  as a wrong power of two.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle.fp8 as fp8
import tensor_model_transformer_tp_gb300 as oz

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oz.build_library()
    L = oz.lib()
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.oases_mx_scale_bytes.argtypes = [i32, i32]
    L.oases_mx_scale_bytes.restype = sz
    L.oases_mx_quantize.argtypes = [vp, i64, i32, i32, i32, i32, vp, i64, vp, vp]
    L.oases_mx_quantize.restype = i32
    L.oases_mx_gemm.argtypes = [i32, i32, i32, vp, i64, vp, vp, i64, vp, i32, vp, i64, i32, vp, vp,
                                vp, i64, vp]
    L.oases_mx_gemm.restype = i32
    return L


def ldq_for(K):
    return (K + 15) // 16 * 16


def quantize(L, x_dev, rows, K, transpose, dtype):
    """MX operand of x (device tensor) through the C ABI: (codes [rows, ldq] uint8
    device tensor, scales device tensor)."""
    ldq = ldq_for(K)
    q = torch.zeros(rows, ldq, dtype=torch.uint8, device="cuda")
    sf = torch.full((max(1, L.oases_mx_scale_bytes(rows, K)),), 0xEE, dtype=torch.uint8,
                    device="cuda")
    ld = x_dev.shape[1]
    st = L.oases_mx_quantize(x_dev.data_ptr(), ld, rows, K, 1 if dtype == "bf16" else 0,
                             transpose, q.data_ptr(), ldq, sf.data_ptr(), None)
    assert st == 0, st
    return q, sf


def scales_from_tiles(sf, rows, K):
    """[rows, ceil(K/32)] scale bytes read back from the tile layout."""
    kg = (K + 127) // 128
    nb = (K + 31) // 32
    out = np.zeros((rows, nb), dtype=np.int64)
    for r in range(rows):
        for j in range(nb):
            off = ((r // 128) * kg + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4
            out[r, j] = sf[off]
    return out


def padding_scale_bytes(sf, rows, K):
    """Every tile byte that belongs to no (row, block) of the matrix."""
    kg = (K + 127) // 128
    nb = (K + 31) // 32
    used = np.zeros(sf.shape[0], dtype=bool)
    for r in range(rows):
        for j in range(nb):
            used[((r // 128) * kg + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4] = True
    return sf[~used]


def oracle_operand(v):
    """Oracle E4M3 codes and scale bytes of v [rows, K] (float64 values)."""
    P, X = fp8.mx_quantize(v)
    return fp8.e4m3_encode(P).astype(np.int64), (np.log2(X).astype(np.int64) + 127)


def special_matrix(rows, K, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, K, generator=g)
    x[0, :min(32, K)] = 0.0                                   # an all-zero block
    if rows > 1:
        x[1, :] *= 1e-30                                      # tiny values (scales near 2^-100)
    if rows > 2:
        x[2, :] *= 1e30                                       # huge values
    if rows > 3 and K > 40:
        x[3, 33] = 1e4                                        # one block dominated by one value
    if rows > 4:
        x[4, :] = torch.randint(-3, 4, (K,), generator=g).float() * 0.25   # exact values
    if rows > 5:
        # with 464 in every block, X = 1: 464 saturates to 448, the others are
        # halfway between two E4M3 values (ties to the even code), 2^-10 is half
        # the smallest subnormal, 7.5 * 2^-9 the subnormal / normal midpoint
        pat = torch.tensor([464.0, 1.0625, 1.1875, 17.0, -17.0, 2.0 ** -10, 7.5 * 2.0 ** -9, -1.0625])
        x[5, :] = pat.repeat(K // 8 + 1)[:K]
        for b in range(0, K, 32):
            x[5, b] = 464.0
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return x.to(tdt)


@pytest.mark.parametrize("rows,K,dtype", [(200, 96, "bf16"), (130, 320, "bf16"), (64, 77, "f32"),
                                          (257, 1000, "bf16"), (1, 31, "f32")])
def test_quantize_rows_bit_exact(L, rows, K, dtype):
    x = special_matrix(rows, K, seed=rows + K, dtype=dtype)
    q, sf = quantize(L, x.cuda(), rows, K, 0, dtype)
    torch.cuda.synchronize()
    codes, scales = oracle_operand(x.double().numpy())
    np.testing.assert_array_equal(q.cpu().numpy()[:, :K].astype(np.int64), codes)
    sfh = sf.cpu().numpy()
    np.testing.assert_array_equal(scales_from_tiles(sfh, rows, K), scales)
    assert np.all(padding_scale_bytes(sfh, rows, K) == 127)


@pytest.mark.parametrize("rows,K,dtype", [(200, 96, "bf16"), (96, 130, "f32"), (300, 512, "bf16")])
def test_quantize_transposed_bit_exact(L, rows, K, dtype):
    """transpose = 1: x is [K, rows]; the operand is x^T, blocks along x's rows."""
    xt = special_matrix(rows, K, seed=7 * rows + K, dtype=dtype)   # the operand [rows, K]
    x = xt.t().contiguous()                                          # what the caller holds
    q, sf = quantize(L, x.cuda(), rows, K, 1, dtype)
    torch.cuda.synchronize()
    codes, scales = oracle_operand(xt.double().numpy())
    np.testing.assert_array_equal(q.cpu().numpy()[:, :K].astype(np.int64), codes)
    np.testing.assert_array_equal(scales_from_tiles(sf.cpu().numpy(), rows, K), scales)


def mx_gemm_dev(L, qa, sfa, qb, sfb, M, N, K, epi=0, c_dtype="f32", C=None, C2=None, bias=None,
                aux=None):
    tdt = torch.float32 if c_dtype == "f32" else torch.bfloat16
    if C is None:
        C = torch.zeros(M, N, dtype=tdt, device="cuda")
    p = lambda t: t.data_ptr() if t is not None else None
    st = L.oases_mx_gemm(M, N, K, qa.data_ptr(), qa.shape[1], sfa.data_ptr(), qb.data_ptr(),
                         qb.shape[1], sfb.data_ptr(), epi, C.data_ptr(), N,
                         0 if c_dtype == "f32" else 1, p(C2), p(bias), p(aux),
                         N if aux is not None else 0, None)
    assert st == 0, st
    return C


def exact_and_abs(A, B):
    """The oracle's MX product and sum |terms| per element (float64)."""
    PA, XA = fp8.mx_quantize(A)
    PB, XB = fp8.mx_quantize(B)
    D = fp8.mx_gemm(A, B)
    absD = np.zeros_like(D)
    for b in range(XA.shape[1]):
        s = slice(32 * b, 32 * (b + 1))
        absD += (XA[:, b:b + 1] * XB[:, b][None, :]) * (np.abs(PA[:, s]) @ np.abs(PB[:, s]).T)
    return D, absD


@pytest.mark.parametrize("M,N,K", [(300, 200, 352), (1024, 1024, 1024), (128, 384, 64),
                                   (777, 129, 2560)])
def test_mx_gemm_within_fp32_summation_bound(L, M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    qa, sfa = quantize(L, A.cuda(), M, K, 0, "bf16")
    qb, sfb = quantize(L, B.cuda(), N, K, 0, "bf16")
    C = mx_gemm_dev(L, qa, sfa, qb, sfb, M, N, K)
    torch.cuda.synchronize()
    D, absD = exact_and_abs(A.double().numpy(), B.double().numpy())
    gk = K * U / (1 - K * U)
    err = np.abs(C.cpu().double().numpy() - D)
    assert np.all(err <= gk * absD + 1e-30), (err / np.maximum(absD, 1e-30)).max()


def test_mx_gemm_epilogues(L):
    M, N, K = 256, 384, 320
    g = torch.Generator().manual_seed(5)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    bias = (torch.randn(N, generator=g) * 0.1).to(torch.bfloat16)
    aux = torch.randn(M, N, generator=g).to(torch.bfloat16)
    qa, sfa = quantize(L, A.cuda(), M, K, 0, "bf16")
    qb, sfb = quantize(L, B.cuda(), N, K, 0, "bf16")
    D, absD = exact_and_abs(A.double().numpy(), B.double().numpy())
    bb, xx = bias.double().numpy(), aux.double().numpy()
    from scipy.special import erf
    gelu = lambda a: 0.5 * a * (1 + erf(a / np.sqrt(2)))
    dgelu = lambda a: 0.5 * (1 + erf(a / np.sqrt(2))) + a * np.exp(-0.5 * a * a) / np.sqrt(2 * np.pi)

    def check(got, ref, tol):
        assert np.abs(got - ref).max() <= tol * (np.abs(ref).max() + 1e-30), np.abs(got - ref).max()

    C = mx_gemm_dev(L, qa, sfa, qb, sfb, M, N, K, epi=1, c_dtype="bf16", bias=bias.cuda())
    check(C.cpu().double().numpy(), D + bb, 2 ** -7)
    C2 = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    C = mx_gemm_dev(L, qa, sfa, qb, sfb, M, N, K, epi=2, c_dtype="bf16", bias=bias.cuda(), C2=C2)
    check(C.cpu().double().numpy(), gelu(D + bb), 2 ** -7)
    check(C2.cpu().double().numpy(), dgelu(D + bb), 2 ** -7)
    C = mx_gemm_dev(L, qa, sfa, qb, sfb, M, N, K, epi=3, c_dtype="bf16", bias=bias.cuda(),
                    aux=aux.cuda())
    check(C.cpu().double().numpy(), D + bb + xx, 2 ** -7)
    C = mx_gemm_dev(L, qa, sfa, qb, sfb, M, N, K, epi=4, c_dtype="bf16", aux=aux.cuda())
    check(C.cpu().double().numpy(), D * xx, 2 ** -7)
    C0 = torch.randn(M, N, generator=g)
    C = mx_gemm_dev(L, qa, sfa, qb, sfb, M, N, K, epi=5, c_dtype="f32", C=C0.clone().cuda())
    gk = K * U / (1 - K * U)
    ref = C0.double().numpy() + D
    err = np.abs(C.cpu().double().numpy() - ref)
    assert np.all(err <= gk * absD + U * np.abs(ref) * 2 + 1e-30)


def test_scale_of_each_row_and_block(L):
    """All elements 1.0 (code 0x38), K = 128 (four blocks): D[m, n] =
    32 * sum_j SA[m, j] SB[n, j].  With SB = 1 and SA[m, j] = 2^e(m, j) the sum
    identifies the four scales the hardware applied to row m."""
    M, N, K = 256, 128, 128
    ldq = 128
    qa = torch.full((M, ldq), 0x38, dtype=torch.uint8, device="cuda")
    qb = torch.full((N, ldq), 0x38, dtype=torch.uint8, device="cuda")
    e = np.zeros((M, 4), dtype=np.int64)
    for m in range(M):
        for j in range(4):
            e[m, j] = (m % 97) - 48 + 6 * j          # distinct per row, four apart per block
    sfa = np.full(L.oases_mx_scale_bytes(M, K), 127, dtype=np.uint8)
    for m in range(M):
        for j in range(4):
            sfa[(m // 128) * 512 + (m % 32) * 16 + ((m % 128) // 32) * 4 + j] = e[m, j] + 127
    sfb = np.full(L.oases_mx_scale_bytes(N, K), 127, dtype=np.uint8)
    sfa_d = torch.from_numpy(sfa).cuda()
    sfb_d = torch.from_numpy(sfb).cuda()
    C = mx_gemm_dev(L, qa, sfa_d, qb, sfb_d, M, N, K)
    torch.cuda.synchronize()
    want = 32.0 * (2.0 ** e).sum(axis=1)
    got = C.cpu().double().numpy()
    np.testing.assert_array_equal(got, np.repeat(want[:, None], N, axis=1))
    # the same with the roles swapped: scales on B's rows
    sfb2 = np.full(L.oases_mx_scale_bytes(N, K), 127, dtype=np.uint8)
    eb = np.zeros((N, 4), dtype=np.int64)
    for n in range(N):
        for j in range(4):
            eb[n, j] = (n % 61) - 30 + 5 * j
            sfb2[(n % 32) * 16 + ((n % 128) // 32) * 4 + j] = eb[n, j] + 127
    sfa1 = torch.full((L.oases_mx_scale_bytes(M, K),), 127, dtype=torch.uint8, device="cuda")
    C = mx_gemm_dev(L, qa, sfa1, qb, torch.from_numpy(sfb2).cuda(), M, N, K)
    torch.cuda.synchronize()
    want = 32.0 * (2.0 ** eb).sum(axis=1)
    np.testing.assert_array_equal(C.cpu().double().numpy(), np.repeat(want[None, :], M, axis=0))


def test_invalid_arguments_rejected_before_launch(L):
    q = torch.zeros(128, 128, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(512, dtype=torch.uint8, device="cuda")
    C = torch.zeros(128, 128, device="cuda")
    # ldq not a multiple of 16
    assert L.oases_mx_quantize(C.data_ptr(), 128, 128, 100, 0, 0, q.data_ptr(), 100,
                               sf.data_ptr(), None) == 1
    # lda < K
    assert L.oases_mx_gemm(128, 128, 256, q.data_ptr(), 128, sf.data_ptr(), q.data_ptr(), 128,
                           sf.data_ptr(), 0, C.data_ptr(), 128, 0, None, None, None, 0, None) == 2
    # Accum into bf16
    assert L.oases_mx_gemm(128, 128, 128, q.data_ptr(), 128, sf.data_ptr(), q.data_ptr(), 128,
                           sf.data_ptr(), 5, C.data_ptr(), 128, 1, None, None, None, 0, None) == 1
    assert L.oases_mx_scale_bytes(300, 129) == 3 * 2 * 512
