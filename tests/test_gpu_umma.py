"""Tensor-core (tcgen05) operand layouts and descriptors of umma.cuh, checked on the GPU
against numpy: one 128 x N x K GEMM per case. bf16 operands K-major or MN-major (B also as a
sub-block of a wider tile); tf32 operands K-major (the form the tensor cores take tf32 in)."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests.csrc import build_selftest
    lib = ctypes.CDLL(build_selftest.build())
    lib.umma_selftest.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 7 + [ctypes.c_void_p]
    lib.umma_selftest.restype = ctypes.c_int
    lib.umma_selftest_ts.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    lib.umma_selftest_ts.restype = ctypes.c_int
    return lib


def _round(x, kind):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    if kind == 1:  # bf16, nearest even
        u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    elif kind == 2:  # tf32, nearest, ties away from zero
        u = (u + 0x1000) >> 13 << 13
    else:  # tf32 by dropping the low 13 bits
        u = u >> 13 << 13
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


CASES = [(kind, N, K, a_mn, b_mn, b_cols)
         for kind in (1, 2) for N in (64, 128) for K in (64, 128) for a_mn in (0, 1) for b_mn in (0, 1)
         for b_cols in {N if b_mn else K, 128}
         if not (kind == 2 and (a_mn or b_mn))  # tf32 operands are K-major only
         and (b_cols == (N if b_mn else K) or (kind == 1 and b_mn and N == 64))]


@pytest.mark.parametrize("kind,N,K,a_mn,b_mn,b_cols", CASES)
def test_tcgen05_gemm(lib, kind, N, K, a_mn, b_mn, b_cols):
    rng = np.random.default_rng(N * 1000 + K * 10 + kind + 7 * b_mn + 3 * a_mn)
    M = 128
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dD = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.umma_selftest(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), err.data_ptr(), M, N, K, kind, a_mn, b_mn,
                           b_cols, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = _round(A, kind) @ _round(B, kind).T
    got = dD.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=1e-4, atol=1e-4 * np.abs(ref).max())


TS_CASES = [(kind, N, K, raw) for kind in (1, 2) for N in (64, 128) for K in (64, 128) for raw in (0, 1)
            if not (raw and kind == 1)]


@pytest.mark.parametrize("kind,N,K,raw", TS_CASES)
def test_tcgen05_gemm_a_from_tmem(lib, kind, N, K, raw):
    """A read from tensor memory (tf32: one column per element; bf16: a pair per column). With
    raw fp32 in the columns the tensor core reads them at tf32 precision: the result equals the
    product of the operands with A's low 13 mantissa bits dropped (checked against that and
    against nearest rounding; the closer one is reported)."""
    rng = np.random.default_rng(N * 1000 + K * 10 + kind + 5 * raw + 11)
    M = 128
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((N, K)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dD = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.umma_selftest_ts(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), err.data_ptr(), N, K, kind, raw,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = dD.cpu().numpy().astype(np.float64)
    Bq = _round(B, kind)
    if not raw:
        ref = _round(A, kind) @ Bq.T
        np.testing.assert_allclose(got, ref, rtol=1e-4, atol=1e-4 * np.abs(ref).max())
        return
    ref_rn, ref_rz = _round(A, 2) @ Bq.T, _round(A, 3) @ Bq.T
    e_rn = np.abs(got - ref_rn).max() / np.abs(ref_rn).max()
    e_rz = np.abs(got - ref_rz).max() / np.abs(ref_rz).max()
    print(f"raw fp32 A from tensor memory: max rel. deviation from nearest-rounded A {e_rn:.3e}, "
          f"from truncated A {e_rz:.3e}")
    assert min(e_rn, e_rz) < 1e-5
