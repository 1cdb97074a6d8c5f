"""Pins for the oracle's GEMMs (per-tensor and block-scaled).

Checked against: exact rational arithmetic (Python fractions) on tiny shapes,
numpy matmul of the decoded operands on non-square shapes (a transposed
operand or swapped index fails), the exact integer dot product, block mode
with uniform scales reducing to per-tensor mode, and a block-scaled
restatement with einsum over distinct per-group / per-block scales.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch


def dec_torch(q):
    """E4M3 decode by PyTorch's float8_e4m3fn (independent of the oracle)."""
    return torch.from_numpy(np.ascontiguousarray(q, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def random_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38   # no NaN codes
    return c


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 1), (3, 2, 16), (1, 2, 128), (2, 1, 256), (3, 3, 3)])
def test_per_tensor_vs_fractions(oracle, M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = np.float32(rng.uniform(0.001, 3)), np.float32(rng.uniform(0.001, 3))
    R = oracle.gemm_per_tensor(qa, sa, qb, sb)
    A, B = dec_torch(qa), dec_torch(qb)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(A[m, k])) * Fraction(float(B[n, k])) for k in range(K))
            exact *= Fraction(float(sa)) * Fraction(float(sb))
            assert abs(Fraction(float(R[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 51)


def test_block_vs_fractions(oracle):
    rng = np.random.default_rng(3)
    M, N, K = 2, 3, 256
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa = rng.uniform(0.01, 2, (K // 128, M)).astype(np.float32)
    sb = rng.uniform(0.01, 2, ((N + 127) // 128, K // 128)).astype(np.float32)
    R = oracle.gemm_block(qa, sa, qb, sb)
    A, B = dec_torch(qa), dec_torch(qb)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            for kb in range(K // 128):
                part = sum(Fraction(float(A[m, k])) * Fraction(float(B[n, k])) for k in range(kb * 128, kb * 128 + 128))
                exact += part * Fraction(float(sa[kb, m])) * Fraction(float(sb[n // 128, kb]))
            assert abs(Fraction(float(R[m, n])) - exact) <= (abs(exact) + 1) * Fraction(1, 2 ** 49)


def test_per_tensor_vs_numpy_nonsquare(oracle):
    rng = np.random.default_rng(4)
    M, N, K = 37, 53, 160
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa, sb = np.float32(0.75), np.float32(1.25)
    R = oracle.gemm_per_tensor(qa, sa, qb, sb)
    # partial sums are multiples of 2^-18 below 2^35: exact in float64 in any order
    ref = (dec_torch(qa) @ dec_torch(qb).T) * float(sa) * float(sb)
    assert np.array_equal(R, ref)


def test_block_vs_einsum_distinct_scales(oracle):
    rng = np.random.default_rng(5)
    M, N, K = 19, 300, 384          # ragged N: the last weight block row holds 44 rows
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa = (2.0 ** rng.integers(-6, 6, (K // 128, M))).astype(np.float32) * np.float32(1.0 + 2 ** -10)
    sb = (2.0 ** rng.integers(-6, 6, ((N + 127) // 128, K // 128))).astype(np.float32)
    R = oracle.gemm_block(qa, sa, qb, sb)
    A = dec_torch(qa).reshape(M, K // 128, 128)
    B = dec_torch(qb).reshape(N, K // 128, 128)
    P = np.einsum("mgk,ngk->mng", A, B)                       # exact partials
    sbn = sb[np.arange(N) // 128, :]                           # [N, KB]
    ref = np.einsum("mng,gm,ng->mn", P, sa.astype(np.float64), sbn.astype(np.float64))
    np.testing.assert_allclose(R, ref, rtol=1e-14, atol=1e-12)


def test_exact_integer_crosscheck(oracle):
    rng = np.random.default_rng(6)
    M, N, K = 8, 9, 11008
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    R = oracle.gemm_per_tensor(qa, 1.0, qb, 1.0)
    units = oracle.dot_units(qa, qb)
    assert np.array_equal(R, units.astype(np.float64) * 2.0 ** -18)


def test_block_with_uniform_scales_is_per_tensor(oracle):
    rng = np.random.default_rng(7)
    M, N, K = 6, 130, 512
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    a, b = np.float32(0.0123), np.float32(3.5)
    sa = np.full((K // 128, M), a, np.float32)
    sb = np.full(((N + 127) // 128, K // 128), b, np.float32)
    Rb = oracle.gemm_block(qa, sa, qb, sb)
    Rp = oracle.gemm_per_tensor(qa, a, qb, b)
    np.testing.assert_allclose(Rb, Rp, rtol=1e-14, atol=1e-14 * np.abs(Rp).max())


def test_row_subset(oracle):
    rng = np.random.default_rng(8)
    M, N, K = 40, 20, 256
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa = rng.uniform(0.1, 1, (K // 128, M)).astype(np.float32)
    sb = rng.uniform(0.1, 1, (1, K // 128)).astype(np.float32)
    rows = np.array([39, 0, 17, 17, 5])
    assert np.array_equal(oracle.gemm_block(qa, sa, qb, sb, rows=rows), oracle.gemm_block(qa, sa, qb, sb)[rows])
    assert np.array_equal(oracle.gemm_per_tensor(qa, 2.0, qb, 0.5, rows=rows),
                          oracle.gemm_per_tensor(qa, 2.0, qb, 0.5)[rows])


def test_tolerance_helper():
    import oracle as o
    R = np.array([1.0, -2.0, 100.0])
    ok, _ = o.within_tolerance(R * (1 + 0.9e-3), R, "f16")
    assert ok
    ok, _ = o.within_tolerance(R + np.array([0, 0, 0.5]), R, "f16")
    assert not ok
    ok, _ = o.within_tolerance(R * (1 + 1.9e-3), R, "bf16")
    assert ok
    # BF16: rounding the exact result itself to BF16 must always pass
    rng = np.random.default_rng(0)
    R = rng.standard_normal(100000) * 3.0
    R[:10] = 1.0 + 2.0 ** -8 * 0.999        # just below a rounding midpoint above 1
    Cb = torch.from_numpy(R).to(torch.bfloat16).double().numpy()
    ok, ratio = o.within_tolerance(Cb, R, "bf16")
    assert ok, ratio
    Ch = R.astype(np.float16).astype(np.float64)
    assert o.within_tolerance(Ch, R, "f16")[0]
    # ... but being two BF16 ulps off at a large value does not
    Cbad = Cb.copy()
    k = int(np.argmax(np.abs(R)))
    Cbad[k] = Cb[k] + np.sign(R[k]) * 2.0 * 2.0 ** (np.frexp(R[k])[1] - 8)
    assert not o.within_tolerance(Cbad, R, "bf16")[0]


# ---------------------------------------------------- per-channel weights
def test_per_channel_vs_fractions(oracle):
    rng = np.random.default_rng(8)
    M, N, K = 3, 4, 48
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sa = np.float32(rng.uniform(0.01, 2))
    sb = rng.uniform(0.001, 3, N).astype(np.float32)
    R = oracle.gemm_per_channel(qa, sa, qb, sb)
    A, B = dec_torch(qa), dec_torch(qb)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(A[m, k])) * Fraction(float(B[n, k])) for k in range(K))
            exact *= Fraction(float(sa)) * Fraction(float(sb[n]))
            assert abs(Fraction(float(R[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 51)


def test_per_channel_scales_columns_not_rows(oracle):
    """Distinct scales per output column on a non-square shape: a scale applied
    by row (a swapped index) or a transposed operand fails."""
    rng = np.random.default_rng(9)
    M, N, K = 29, 41, 96
    qa, qb = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sb = (2.0 ** rng.integers(-6, 6, N)).astype(np.float32)   # powers of two: the products stay exact
    R = oracle.gemm_per_channel(qa, np.float32(0.5), qb, sb)
    ref = (dec_torch(qa) @ dec_torch(qb).T) * 0.5 * sb[None, :].astype(np.float64)
    assert np.array_equal(R, ref)
    # uniform per-channel scales are the per-tensor GEMM
    u = np.full(N, 1.75, np.float32)
    assert np.array_equal(oracle.gemm_per_channel(qa, np.float32(0.5), qb, u),
                          oracle.gemm_per_tensor(qa, np.float32(0.5), qb, np.float32(1.75)))
