"""Pins for the oracle's block-scaled GEMM (news.qq.com/rain/a/20241229A05OQF00,
"FP8 低精度训练": 1x128 / 128x128 scales, Fig. 7a; FP32 promotion of the MMA
partial sums, Fig. 7b).

- Exact rational brute force (fractions.Fraction) on tiny shapes: the FP64
  block partials must equal the exact sums, and the FP32 result must sit
  within the FP32 rounding bound of the exact real value.
- Unit scales: the result equals a library FP64 matmul of the decoded codes,
  rounded to FP32 per block and summed in FP32 in K-block order.
- Scale indexing across 128-column blocks of B and 128-wide K blocks.
A dropped term, a wrong sign, a wrong scale index or a transposed operand
fails one of these."""
from fractions import Fraction

import numpy as np
import pytest

import oracle

FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


def _dec_exact(c):
    return Fraction(float(oracle.e4m3_decode(np.array([c], dtype=np.uint8))[0]))


def _rand_case(rng, M, N, K):
    KB, NB = -(-K // 128), -(-N // 128)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.uniform(1e-4, 2.0, size=(M, KB)).astype(np.float32)
    sb = rng.uniform(1e-4, 2.0, size=(NB, KB)).astype(np.float32)
    sa[rng.random(sa.shape) < 0.2] *= -1  # the bound must not assume positive scales
    return qa, sa, qb, sb


def _exact(qa, sa, qb, sb, m, n):
    """Exact real value sum_k A[m,k] sa[m,k/128] B[n,k] sb[n/128,k/128], the
    exact block partials, and the exact sum of |terms|."""
    K = qa.shape[1]
    KB = -(-K // 128)
    parts, total, S = [], Fraction(0), Fraction(0)
    for kb in range(KB):
        p, pabs = Fraction(0), Fraction(0)
        for k in range(kb * 128, min(K, kb * 128 + 128)):
            t = _dec_exact(qa[m, k]) * _dec_exact(qb[n, k])
            p += t
            pabs += abs(t)
        sc = Fraction(float(sa[m, kb])) * Fraction(float(sb[n // 128, kb]))
        parts.append(p)
        total += p * sc
        S += pabs * abs(sc)
    return parts, total, S


@pytest.mark.parametrize("M,N,K", [(3, 5, 128), (4, 2, 256), (2, 3, 384), (5, 4, 200), (1, 1, 16)])
def test_fraction_brute_force(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    qa, sa, qb, sb = _rand_case(rng, M, N, K)
    KB = -(-K // 128)
    c32, S = oracle.gemm(qa, sa, qb, sb)
    u = 2.0 ** -24
    for m in range(M):
        for n in range(N):
            parts, exact, S_exact = _exact(qa, sa, qb, sb, m, n)
            P = oracle.block_partials(qa, qb, m, n)
            assert [Fraction(float(p)) for p in P] == parts  # FP64 partials are exact
            # FP32: 3 roundings per block term (fl32(P), the scale product,
            # the product) and KB - 1 roundings in the running sum.
            err = abs(Fraction(float(c32[m, n])) - exact)
            assert err <= Fraction((KB + 3) * u * 1.0001) * S_exact + Fraction(2.0 ** -149)
            assert abs(Fraction(float(S[m, n])) - S_exact) <= Fraction(1e-12) * S_exact


def test_result_not_transposed_and_rows_cols_independent():
    rng = np.random.default_rng(99)
    qa, sa, qb, sb = _rand_case(rng, 6, 3, 256)
    c_all, _ = oracle.gemm(qa, sa, qb, sb)
    c_sel, _ = oracle.gemm(qa, sa, qb, sb, rows=[5, 0], cols=[2, 1])
    assert np.array_equal(c_sel, c_all[np.ix_([5, 0], [2, 1])])
    _, exact, _ = _exact(qa, sa, qb, sb, 5, 2)
    assert abs(float(exact) - float(c_all[5, 2])) < 1e-4 * abs(float(exact)) + 1e-30


def test_unit_scales_equal_library_matmul_rounded_per_block():
    rng = np.random.default_rng(5)
    M, N, K = 7, 9, 640
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    ones_a = np.ones((M, K // 128), np.float32)
    ones_b = np.ones((1, K // 128), np.float32)
    c32, _ = oracle.gemm(qa, ones_a, qb, ones_b)
    A, B = oracle.e4m3_decode(qa), oracle.e4m3_decode(qb)
    acc = np.zeros((M, N), np.float32)
    for kb in range(K // 128):
        blk = A[:, kb * 128:(kb + 1) * 128] @ B[:, kb * 128:(kb + 1) * 128].T  # exact in FP64
        acc = (acc + blk.astype(np.float32)).astype(np.float32)
    assert np.array_equal(c32, acc)


def test_b_scale_indexed_by_column_block():
    # N = 384: columns 0..127 use sb[0], 128..255 sb[1], 256..383 sb[2].
    rng = np.random.default_rng(12)
    M, N, K = 2, 384, 256
    qa, sa, qb, sb = _rand_case(rng, M, N, K)
    cols = [0, 127, 128, 255, 256, 383]
    c32, _ = oracle.gemm(qa, sa, qb, sb, cols=cols)
    for i, m in enumerate(range(M)):
        for j, n in enumerate(cols):
            _, exact, S = _exact(qa, sa, qb, sb, m, n)
            assert abs(Fraction(float(c32[i, j])) - exact) <= Fraction(6 * 2.0 ** -24) * S


def test_grouped_fraction_brute_force():
    # 3 experts, the middle one empty; rows map to experts by the offsets.
    rng = np.random.default_rng(21)
    E, N, K = 3, 4, 256
    off = np.array([0, 3, 3, 5], dtype=np.int32)
    qa = rng.choice(FINITE, size=(5, K)).astype(np.uint8)
    sa = rng.uniform(0.01, 1, (5, 2)).astype(np.float32)
    qb = rng.choice(FINITE, size=(E, N, K)).astype(np.uint8)
    sb = rng.uniform(0.01, 1, (E, 1, 2)).astype(np.float32)
    c32, S = oracle.grouped_gemm(qa, sa, qb, sb, off, rows=np.arange(5))
    for m in range(5):
        e = 0 if m < 3 else 2
        for n in range(N):
            _, exact, Se = _exact(qa, sa, qb[e], sb[e], m, n)
            assert abs(Fraction(float(c32[m, n])) - exact) <= Fraction(5 * 2.0 ** -24) * Se
            # and not the other experts' weights
            _, other, _ = _exact(qa, sa, qb[2 - e], sb[2 - e], m, n)
            assert other != exact


def test_acceptance_helpers():
    assert oracle.bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert oracle.bf16_ulp(np.array([3.0]))[0] == 2.0 ** -6
    assert oracle.bf16_ulp(np.array([-0.75]))[0] == 2.0 ** -8
    assert oracle.bf16_ulp(np.array([0.0]))[0] == 2.0 ** -133
    ok, worst, _ = oracle.gemm_check(np.array([1.0 + 2.0 ** -8]), np.array([1.0]), np.array([0.0]))
    assert ok and worst == 0.5
    ok, _, _ = oracle.gemm_check(np.array([1.01]), np.array([1.0]), np.array([0.0]))
    assert not ok
    ok, _, _ = oracle.gemm_check(np.array([1.01]), np.array([1.0]), np.array([1e3]))
    assert ok


# ---- the weight-gradient GEMM: one B scale per row (1x128 tiles on both sides)
def _exact_rows(qa, sa, qb, sb, m, n):
    """Exact sum_k A[m,k] sa[m,k/128] B[n,k] sb[n,k/128] and sum |terms|."""
    K = qa.shape[1]
    total, S = Fraction(0), Fraction(0)
    for kb in range(-(-K // 128)):
        p, pabs = Fraction(0), Fraction(0)
        for k in range(kb * 128, min(K, kb * 128 + 128)):
            t = _dec_exact(qa[m, k]) * _dec_exact(qb[n, k])
            p += t
            pabs += abs(t)
        sc = Fraction(float(sa[m, kb])) * Fraction(float(sb[n, kb]))
        total += p * sc
        S += pabs * abs(sc)
    return total, S


@pytest.mark.parametrize("M,N,K", [(3, 5, 128), (2, 4, 384), (4, 3, 208)])
def test_wgrad_fraction_brute_force(M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    KB = -(-K // 128)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.uniform(1e-3, 2.0, size=(M, KB)).astype(np.float32)
    sb = rng.uniform(1e-3, 2.0, size=(N, KB)).astype(np.float32)
    sb[rng.random(sb.shape) < 0.3] *= -1
    c32, S = oracle.wgrad_gemm(qa, sa, qb, sb)
    u = 2.0 ** -24
    for m in range(M):
        for n in range(N):
            exact, Se = _exact_rows(qa, sa, qb, sb, m, n)
            err = abs(Fraction(float(c32[m, n])) - exact)
            assert err <= Fraction((KB + 3) * u * 1.0001) * Se + Fraction(2.0 ** -149)
            assert abs(Fraction(float(S[m, n])) - Se) <= Fraction(1e-12) * Se
    # each row of B has its own scale: rescaling row 1 of sb changes only column 1
    sb2 = sb.copy()
    sb2[1] *= 2
    c2, _ = oracle.wgrad_gemm(qa, sa, qb, sb2)
    assert np.array_equal(np.delete(c2, 1, axis=1), np.delete(c32, 1, axis=1))
    assert np.array_equal(c2[:, 1], c32[:, 1] * 2)


def test_wgrad_with_block_constant_row_scales_equals_block_gemm():
    # when the 128 rows of each B block share their scales, the per-row form
    # is the forward GEMM with 128x128 block scales, bit for bit.
    rng = np.random.default_rng(41)
    M, N, K = 5, 300, 256
    qa, sa, qb, sb_blocks = _rand_case(rng, M, N, K)
    sb_rows = np.repeat(sb_blocks, 128, axis=0)[:N]
    c_rows, S_rows = oracle.wgrad_gemm(qa, sa, qb, sb_rows)
    c_blk, S_blk = oracle.gemm(qa, sa, qb, sb_blocks)
    assert np.array_equal(c_rows, c_blk) and np.array_equal(S_rows, S_blk)
