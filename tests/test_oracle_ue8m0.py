"""Pins for the oracle's power-of-two (UE8M0) scale mode, a variant outside
the pages (scales rounded up to a power of two so that a tensor core with
hardware block scaling can apply them).

- The defining inequality, checked tile by tile with exact arithmetic:
  amax / 2^e <= 448 < amax / 2^(e-1).
- Closed forms: amax = 448 * 2^k gives byte 127 + k and the amax element
  encodes to 0x7E; the next bf16 above it gives byte 128 + k.
- Codes: x / 2^e is exact, so the codes equal an independent library codec
  (ml_dtypes float8_e4m3fn) applied to x * 2^-e.
- All-zero tiles: byte 0 and codes 0; weight blocks span 128 rows.
- The UE8M0 GEMM at unit scale bytes equals a library FP64 matmul rounded
  per block, and matches exact rational brute force for random bytes."""
from fractions import Fraction

import ml_dtypes
import numpy as np
import torch

import oracle

FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_scale_is_the_smallest_power_of_two_that_fits():
    rng = np.random.default_rng(1)
    x = _bf16(rng.standard_normal((64, 512)) * np.exp2(rng.integers(-40, 40, size=(64, 1))))
    q, s = oracle.quant_act_ue8m0(_bits(x))
    xf = x.float().numpy().astype(np.float64)
    for m in range(64):
        for kb in range(4):
            amax = Fraction(float(np.abs(xf[m, 128 * kb:128 * kb + 128]).max()))
            e = int(s[m, kb]) - 127
            sc = Fraction(2) ** e
            assert amax / sc <= 448 < amax / (sc / 2), (m, kb, e)


def test_closed_forms_at_power_of_two_multiples_of_448():
    for k in (-20, -3, 0, 4, 30):
        x = torch.zeros(2, 128, dtype=torch.bfloat16)
        x[0, 7] = 448.0 * 2.0 ** k
        x[1, 7] = 448.0 * 2.0 ** k
        x[1, 9] = 450.0 * 2.0 ** k  # the next bf16 above 448 * 2^k
        q, s = oracle.quant_act_ue8m0(_bits(x))
        assert s[0, 0] == 127 + k and q[0, 7] == 0x7E
        assert s[1, 0] == 128 + k


def test_codes_equal_library_codec_on_exact_quotients():
    rng = np.random.default_rng(2)
    x = _bf16(rng.standard_normal((32, 384)) * 3.0)
    q, s = oracle.quant_act_ue8m0(_bits(x))
    xf = x.float().numpy()
    scale = np.repeat(oracle.ue8m0_to_f32(s), 128, axis=1)
    y = xf / scale  # exact: division by a power of two in range
    ref = y.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(q, ref)
    assert np.all(np.abs(y) <= 448)


def test_zero_tiles_and_weight_blocks():
    x = torch.zeros(3, 256, dtype=torch.bfloat16)
    x[1, :128] = -0.0
    q, s = oracle.quant_act_ue8m0(_bits(x))
    assert np.all(s == 0) and np.all(q == 0)
    w = torch.zeros(256, 128, dtype=torch.bfloat16)
    w[200, 5] = 3.0  # the second block row's amax
    qw, sw = oracle.quant_weight_ue8m0(_bits(w))
    assert sw[0, 0] == 0 and sw[1, 0] == 127 - 7  # 3 / 2^-7 = 384 <= 448 < 768
    assert qw[200, 5] == np.float32(384.0).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)


def test_ue8m0_gemm_unit_bytes_equal_library_matmul_rounded_per_block():
    rng = np.random.default_rng(5)
    M, N, K = 6, 9, 384
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    c32, _ = oracle.gemm_ue8m0(qa, np.full((M, 3), 127, np.uint8), qb, np.full((1, 3), 127, np.uint8))
    A, B = oracle.e4m3_decode(qa), oracle.e4m3_decode(qb)
    acc = np.zeros((M, N), np.float32)
    for kb in range(3):
        acc = (acc + (A[:, 128 * kb:128 * kb + 128] @ B[:, 128 * kb:128 * kb + 128].T).astype(np.float32)).astype(np.float32)
    assert np.array_equal(c32, acc)


def test_ue8m0_gemm_fraction_brute_force():
    rng = np.random.default_rng(6)
    M, N, K = 3, 4, 256
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.integers(100, 150, size=(M, 2)).astype(np.uint8)
    sb = rng.integers(100, 150, size=(1, 2)).astype(np.uint8)
    c32, S = oracle.gemm_ue8m0(qa, sa, qb, sb)
    dec = lambda c: Fraction(float(oracle.e4m3_decode(np.array([c], np.uint8))[0]))
    for m in range(M):
        for n in range(N):
            exact, Se = Fraction(0), Fraction(0)
            for kb in range(2):
                sc = Fraction(2) ** (int(sa[m, kb]) - 127 + int(sb[0, kb]) - 127)
                for k in range(128 * kb, 128 * kb + 128):
                    t = dec(qa[m, k]) * dec(qb[n, k]) * sc
                    exact += t
                    Se += abs(t)
            # the per-block scaling is exact; only the FP32 roundings of the
            # two block terms and their sum remain
            assert abs(Fraction(float(c32[m, n])) - exact) <= Fraction(3 * 2.0 ** -24) * Se


def test_act_t_ue8m0_bytes_follow_the_rule_per_column_tile():
    # 128x1 tiles along M: byte[k, mb] is the smallest 2^e with
    # max_{m in block} |x[m, k]| / 2^e <= 448, checked exactly from x
    rng = np.random.default_rng(9)
    M, K = 300, 48
    x = _bf16(rng.standard_normal((M, K)) * np.exp2(rng.integers(-30, 30, size=(1, K))))
    qt, st = oracle.quant_act_t_ue8m0(_bits(x))
    assert qt.shape == (K, M) and st.shape == (K, 3)
    xf = x.float().numpy().astype(np.float64)
    for k in range(K):
        for mb in range(3):
            amax = Fraction(float(np.abs(xf[128 * mb:min(M, 128 * mb + 128), k]).max()))
            sc = Fraction(2) ** (int(st[k, mb]) - 127)
            assert amax / sc <= 448 < amax / (sc / 2)
    # codes: the exact quotients through the library codec
    scale = np.repeat(oracle.ue8m0_to_f32(st), 128, axis=1)[:, :M]
    ref = (xf.T.astype(np.float32) / scale).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(qt, ref)


def test_wgrad_ue8m0_fraction_brute_force():
    rng = np.random.default_rng(10)
    M, N, K = 3, 4, 256
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.integers(110, 145, size=(M, 2)).astype(np.uint8)
    sb = rng.integers(110, 145, size=(N, 2)).astype(np.uint8)  # one byte per B row
    c32, S = oracle.wgrad_gemm_ue8m0(qa, sa, qb, sb)
    dec = lambda c: Fraction(float(oracle.e4m3_decode(np.array([c], np.uint8))[0]))
    for m in range(M):
        for n in range(N):
            exact, Se = Fraction(0), Fraction(0)
            for kb in range(2):
                sc = Fraction(2) ** (int(sa[m, kb]) + int(sb[n, kb]) - 254)
                for k in range(128 * kb, 128 * kb + 128):
                    t = dec(qa[m, k]) * dec(qb[n, k]) * sc
                    exact += t
                    Se += abs(t)
            assert abs(Fraction(float(c32[m, n])) - exact) <= Fraction(3 * 2.0 ** -24) * Se
