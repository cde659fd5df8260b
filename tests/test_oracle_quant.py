"""Pins for the oracle's fine-grained quantizers (1x128 activation tiles,
128x128 weight blocks; news.qq.com/rain/a/20241229A05OQF00, "FP8 低精度训练",
Fig. 7a). Each check rests on something the format or the mathematics fixes:
closed forms (zero tiles, spike tiles, grid values times a power of two),
the half-ulp error bound, an independent library codec, and tile membership
at ragged tails."""
import ml_dtypes
import numpy as np
import torch

import oracle


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _e4m3_ulp(y):
    """Grid step of E4M3 at |y|: 2^(max(floor(log2|y|), -6) - 3)."""
    a = np.abs(np.asarray(y, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 2.0 ** -20)))
    return np.exp2(np.maximum(e, -6) - 3)


def test_all_zero_tile_gives_zero_scale_and_zero_codes():
    x = torch.zeros(3, 256, dtype=torch.bfloat16)
    x[1, :128] = -0.0  # negative zeros too: an all-zero tile encodes to 0x00
    q, s = oracle.quant_act(_bits(x))
    assert np.all(s == 0) and np.all(q == 0)
    qw, sw = oracle.quant_weight(_bits(x))
    assert np.all(sw == 0) and np.all(qw == 0)


def test_spike_tile():
    for v in (3.5, -1234.0, 2.0 ** -20, 6.0e4):
        x = torch.zeros(1, 128, dtype=torch.bfloat16)
        x[0, 37] = v
        vb = float(x[0, 37])
        q, s = oracle.quant_act(_bits(x))
        assert s[0, 0] == np.float32(abs(vb)) / np.float32(448)
        want = np.zeros(128, dtype=np.uint8)
        want[37] = 0x7E | (0x80 if vb < 0 else 0)
        assert np.array_equal(q[0], want)


def test_grid_values_times_power_of_two_round_trip_exactly():
    # A tile whose values are E4M3 grid values g_i times 2^j, with max |g_i|
    # = 448, has s = 2^j exactly, so x / s = g_i and the codes are g's codes.
    rng = np.random.default_rng(3)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    for j in (-20, -7, 0, 5, 30):
        codes = rng.choice(finite, size=(4, 384)).astype(np.uint8)
        codes[:, ::128] = 0x7E  # each tile holds +448 somewhere
        codes[1, 128] = 0xFE    # ... or -448
        g = oracle.e4m3_decode(codes)
        x = _bf16(g * 2.0 ** j)
        assert np.array_equal(x.float().numpy().astype(np.float64), g * 2.0 ** j)  # exact in bf16
        q, s = oracle.quant_act(_bits(x))
        assert np.all(s == np.float32(2.0 ** j))
        assert np.array_equal(q, codes)
        # the same block as a weight matrix: 128x128 blocks, scale 2^j
        wc = rng.choice(finite, size=(256, 256)).astype(np.uint8)
        wc[0, 0] = wc[0, 128] = wc[128, 0] = wc[255, 255] = 0x7E
        w = _bf16(oracle.e4m3_decode(wc) * 2.0 ** j)
        qw, sw = oracle.quant_weight(_bits(w))
        assert np.all(sw == np.float32(2.0 ** j)) and np.array_equal(qw, wc)


def _random_act(M, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g)
    x[:, torch.randperm(K, generator=g)[:3]] *= 100.0  # outlier channels
    x[0, :] *= 1e-30  # a row of tiny values
    return x.to(torch.bfloat16)


def test_half_ulp_error_bound():
    x = _random_act(64, 1024, 11)
    q, s = oracle.quant_act(_bits(x))
    xf = x.float().numpy().astype(np.float64)
    sf = np.repeat(s.astype(np.float64), 128, axis=1)
    deq = oracle.e4m3_decode(q) * sf
    y = xf / np.where(sf > 0, sf, 1)
    bound = 0.5 * _e4m3_ulp(y) * sf + np.abs(xf) * 2.0 ** -24
    assert np.all(np.abs(xf - deq) <= bound)
    assert np.all(np.abs(y) <= 448 * (1 + 2.0 ** -23))


def test_codes_match_library_codec_on_quotients():
    x = _random_act(32, 768, 5)
    q, s = oracle.quant_act(_bits(x))
    xf = x.float().numpy()
    sf = np.repeat(s, 128, axis=1)
    y = xf / sf  # numpy float32 divide: IEEE round to nearest
    lib = np.clip(y, -448, 448).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(q, lib)
    # and the scale is the amax of each tile over 448
    amax = np.abs(xf).reshape(32, 6, 128).max(axis=2)
    assert np.array_equal(s, amax.astype(np.float32) / np.float32(448))


def test_act_tail_tile_covers_present_elements_only():
    # K = 200: one full tile [0,128) and a tail tile [128,200).
    g = torch.Generator().manual_seed(2)
    x = torch.randn(5, 200, generator=g)
    x[:, 100] = 50.0  # the full tile's max; must not leak into the tail tile
    x = x.to(torch.bfloat16)
    q, s = oracle.quant_act(_bits(x))
    xf = x.float().numpy()
    assert s.shape == (5, 2)
    assert np.all(s[:, 0] == np.float32(50.0) / np.float32(448))
    assert np.array_equal(s[:, 1], np.abs(xf[:, 128:]).max(axis=1) / np.float32(448))
    lib = np.clip(xf[:, 128:] / s[:, 1:2], -448, 448).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(q[:, 128:], lib)


def test_weight_blocks_and_tails():
    # N = 200, K = 336: blocks of 128x128, 128x80, 72x128, 72x80.
    g = torch.Generator().manual_seed(4)
    w = (torch.randn(200, 336, generator=g) * 0.01).to(torch.bfloat16)
    q, s = oracle.quant_weight(_bits(w))
    assert s.shape == (2, 3)
    wf = w.float().numpy()
    for nb in range(2):
        for kb in range(3):
            blk = wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            sc = np.float32(np.abs(blk).max()) / np.float32(448)
            assert s[nb, kb] == sc
            lib = np.clip(blk / sc, -448, 448).astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
            assert np.array_equal(q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128], lib)


def test_weight_block_amax_spans_all_128_rows():
    # A single large value in row 127 of a block sets the scale of that whole
    # block (all 128 rows), and of no other block.
    w = torch.ones(256, 256, dtype=torch.bfloat16)
    w[127, 5] = 64.0
    q, s = oracle.quant_weight(_bits(w))
    assert s[0, 0] == np.float32(64.0) / np.float32(448)
    assert np.all(s.ravel()[1:] == np.float32(1.0) / np.float32(448))
    assert q[127, 5] == 0x7E and q[0, 0] == oracle.e4m3_encode(np.array([448 / 64], np.float32))[0]


def test_threading_does_not_change_results():
    x = _random_act(37, 512, 8)
    a = oracle.quant_act(_bits(x), threads=1)
    b = oracle.quant_act(_bits(x), threads=8)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# ---- the backward-pass layouts: 128x1 activation tiles and transposed weights
def test_act_t_scales_are_column_maxima_over_128_rows():
    # 128x1 tiles along M: st[k, mb] = fl32(max_{m in block mb} |x[m, k]| / 448),
    # computed here straight from x with numpy; a ragged last block (M = 300)
    # covers rows 256..299 only.
    rng = np.random.default_rng(31)
    M, K = 300, 136
    x = _bf16(rng.standard_normal((M, K)) * np.exp2(rng.integers(-8, 8, size=(1, K))))
    qt, st = oracle.quant_act_t(_bits(x))
    assert qt.shape == (K, M) and st.shape == (K, 3)
    xf = x.float().numpy()
    for mb in range(3):
        amax = np.abs(xf[128 * mb:min(M, 128 * mb + 128)]).max(axis=0)
        assert np.array_equal(st[:, mb], amax.astype(np.float32) / np.float32(448))


def test_act_t_codes_decode_to_the_transposed_input():
    # q[k, m] * st[k, m / 128] approximates x[m, k] within half an E4M3 step
    # of the quotient (plus the quotient's own rounding): this fails for a
    # transposed operand or a scale taken from the wrong block.
    rng = np.random.default_rng(32)
    M, K = 256, 128
    x = _bf16(rng.standard_normal((M, K)))
    x[:, 5] *= 1000.0  # one loud column must not change its neighbours' scales
    qt, st = oracle.quant_act_t(_bits(x))
    xf = x.float().numpy().astype(np.float64)
    deq = oracle.e4m3_decode(qt) * np.repeat(st.astype(np.float64), 128, axis=1)[:, :M]
    y = xf.T / np.repeat(st.astype(np.float64), 128, axis=1)[:, :M]
    bound = 0.5 * _e4m3_ulp(y) * np.repeat(st, 128, axis=1)[:, :M] + np.abs(xf.T) * 2.0 ** -23
    assert np.all(np.abs(deq - xf.T) <= bound)
    assert st[5, 0] > 100 * st[4, 0] and st[5, 1] > 100 * st[6, 1]


def test_act_t_spike_in_one_column_and_block():
    # a single nonzero at (m, k) = (200, 3): only tile (k = 3, mb = 1) has a
    # nonzero scale, and its code at m = 200 is 0x7E (+448).
    x = torch.zeros(256, 16, dtype=torch.bfloat16)
    x[200, 3] = 7.0
    qt, st = oracle.quant_act_t(_bits(x))
    want_s = np.zeros((16, 2), np.float32)
    want_s[3, 1] = np.float32(7.0) / np.float32(448)
    assert np.array_equal(st, want_s)
    want_q = np.zeros((16, 256), np.uint8)
    want_q[3, 200] = 0x7E
    assert np.array_equal(qt, want_q)


def test_weight_t_is_the_same_blocks_in_the_other_layout():
    # the transposed outputs hold, for code (k, n), the code of w[n, k] and the
    # scale of block (n / 128, k / 128); checked through the block amax
    # computed with numpy and the decode bound, not through the transpose.
    rng = np.random.default_rng(33)
    N, K = 320, 272
    w = _bf16(rng.standard_normal((N, K)) * 0.02)
    q, s, qt, st = oracle.quant_weight_t(_bits(w))
    assert qt.shape == (K, N) and st.shape == (3, 3)
    wf = w.float().numpy()
    for kb in range(3):
        for nb in range(3):
            blk = wf[128 * nb:128 * nb + 128, 128 * kb:128 * kb + 128]
            assert st[kb, nb] == np.float32(np.abs(blk).max()) / np.float32(448)
    sc = np.repeat(np.repeat(st.astype(np.float64), 128, 0), 128, 1)[:K, :N]
    deq = oracle.e4m3_decode(qt) * sc
    y = wf.T.astype(np.float64) / sc
    assert np.all(np.abs(deq - wf.T) <= 0.5 * _e4m3_ulp(y) * sc + np.abs(wf.T) * 2.0 ** -23)
    assert np.array_equal(qt.T, q) and np.array_equal(st.T, s)
