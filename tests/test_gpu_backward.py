"""GPU backward-pass pieces vs the CPU oracle.

- fp8q_quant_act_t (128x1 tiles along tokens, codes transposed): codes and
  scales bit-exact with the oracle, ragged M and K tails included.
- fp8q_quant_weight_t (128x128 blocks in both layouts): both layouts
  bit-exact, and the forward layout identical to fp8q_quant_weight.
- fp8_wgrad_gemm (one B scale per row): within the GEMM acceptance bound,
  both tile widths and pair mode, ragged shapes.
- The two backward GEMMs of a dense layer at full size, from bf16 dY, X
  and W through the quantizers, on sampled outputs: dX = dY W as
  fp8_block_gemm(quant_act(dY), qt(W)) and dW = dY^T X as
  fp8_wgrad_gemm(quant_act_t(dY), quant_act_t(X)).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_25_b300 import workloads
from gpu_helpers import DEV, assert_codes_equal, assert_gemm_ok, assert_scales_equal, bits, to_f32

pytestmark = pytest.mark.gpu

FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


@pytest.fixture(scope="module")
def q():
    from fp8_fine_grained_25_b300 import fp8q as mod
    mod.fp8q_get_device_status()
    yield mod
    mod.fp8q_set_gemm_tile_n(0)
    mod.fp8q_set_gemm_pairs(True)


ACT_T_SHAPES = [(128, 128), (16, 16), (400, 208), (256, 7168), (4096, 576), (1040, 1552)]


@pytest.mark.parametrize("M,K", ACT_T_SHAPES)
def test_quant_act_t_matches_oracle(q, M, K):
    x = workloads.activations_with_outliers(M, K, seed=M * 7 + K, device=DEV)
    qt, st = q.fp8q_quant_act_t(x)
    torch.cuda.synchronize()
    qt_ref, st_ref = oracle.quant_act_t(bits(x))
    assert_codes_equal(qt, qt_ref, f"quant_act_t {M}x{K} codes")
    assert_scales_equal(st, st_ref, f"quant_act_t {M}x{K} scales")
    assert q.fp8q_get_device_status() == 0


def test_quant_act_t_zero_and_tiny_columns(q):
    # an all-zero column tile (scale 0, codes 0), a column of negative zeros,
    # and a column whose amax lies in the IEEE-divide range (< 2^-90)
    x = torch.zeros(256, 64, dtype=torch.float32)
    x[:, 1] = -0.0
    x[:, 2] = torch.linspace(-1, 1, 256) * 2.0 ** -100
    x[130, 3] = 5.0
    x = x.to(torch.bfloat16).to(DEV)
    qt, st = q.fp8q_quant_act_t(x)
    torch.cuda.synchronize()
    qt_ref, st_ref = oracle.quant_act_t(bits(x))
    assert_codes_equal(qt, qt_ref, "quant_act_t special columns codes")
    assert_scales_equal(st, st_ref, "quant_act_t special columns scales")


def test_quant_act_t_full_size(q):
    # the weight-gradient operands of the dense layer: X and dY [8192, 7168]
    x = workloads.activations_with_outliers(8192, 7168, seed=11, device=DEV)
    qt, st = q.fp8q_quant_act_t(x)
    torch.cuda.synchronize()
    qt_ref, st_ref = oracle.quant_act_t(bits(x))
    assert_codes_equal(qt, qt_ref, "quant_act_t 8192x7168 codes")
    assert_scales_equal(st, st_ref, "quant_act_t 8192x7168 scales")


WEIGHT_T_SHAPES = [(256, 512), (320, 272), (16, 16), (576, 7168), (2112, 1040)]


@pytest.mark.parametrize("N,K", WEIGHT_T_SHAPES)
def test_quant_weight_t_matches_oracle(q, N, K):
    w = workloads.normal_bf16((N, K), 0.02, seed=N + 5 * K, device=DEV)
    qw, sw, qt, st = q.fp8q_quant_weight_t(w)
    torch.cuda.synchronize()
    q_ref, s_ref, qt_ref, st_ref = oracle.quant_weight_t(bits(w))
    assert_codes_equal(qw, q_ref, f"quant_weight_t {N}x{K} forward codes")
    assert_scales_equal(sw, s_ref, f"quant_weight_t {N}x{K} forward scales")
    assert_codes_equal(qt, qt_ref, f"quant_weight_t {N}x{K} transposed codes")
    assert_scales_equal(st, st_ref, f"quant_weight_t {N}x{K} transposed scales")
    # the forward layout is exactly what fp8q_quant_weight writes
    q1, s1 = q.fp8q_quant_weight(w)
    assert torch.equal(q1, qw) and torch.equal(s1.view(torch.int32), sw.view(torch.int32))
    # and the transposed-only call writes the same transposed outputs
    _, _, qt2, st2 = q.fp8q_quant_weight_t(w, with_forward=False)
    assert torch.equal(qt2, qt) and torch.equal(st2.view(torch.int32), st.view(torch.int32))


def test_quant_weight_t_full_size(q):
    w = workloads.normal_bf16((7168, 7168), 0.01, seed=3, device=DEV)
    _, _, qt, st = q.fp8q_quant_weight_t(w)
    torch.cuda.synchronize()
    _, _, qt_ref, st_ref = oracle.quant_weight_t(bits(w))
    assert_codes_equal(qt, qt_ref, "quant_weight_t 7168x7168 transposed codes")
    assert_scales_equal(st, st_ref, "quant_weight_t 7168x7168 transposed scales")


def test_transposed_entry_points_reject_bad_alignment(q):
    x = torch.zeros(24, 32, dtype=torch.bfloat16, device=DEV)  # M % 16 != 0
    with pytest.raises(q.FP8QError) as e:
        q.fp8q_quant_act_t(x)
    assert e.value.status == q.ERR_ALIGN
    w = torch.zeros(40, 32, dtype=torch.bfloat16, device=DEV)  # N % 16 != 0
    with pytest.raises(q.FP8QError) as e:
        q.fp8q_quant_weight_t(w)
    assert e.value.status == q.ERR_ALIGN


def _rowscaled_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    KB = -(-K // 128)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.uniform(0.01, 4.0, size=(M, KB)).astype(np.float32)
    sb = rng.uniform(0.01, 4.0, size=(N, KB)).astype(np.float32)
    return qa, sa, qb, sb


def _run_wgrad(q, qa, sa, qb, sb):
    M, K = qa.shape
    N = qb.shape[0]
    t = lambda a: torch.from_numpy(a).to(DEV)
    Cbuf = torch.full((M + 1, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = q.fp8_wgrad_gemm(t(qa), t(sa), t(qb), t(sb), Cbuf[:M])
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(Cbuf[M])), "GEMM wrote past the end of C"
    return C


WGRAD_SHAPES = [(256, 256, 512), (128, 8, 16), (300, 520, 400), (384, 200, 208),
                (640, 1536, 1024), (257, 264, 8192)]


@pytest.mark.parametrize("pairs", [True, False])
@pytest.mark.parametrize("bn", [0, 128, 256])
@pytest.mark.parametrize("M,N,K", WGRAD_SHAPES)
def test_wgrad_gemm_random_codes_full_output(q, M, N, K, bn, pairs):
    q.fp8q_set_gemm_tile_n(bn)
    q.fp8q_set_gemm_pairs(pairs)
    try:
        qa, sa, qb, sb = _rowscaled_operands(M, N, K, M + 3 * N + 7 * K)
        C = _run_wgrad(q, qa, sa, qb, sb)
    finally:
        q.fp8q_set_gemm_tile_n(0)
        q.fp8q_set_gemm_pairs(True)
    c32, S = oracle.wgrad_gemm(qa, sa, qb, sb)
    assert not np.isnan(to_f32(C)).any(), "unwritten outputs"
    assert_gemm_ok(to_f32(C), c32, S, f"wgrad {M}x{N}x{K} bn={bn} pairs={pairs}")
    assert q.fp8q_get_device_status() == 0


@pytest.mark.parametrize("bn", [128, 256])
def test_wgrad_gemm_several_tiles_per_cluster(q, bn):
    """4096 x 2056 outputs in 256-row pair tiles are 2-4 tiles per 2-CTA
    cluster: warp 3 stores each staged tile while the promotion warps go on
    to the next one, and the staging is reused only after those stores have
    read it (ragged last n-tile included); full output, two runs in a row."""
    qa, sa, qb, sb = _rowscaled_operands(4096, 2056, 256, 19 + bn)
    c32, S = oracle.wgrad_gemm(qa, sa, qb, sb)
    q.fp8q_set_gemm_tile_n(bn)
    try:
        for rep in range(2):
            C = _run_wgrad(q, qa, sa, qb, sb)
            assert q.fp8q_get_device_status() == 0
            assert_gemm_ok(to_f32(C), c32, S, f"wgrad 4096x2056x256 bn={bn} run {rep}")
    finally:
        q.fp8q_set_gemm_tile_n(0)


def test_wgrad_gemm_uses_each_b_row_scale(q):
    # B scales that differ by row inside one 128-row block: a kernel that
    # took one scale per block would be off by the ratio.
    qa, sa, qb, sb = _rowscaled_operands(256, 256, 1024, 77)
    sb[1::2] *= 8.0
    C = _run_wgrad(q, qa, sa, qb, sb)
    c32, S = oracle.wgrad_gemm(qa, sa, qb, sb)
    assert_gemm_ok(to_f32(C), c32, S, "wgrad alternating row scales")


def _sample(n, count, rng):
    idx = np.concatenate([[0, n - 1], rng.choice(n, size=count, replace=False)])
    return np.unique(idx)


def test_dense_layer_backward_full_size(q):
    # Dense layer y = x W^T with T = 8192 tokens, W [7168, 7168]:
    #   dX [T, 7168] = dY W        (input gradient)
    #   dW [7168, 7168] = dY^T X   (weight gradient)
    T, N, K = 8192, 7168, 7168
    X = workloads.activations_with_outliers(T, K, seed=21, device=DEV)
    dY = workloads.normal_bf16((T, N), 1.0, seed=22, device=DEV)
    W = workloads.normal_bf16((N, K), 0.01, seed=23, device=DEV)
    qdy, sdy = q.fp8q_quant_act(dY)
    _, _, qwt, swt = q.fp8q_quant_weight_t(W, with_forward=False)
    dX = q.fp8_block_gemm(qdy, sdy, qwt, swt)
    qdyt, sdyt = q.fp8q_quant_act_t(dY)
    qxt, sxt = q.fp8q_quant_act_t(X)
    dW = q.fp8_wgrad_gemm(qdyt, sdyt, qxt, sxt)
    torch.cuda.synchronize()
    assert q.fp8q_get_device_status() == 0

    rng = np.random.default_rng(5)
    # input gradient, from the oracle's own quantization of dY and W
    qdy_r, sdy_r = oracle.quant_act(bits(dY))
    _, _, qwt_r, swt_r = oracle.quant_weight_t(bits(W))
    rows, cols = _sample(T, 24, rng), _sample(K, 24, rng)
    c32, S = oracle.gemm(qdy_r, sdy_r, qwt_r, swt_r, rows=rows, cols=cols)
    assert_gemm_ok(to_f32(dX)[np.ix_(rows, cols)], c32, S, "dgrad 8192x7168x7168")
    # weight gradient
    qdyt_r, sdyt_r = oracle.quant_act_t(bits(dY))
    qxt_r, sxt_r = oracle.quant_act_t(bits(X))
    rows, cols = _sample(N, 24, rng), _sample(K, 24, rng)
    c32, S = oracle.wgrad_gemm(qdyt_r, sdyt_r, qxt_r, sxt_r, rows=rows, cols=cols)
    assert_gemm_ok(to_f32(dW)[np.ix_(rows, cols)], c32, S, "wgrad 7168x7168x8192")
