"""GPU power-of-two (UE8M0) scale mode vs the CPU oracle: codes and scale
bytes bit-exact (ragged tails, zero tiles, tiny and huge amax, full size)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_25_b300 import workloads
from gpu_helpers import DEV, assert_codes_equal, bits, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    from fp8_fine_grained_25_b300 import fp8q as mod
    mod.fp8q_get_device_status()
    return mod


def _bytes_equal(s_gpu, s_ref, what):
    sg = host(s_gpu)
    if not np.array_equal(sg, s_ref):
        i = tuple(np.argwhere(sg != s_ref)[0])
        raise AssertionError(f"{what}: scale bytes differ at {i}: gpu {sg[i]} oracle {s_ref[i]}")


@pytest.mark.parametrize("M,K", [(1, 16), (130, 400), (256, 7168), (4096, 576)])
def test_quant_act_ue8m0_matches_oracle(q, M, K):
    x = workloads.activations_with_outliers(M, K, seed=M + K, device=DEV)
    qa, sa = q.fp8q_quant_act_ue8m0(x)
    torch.cuda.synchronize()
    qr, sr = oracle.quant_act_ue8m0(bits(x))
    assert_codes_equal(qa, qr, f"act ue8m0 {M}x{K} codes")
    _bytes_equal(sa, sr, f"act ue8m0 {M}x{K}")


@pytest.mark.parametrize("N,K", [(256, 512), (576, 7168), (200, 144)])
def test_quant_weight_ue8m0_matches_oracle(q, N, K):
    w = workloads.normal_bf16((N, K), 0.02, seed=N * 3 + K, device=DEV)
    qw, sw = q.fp8q_quant_weight_ue8m0(w)
    torch.cuda.synchronize()
    qr, sr = oracle.quant_weight_ue8m0(bits(w))
    assert_codes_equal(qw, qr, f"weight ue8m0 {N}x{K} codes")
    _bytes_equal(sw, sr, f"weight ue8m0 {N}x{K}")


def test_ue8m0_special_tiles(q):
    # zero tiles (incl. -0), amax exactly 448 * 2^k and just above, tiny amax
    # (scale clamped at 2^-127), huge amax, one tile per row
    x = torch.zeros(8, 128, dtype=torch.float32)
    x[1] = -0.0
    x[2, 3] = 448.0 * 2.0 ** 5
    x[3, 3] = 450.0 * 2.0 ** 5
    x[4] = torch.linspace(-1, 1, 128) * 2.0 ** -130
    x[5] = torch.linspace(-1, 1, 128) * 2.0 ** 120
    x[6, :64] = 1.0
    x[7] = torch.linspace(-3, 3, 128)
    x = x.to(torch.bfloat16).to(DEV)
    qa, sa = q.fp8q_quant_act_ue8m0(x)
    torch.cuda.synchronize()
    qr, sr = oracle.quant_act_ue8m0(bits(x))
    assert_codes_equal(qa, qr, "ue8m0 special tiles codes")
    _bytes_equal(sa, sr, "ue8m0 special tiles")
    assert sr[0, 0] == 0 and sr[1, 0] == 0 and sr[2, 0] == 132 and sr[3, 0] == 133


def test_quant_act_ue8m0_full_size(q):
    x = workloads.activations_with_outliers(8192, 7168, seed=0, device=DEV)
    qa, sa = q.fp8q_quant_act_ue8m0(x)
    torch.cuda.synchronize()
    qr, sr = oracle.quant_act_ue8m0(bits(x))
    assert_codes_equal(qa, qr, "act ue8m0 8192x7168 codes")
    _bytes_equal(sa, sr, "act ue8m0 8192x7168")
    assert q.fp8q_get_device_status() == 0


FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


def _run_bs(q, qa, sa, qb, sb):
    M, K = qa.shape
    N = qb.shape[0]
    t = lambda a: torch.from_numpy(a).to(DEV)
    Cbuf = torch.full((M + 1, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = q.fp8_block_gemm_ue8m0(t(qa), t(sa), t(qb), t(sb), Cbuf[:M])
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(Cbuf[M])), "GEMM wrote past the end of C"
    return C


BS_SHAPES = [(128, 224, 128), (1, 8, 16), (300, 520, 400), (129, 264, 144), (257, 576, 7168),
             (640, 1536, 1024), (1000, 2056, 256), (384, 448, 2048), (512, 224, 640)]


@pytest.mark.parametrize("pairs", [True, False])
@pytest.mark.parametrize("M,N,K", BS_SHAPES)
def test_block_gemm_ue8m0_random_codes(q, M, N, K, pairs):
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    KB, NB = -(-K // 128), -(-N // 128)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.integers(110, 140, size=(M, KB)).astype(np.uint8)
    sb = rng.integers(110, 140, size=(NB, KB)).astype(np.uint8)
    q.fp8q_set_gemm_pairs(pairs)
    try:
        C = _run_bs(q, qa, sa, qb, sb)
    finally:
        q.fp8q_set_gemm_pairs(True)
    c32, S = oracle.gemm_ue8m0(qa, sa, qb, sb)
    from gpu_helpers import assert_gemm_ok, to_f32
    assert not np.isnan(to_f32(C)).any(), "unwritten outputs"
    assert_gemm_ok(to_f32(C), c32, S, f"ue8m0 gemm {M}x{N}x{K}")
    assert q.fp8q_get_device_status() == 0


def test_block_gemm_ue8m0_from_quantizers_full_size(q):
    # the dense layer with power-of-two scales, sampled outputs
    from gpu_helpers import assert_gemm_ok, to_f32
    w = workloads.dense_square(seed=0, device=DEV)
    qa, sa = q.fp8q_quant_act_ue8m0(w.A)
    qb, sb = q.fp8q_quant_weight_ue8m0(w.weights["B"])
    C = q.fp8_block_gemm_ue8m0(qa, sa, qb, sb)
    torch.cuda.synchronize()
    assert q.fp8q_get_device_status() == 0
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([[0, 8191], rng.choice(8192, 24, replace=False)]))
    cols = np.unique(np.concatenate([[0, 7167], rng.choice(7168, 24, replace=False)]))
    qar, sar = oracle.quant_act_ue8m0(bits(w.A[torch.as_tensor(rows, device=DEV)]))
    qbr, sbr = oracle.quant_weight_ue8m0(bits(w.weights["B"]))
    c32, S = oracle.gemm_ue8m0(qar, sar, qbr, sbr, cols=cols)
    assert_gemm_ok(to_f32(C)[np.ix_(rows, cols)], c32, S, "ue8m0 dense 8192x7168x7168")


# ---- UE8M0 backward: 128x1 activation tiles, transposed weight blocks,
# ---- and the row-scaled GEMM with hardware block scaling
@pytest.mark.parametrize("M,K", [(128, 128), (400, 208), (4096, 576)])
def test_quant_act_t_ue8m0_matches_oracle(q, M, K):
    x = workloads.activations_with_outliers(M, K, seed=M + 2 * K, device=DEV)
    qt, st = q.fp8q_quant_act_t_ue8m0(x)
    torch.cuda.synchronize()
    qr, sr = oracle.quant_act_t_ue8m0(bits(x))
    assert_codes_equal(qt, qr, f"act_t ue8m0 {M}x{K} codes")
    _bytes_equal(st, sr, f"act_t ue8m0 {M}x{K}")


@pytest.mark.parametrize("N,K", [(256, 512), (320, 272)])
def test_quant_weight_t_ue8m0_matches_oracle(q, N, K):
    w = workloads.normal_bf16((N, K), 0.02, seed=N + 7 * K, device=DEV)
    qw, sw, qt, st = q.fp8q_quant_weight_t_ue8m0(w)
    torch.cuda.synchronize()
    q_r, s_r, qt_r, st_r = oracle.quant_weight_t_ue8m0(bits(w))
    assert_codes_equal(qw, q_r, f"weight_t ue8m0 {N}x{K} forward codes")
    _bytes_equal(sw, s_r, f"weight_t ue8m0 {N}x{K} forward")
    assert_codes_equal(qt, qt_r, f"weight_t ue8m0 {N}x{K} transposed codes")
    _bytes_equal(st, st_r, f"weight_t ue8m0 {N}x{K} transposed")


@pytest.mark.parametrize("pairs", [True, False])
@pytest.mark.parametrize("M,N,K", [(256, 224, 512), (300, 520, 400), (384, 448, 2048)])
def test_wgrad_gemm_ue8m0_random_codes(q, M, N, K, pairs):
    from gpu_helpers import assert_gemm_ok, to_f32
    rng = np.random.default_rng(M * 5 + N + K)
    KB = -(-K // 128)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.integers(110, 140, size=(M, KB)).astype(np.uint8)
    sb = rng.integers(110, 140, size=(N, KB)).astype(np.uint8)
    t = lambda a: torch.from_numpy(a).to(DEV)
    q.fp8q_set_gemm_pairs(pairs)
    try:
        C = q.fp8_wgrad_gemm_ue8m0(t(qa), t(sa), t(qb), t(sb))
        torch.cuda.synchronize()
    finally:
        q.fp8q_set_gemm_pairs(True)
    c32, S = oracle.wgrad_gemm_ue8m0(qa, sa, qb, sb)
    assert_gemm_ok(to_f32(C), c32, S, f"wgrad ue8m0 {M}x{N}x{K} pairs={pairs}")
    assert q.fp8q_get_device_status() == 0
