"""GPU block-scaled GEMM vs the CPU oracle, within
|C - C_oracle| <= 1 bf16 ulp + 1e-5 * sum_k |a_k b_k|, on ragged small
shapes (full output), random codes with wide dynamic range, every tile
width (128, 160, 224, 256), and sampled outputs of the full-size workloads."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_gemm_ok, bits, host, to_f32

pytestmark = pytest.mark.gpu

FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


@pytest.fixture(scope="module")
def q():
    from fp8_fine_grained_25_b300 import fp8q as mod
    mod.fp8q_get_device_status()
    yield mod
    mod.fp8q_set_gemm_tile_n(0)
    mod.fp8q_set_gemm_pairs(True)


def _random_operands(M, N, K, seed):
    """Uniformly random finite E4M3 codes (values from 2^-9 to 448, both
    signs) and random positive scales: every block mixes magnitudes over
    ~17 binades, which stresses the in-block accumulation."""
    rng = np.random.default_rng(seed)
    KB, NB = -(-K // 128), -(-N // 128)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.uniform(0.01, 4.0, size=(M, KB)).astype(np.float32)
    sb = rng.uniform(0.01, 4.0, size=(NB, KB)).astype(np.float32)
    return qa, sa, qb, sb


def _run(q, qa, sa, qb, sb, guard=True):
    M, K = qa.shape
    N = qb.shape[0]
    t = lambda a: torch.from_numpy(a).to(DEV)
    Cbuf = torch.full((M + 1, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = q.fp8_block_gemm(t(qa), t(sa), t(qb), t(sb), Cbuf[:M])
    torch.cuda.synchronize()
    if guard:
        assert torch.all(torch.isnan(Cbuf[M])), "GEMM wrote past the end of C"
    return C


# (300, 8, 64) and (257, 24, 128): pair tiles whose output is narrower than one
# store box (every width clips its first box and skips the rest) over less
# than one K block
SHAPES = [(128, 256, 512), (1, 8, 16), (300, 520, 400), (129, 264, 144), (257, 576, 7168),
          (640, 1536, 1024), (1000, 2056, 256), (384, 384, 2048), (300, 8, 64), (257, 24, 128)]


@pytest.mark.parametrize("bn", [0, 128, 160, 224, 256])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_random_codes_full_output(q, M, N, K, bn):
    q.fp8q_set_gemm_tile_n(bn)
    qa, sa, qb, sb = _random_operands(M, N, K, M + 3 * N + 7 * K)
    C = _run(q, qa, sa, qb, sb)
    c32, S = oracle.gemm(qa, sa, qb, sb)
    assert not np.isnan(to_f32(C)).any(), "unwritten outputs"
    assert_gemm_ok(to_f32(C), c32, S, f"gemm {M}x{N}x{K} bn={bn}")
    q.fp8q_set_gemm_tile_n(0)


# Ragged last tiles whose second warpgroup stores some 16-column boxes past
# N and then its lowest box (224-wide tiles keep that box for last): the
# staging buffer of a skipped box must not be handed to the next store while
# an earlier store still reads it. Repeated, since a race shows up by chance.
@pytest.mark.parametrize("M,N,K,bn", [(300, 376, 512, 224), (1000, 2176, 256, 224),
                                      (129, 600, 384, 224), (300, 376, 512, 160),
                                      (129, 600, 384, 160)])
def test_gemm_ragged_last_tile_stores(q, M, N, K, bn):
    qa, sa, qb, sb = _random_operands(M, N, K, 3 * M + N + K)
    c32, S = oracle.gemm(qa, sa, qb, sb)
    q.fp8q_set_gemm_tile_n(bn)
    try:
        for rep in range(4):
            C = _run(q, qa, sa, qb, sb)
            assert_gemm_ok(to_f32(C), c32, S, f"gemm {M}x{N}x{K} bn={bn} run {rep}")
    finally:
        q.fp8q_set_gemm_tile_n(0)


@pytest.mark.parametrize("pairs", [True, False])
def test_gemm_tile_widths_agree_bitwise(q, pairs):
    # Every tile width runs the same arithmetic per output element. N = 776
    # puts 224-wide tiles at column offsets 0, 96 and 64 of a 128-column
    # scale block (160-wide: 0, 32, 64, 96), and ends in a partial tile.
    # 160-wide tiles are pair tiles only: without pairs the call runs at
    # the automatic width.
    qa, sa, qb, sb = _random_operands(333, 776, 1024, 5)
    q.fp8q_set_gemm_pairs(pairs)
    try:
        out = {}
        for bn in (128, 160, 224, 256):
            q.fp8q_set_gemm_tile_n(bn)
            out[bn] = _run(q, qa, sa, qb, sb).clone()
    finally:
        q.fp8q_set_gemm_tile_n(0)
        q.fp8q_set_gemm_pairs(True)
    for bn in (128, 160, 224):
        assert torch.equal(out[bn].view(torch.int16), out[256].view(torch.int16)), bn


@pytest.mark.parametrize("bn", [128, 160, 224, 256])
def test_gemm_several_tiles_per_cluster(q, bn):
    """4096 x 2048 outputs in 256-row pair tiles are 2-4 tiles per 2-CTA
    cluster, so each CTA stages and stores several output tiles through the
    same shared memory (224 wide: a 32-column last tile; 160 wide: 128
    columns, and three TMEM accumulators in turn); the full output is
    checked on two runs in a row."""
    qa, sa, qb, sb = _random_operands(4096, 2048, 256, 11 + bn)
    c32, S = oracle.gemm(qa, sa, qb, sb)
    q.fp8q_set_gemm_tile_n(bn)
    try:
        for rep in range(2):
            C = _run(q, qa, sa, qb, sb)
            assert q.fp8q_get_device_status() == 0
            assert_gemm_ok(to_f32(C), c32, S, f"gemm 4096x2048x256 bn={bn} run {rep}")
    finally:
        q.fp8q_set_gemm_tile_n(0)


def test_gemm_repeatable(q):
    qa, sa, qb, sb = _random_operands(256, 512, 768, 9)
    c1 = _run(q, qa, sa, qb, sb).clone()
    c2 = _run(q, qa, sa, qb, sb)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


def test_gemm_accumulation_precision_probe(q):
    """One large product (448^2 ~ 2^17.6) plus 127 mid-size ones (0.25 .. 64,
    random mantissas) in every K block. An in-block accumulator that kept
    only ~14 significant bits relative to the largest term (the limitation
    the pages cite as the reason for promotion) would drop ~2^4 per term and
    fail the 1e-5 * sum|ab| bound by a wide margin."""
    M = N = 128
    K = 1024
    rng = np.random.default_rng(17)
    qa = rng.integers(0x30, 0x50, size=(M, K)).astype(np.uint8)   # 0.5 .. 8
    qb = rng.integers(0x30, 0x50, size=(N, K)).astype(np.uint8)
    qa[:, ::128] = 0x7E
    qb[:, ::128] = 0x7E
    sa = np.ones((M, K // 128), np.float32)
    sb = np.ones((1, K // 128), np.float32)
    C = _run(q, qa, sa, qb, sb)
    c32, S = oracle.gemm(qa, sa, qb, sb)
    assert_gemm_ok(to_f32(C), c32, S, "precision probe")


def test_gemm_from_quantized_tiny_config(q):
    """The tiny workload end to end: quantize on the GPU (checked bit-exact
    elsewhere) and multiply; the oracle quantizes the same bf16 inputs itself."""
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.tiny(seed=0, device=DEV)
    qa, sa = q.fp8q_quant_act(w.A)
    qb, sb = q.fp8q_quant_weight(w.weights["B"])
    C = q.fp8_block_gemm(qa, sa, qb, sb)
    oqa, osa = oracle.quant_act(bits(w.A))
    oqb, osb = oracle.quant_weight(bits(w.weights["B"]))
    c32, S = oracle.gemm(oqa, osa, oqb, osb)
    assert_gemm_ok(to_f32(C), c32, S, "tiny workload")


def _sampled_check(q, A, W, name, n_rows=128, n_cols=64, seed=0):
    """Quantize + GEMM on the GPU at full size; the oracle checks every
    output of: the first and last m-tile, n_rows random rows (all columns),
    and n_cols random columns plus the last n-block's columns (all rows)."""
    M, K = A.shape
    N = W.shape[0]
    qa, sa = q.fp8q_quant_act(A)
    qb, sb = q.fp8q_quant_weight(W)
    C = q.fp8_block_gemm(qa, sa, qb, sb)
    torch.cuda.synchronize()
    assert q.fp8q_get_device_status() == 0
    oqa, osa = oracle.quant_act(bits(A))
    oqb, osb = oracle.quant_weight(bits(W))
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([np.arange(min(128, M)), np.arange(max(0, M - 128), M),
                                     rng.choice(M, size=min(n_rows, M), replace=False)]))
    cols = np.unique(np.concatenate([rng.choice(N, size=min(n_cols, N), replace=False),
                                     np.arange((N - 1) // 128 * 128, N)]))
    c32, S = oracle.gemm(oqa, osa, oqb, osb, rows=rows)
    worst = assert_gemm_ok(host(C[torch.from_numpy(rows).to(DEV)].float()), c32, S,
                           f"{name} sampled rows")
    c32, S = oracle.gemm(oqa, osa, oqb, osb, cols=cols)
    worst = max(worst, assert_gemm_ok(host(C[:, torch.from_numpy(cols).to(DEV)].float()), c32, S,
                                      f"{name} sampled columns"))
    return worst


@pytest.mark.slow
def test_gemm_mla_full_size(q):
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.mla_down(seed=0, device=DEV)
    _sampled_check(q, w.A, w.weights["Wq"], "MLA Wq")
    _sampled_check(q, w.A, w.weights["Wkv"], "MLA Wkv (64-row N tail)")


@pytest.mark.slow
def test_gemm_dense_square_full_size(q):
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.dense_square(seed=0, device=DEV)
    _sampled_check(q, w.A, w.weights["B"], "dense 8192x7168x7168")


@pytest.mark.slow
def test_gemm_large_m_full_size(q):
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.large_m(seed=0, device=DEV)
    _sampled_check(q, w.A, w.weights["B"], "large-M 32768x18432x7168", n_rows=96, n_cols=32)


@pytest.mark.slow
def test_mla_fused_equals_separate_projections(q):
    """Stacking Wq||Wkv (1536 = 12 * 128, so the 128x128 blocks line up) gives
    one GEMM whose column ranges are the two projections, bit for bit; the
    fused output is also checked against the oracle on sampled rows."""
    from fp8_fine_grained_25_b300 import workloads
    sep = workloads.mla_down(seed=0, device=DEV)
    fused = workloads.mla_down_fused(seed=0, device=DEV)
    qa, sa = q.fp8q_quant_act(sep.A)
    outs = []
    for name in ("Wq", "Wkv"):
        qb, sb = q.fp8q_quant_weight(sep.weights[name])
        outs.append(q.fp8_block_gemm(qa, sa, qb, sb))
    qf, sf = q.fp8q_quant_weight(fused.weights["Wqkv"])
    Cf = q.fp8_block_gemm(qa, sa, qf, sf)
    torch.cuda.synchronize()
    assert torch.equal(Cf[:, :1536].view(torch.int16), outs[0].view(torch.int16))
    assert torch.equal(Cf[:, 1536:].view(torch.int16), outs[1].view(torch.int16))
    _sampled_check(q, fused.A, fused.weights["Wqkv"], "MLA fused Wq||Wkv", n_rows=64, n_cols=32)
