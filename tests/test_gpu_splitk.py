"""Split K (fp8_block_gemm_ws): the K blocks of each output tile cut into
ranges computed by different work units, with the FP32 partial tiles summed
by the last unit of each tile through a caller-owned workspace. Checked
against the CPU oracle on ragged shapes (full output, every tile width, pairs
on and off, 2 to 4 ranges), for run-to-run repeatability, for workspace reuse
across calls and shapes (no initialisation needed), for the fallback to fewer
ranges when the workspace is small, and on the full-size MLA projections."""
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
    mod.fp8q_set_gemm_splits(0)


def _random_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    KB, NB = -(-K // 128), -(-N // 128)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.uniform(0.01, 4.0, size=(M, KB)).astype(np.float32)
    sb = rng.uniform(0.01, 4.0, size=(NB, KB)).astype(np.float32)
    return qa, sa, qb, sb


def _dev(*arrs):
    return [torch.from_numpy(a).to(DEV) for a in arrs]


def _run_ws(q, ops, ws, guard=True):
    qa, sa, qb, sb = ops
    M, N = qa.shape[0], qb.shape[0]
    Cbuf = torch.full((M + 1, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = q.fp8_block_gemm_ws(qa, sa, qb, sb, Cbuf[:M], workspace=ws)
    torch.cuda.synchronize()
    assert q.fp8q_get_device_status() == 0
    if guard:
        assert torch.all(torch.isnan(Cbuf[M])), "GEMM wrote past the end of C"
    return C


def _workspace(q, M, N, K):
    n = q.fp8_block_gemm_workspace_size(M, N, K)
    # garbage contents: the call must not rely on any initialisation
    return torch.randint(0, 256, (max(n, 256),), dtype=torch.uint8, device=DEV)


SHAPES = [(300, 520, 2048), (129, 264, 1040), (257, 576, 7168), (1, 8, 1024), (640, 1536, 1536)]


@pytest.mark.parametrize("pairs", [True, False])
@pytest.mark.parametrize("bn", [128, 224, 256])
@pytest.mark.parametrize("splits", [2, 3, 4])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_split_k_full_output(q, M, N, K, splits, bn, pairs):
    q.fp8q_set_gemm_tile_n(bn)
    q.fp8q_set_gemm_pairs(pairs)
    q.fp8q_set_gemm_splits(splits)
    try:
        host_ops = _random_operands(M, N, K, M + 5 * N + 3 * K + splits)
        ws = _workspace(q, M, N, K)
        C = _run_ws(q, _dev(*host_ops), ws)
    finally:
        q.fp8q_set_gemm_tile_n(0)
        q.fp8q_set_gemm_pairs(True)
        q.fp8q_set_gemm_splits(0)
    c32, S = oracle.gemm(*host_ops)
    assert not np.isnan(to_f32(C)).any(), "unwritten outputs"
    assert_gemm_ok(to_f32(C), c32, S, f"split-K {M}x{N}x{K} S={splits} bn={bn} pairs={pairs}")


def test_split_k_repeatable_and_reusable(q):
    """The same call twice gives the same bits (the partials are added in
    range order whichever unit finishes last); a workspace left by one call
    (another shape, another split count) serves the next one unchanged."""
    a = _random_operands(384, 776, 3072, 11)
    b = _random_operands(200, 264, 2048, 12)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=DEV)
    q.fp8q_set_gemm_splits(3)
    try:
        da, db = _dev(*a), _dev(*b)
        c1 = _run_ws(q, da, ws).clone()
        c2 = _run_ws(q, da, ws).clone()
        assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))
        q.fp8q_set_gemm_splits(2)
        cb = _run_ws(q, db, ws).clone()
        q.fp8q_set_gemm_splits(3)
        c3 = _run_ws(q, da, ws)
        assert torch.equal(c1.view(torch.int16), c3.view(torch.int16))
    finally:
        q.fp8q_set_gemm_splits(0)
    for C, ops, name in ((c1, a, "a"), (cb, b, "b")):
        c32, S = oracle.gemm(*ops)
        assert_gemm_ok(to_f32(C), c32, S, f"reused workspace {name}")


def test_split_k_small_workspace_falls_back(q):
    """A workspace too small for the requested ranges: fewer ranges are used;
    with no room at all the call is fp8_block_gemm, bit for bit."""
    ops = _dev(*_random_operands(256, 512, 4096, 13))
    q.fp8q_set_gemm_splits(4)
    try:
        C0 = _run_ws(q, ops, torch.empty(256, dtype=torch.uint8, device=DEV)).clone()
        need2 = 2 * 256 * 512 * 4 + 4096
        C2 = _run_ws(q, ops, torch.empty(need2, dtype=torch.uint8, device=DEV)).clone()
    finally:
        q.fp8q_set_gemm_splits(0)
    plain = q.fp8_block_gemm(*ops)
    assert torch.equal(C0.view(torch.int16), plain.view(torch.int16))
    c32, S = oracle.gemm(*[host(t) for t in ops])
    assert_gemm_ok(to_f32(C2), c32, S, "two ranges in a small workspace")


def test_split_k_with_160_wide_tiles_runs_unsplit(q):
    """160-wide pair tiles have no split-K form: with that width forced, the
    workspace query says 0 bytes and fp8_block_gemm_ws gives the bits of
    fp8_block_gemm at that width; without pairs the call runs at another
    width and splits again."""
    host_ops = _random_operands(257, 576, 4096, 21)
    ops = _dev(*host_ops)
    ws = torch.randint(0, 256, (32 << 20,), dtype=torch.uint8, device=DEV)
    q.fp8q_set_gemm_tile_n(160)
    q.fp8q_set_gemm_splits(3)
    try:
        assert q.fp8_block_gemm_workspace_size(257, 576, 4096) == 0
        C = _run_ws(q, ops, ws).clone()
        plain = q.fp8_block_gemm(*ops)
        torch.cuda.synchronize()
        assert torch.equal(C.view(torch.int16), plain.view(torch.int16))
        q.fp8q_set_gemm_pairs(False)
        assert q.fp8_block_gemm_workspace_size(257, 576, 4096) > 0
        C1 = _run_ws(q, ops, ws)
    finally:
        q.fp8q_set_gemm_tile_n(0)
        q.fp8q_set_gemm_splits(0)
        q.fp8q_set_gemm_pairs(True)
    c32, S = oracle.gemm(*host_ops)
    assert_gemm_ok(to_f32(C), c32, S, "160 wide, split request ignored")
    assert_gemm_ok(to_f32(C1), c32, S, "one-CTA tiles, three ranges")


def _sampled_ws(q, A, W, name, n_rows=96, n_cols=48, seed=0):
    M, K = A.shape
    N = W.shape[0]
    qa, sa = q.fp8q_quant_act(A)
    qb, sb = q.fp8q_quant_weight(W)
    C = q.fp8_block_gemm_ws(qa, sa, qb, sb)
    torch.cuda.synchronize()
    assert q.fp8q_get_device_status() == 0
    oqa, osa = oracle.quant_act(bits(A))
    oqb, osb = oracle.quant_weight(bits(W))
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([np.arange(min(128, M)), np.arange(max(0, M - 128), M),
                                     rng.choice(M, size=n_rows, replace=False)]))
    cols = np.unique(np.concatenate([rng.choice(N, size=n_cols, replace=False),
                                     np.arange((N - 1) // 128 * 128, N)]))
    c32, S = oracle.gemm(oqa, osa, oqb, osb, rows=rows)
    assert_gemm_ok(host(C[torch.from_numpy(rows).to(DEV)].float()), c32, S, f"{name} rows")
    c32, S = oracle.gemm(oqa, osa, oqb, osb, cols=cols)
    assert_gemm_ok(host(C[:, torch.from_numpy(cols).to(DEV)].float()), c32, S, f"{name} columns")


@pytest.mark.slow
def test_split_k_mla_full_size(q):
    """The MLA projections at 4096 tokens with three K ranges forced (the
    automatic choice does not split there), and at 512 tokens, where it
    does."""
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.mla_down(seed=0, device=DEV)
    q.fp8q_set_gemm_splits(3)
    try:
        _sampled_ws(q, w.A, w.weights["Wq"], "split-K MLA Wq")
        _sampled_ws(q, w.A, w.weights["Wkv"], "split-K MLA Wkv")
        f = workloads.mla_down_fused(seed=0, device=DEV)
        _sampled_ws(q, f.A, f.weights["Wqkv"], "split-K MLA fused Wq||Wkv")
    finally:
        q.fp8q_set_gemm_splits(0)
    assert q.fp8_block_gemm_workspace_size(4096, 576, 7168) == 0
    assert q.fp8_block_gemm_workspace_size(512, 576, 7168) > 0, "no split chosen at 512 tokens"
    A = w.A[:512].contiguous()
    _sampled_ws(q, A, w.weights["Wkv"], "split-K MLA Wkv, 512 tokens", n_rows=64, n_cols=48)


def test_split_k_stalled_stage_times_out(q):
    """The injected never-completing first stage: the waits expire, the
    status reports the timeout, and the next split-K call on the same
    workspace is correct (the arrival words of the failed call are stale)."""
    host_ops = _random_operands(512, 512, 2048, 14)
    ops = _dev(*host_ops)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device=DEV)
    q.fp8q_set_gemm_splits(3)
    try:
        q.fp8q_set_wait_timeout_ns(20_000_000)
        q.fp8q_set_fault_injection(q.INJECT_STALLED_STAGE)
        q.fp8_block_gemm_ws(*ops, workspace=ws)
        assert q.fp8q_get_device_status() & q.DEVSTATUS_TIMEOUT
        q.fp8q_set_fault_injection(0)
        q.fp8q_set_wait_timeout_ns(0)
        C = _run_ws(q, ops, ws, guard=False)
    finally:
        q.fp8q_set_fault_injection(0)
        q.fp8q_set_wait_timeout_ns(0)
        q.fp8q_set_gemm_splits(0)
    c32, S = oracle.gemm(*host_ops)
    assert_gemm_ok(to_f32(C), c32, S, "split-K after an injected timeout")
