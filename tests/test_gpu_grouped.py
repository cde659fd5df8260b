"""GPU grouped (per-expert) block-scaled GEMM vs the CPU oracle: ragged
expert row ranges including empty experts and single rows, an N tail, the
device-side offsets check, and the full-size MoE workload (per-expert
samples)."""
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
    return mod


def _operands(sizes, N, K, seed):
    rng = np.random.default_rng(seed)
    E, M = len(sizes), int(sum(sizes))
    KB, NB = -(-K // 128), -(-N // 128)
    off = np.zeros(E + 1, np.int32)
    off[1:] = np.cumsum(sizes)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    sa = rng.uniform(0.01, 4.0, (M, KB)).astype(np.float32)
    qb = rng.choice(FINITE, size=(E, N, K)).astype(np.uint8)
    sb = rng.uniform(0.01, 4.0, (E, NB, KB)).astype(np.float32)
    return qa, sa, qb, sb, off


def _run(q, qa, sa, qb, sb, off):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    M, N = qa.shape[0], qb.shape[1]
    Cbuf = torch.full((M + 1, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    C = q.fp8_grouped_gemm(t(qa), t(sa), t(qb), t(sb), t(off), Cbuf[:M])
    status = q.fp8q_get_device_status()
    assert torch.all(torch.isnan(Cbuf[M])), "grouped GEMM wrote past the end of C"
    return C, status


@pytest.mark.parametrize("sizes,N,K", [
    ([100, 0, 200, 1], 256, 512),
    ([0, 1, 127, 128, 129, 255, 256, 300], 264, 400),
    ([513], 520, 272),
    ([0, 0, 7, 0], 16, 16),
    ([130] * 12, 256, 1024),
])
def test_grouped_full_output(q, sizes, N, K):
    qa, sa, qb, sb, off = _operands(sizes, N, K, sum(sizes) + N + K)
    C, status = _run(q, qa, sa, qb, sb, off)
    assert status == 0
    assert not np.isnan(to_f32(C)).any(), "unwritten outputs"
    c32, S = oracle.grouped_gemm(qa, sa, qb, sb, off, rows=np.arange(qa.shape[0]))
    assert_gemm_ok(to_f32(C), c32, S, f"grouped {sizes} N={N} K={K}")


def test_single_expert_matches_dense_bitwise(q):
    qa, sa, qb, sb, off = _operands([777], 512, 640, 3)
    C, _ = _run(q, qa, sa, qb, sb, off)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    D = q.fp8_block_gemm(t(qa), t(sa), t(qb[0]), t(sb[0]))
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), D.view(torch.int16))


@pytest.mark.parametrize("bad", ["decreasing", "first_nonzero", "last_mismatch"])
def test_malformed_offsets_are_reported_and_nothing_written(q, bad):
    qa, sa, qb, sb, off = _operands([64, 64, 64], 256, 256, 11)
    off = off.copy()
    if bad == "decreasing":
        off[1], off[2] = 100, 50
    elif bad == "first_nonzero":
        off[0] = 1
    else:
        off[3] = 150
    C, status = _run(q, qa, sa, qb, sb, off)
    assert status & q.DEVSTATUS_BAD_OFFSETS
    assert torch.all(torch.isnan(C.float())), "C written despite malformed offsets"


@pytest.mark.slow
def test_grouped_moe_full_size(q):
    """T=4096 tokens, 256 experts, top-8 (32768 routed rows), W [256, 2048,
    7168]: for every expert its first, last and two random rows, all 2048
    columns; empty experts produce no rows."""
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.moe_grouped(seed=0, device=DEV)
    W = w.weights["W"]
    qa, sa = q.fp8q_quant_act(w.A)
    qb, sb = q.fp8q_quant_weight(W)
    C = q.fp8_grouped_gemm(qa, sa, qb, sb, w.offsets)
    assert q.fp8q_get_device_status() == 0
    off = host(w.offsets).astype(np.int64)
    rng = np.random.default_rng(0)
    rows = []
    for e in range(len(off) - 1):
        lo, hi = off[e], off[e + 1]
        if hi > lo:
            rows += [lo, hi - 1] + list(rng.integers(lo, hi, 2))
    rows = np.unique(np.array(rows, dtype=np.int64))
    oqa, osa = oracle.quant_act(bits(w.A))
    oqb = np.empty(tuple(W.shape), np.uint8)
    osb = np.empty(tuple(sb.shape), np.float32)
    for e in range(W.shape[0]):  # per expert keeps host memory bounded
        oqb[e], osb[e] = oracle.quant_weight(bits(W[e]))
    c32, S = oracle.grouped_gemm(oqa, osa, oqb, osb, off.astype(np.int32), rows=rows)
    assert_gemm_ok(host(C[torch.from_numpy(rows).to(DEV)].float()), c32, S, "MoE grouped sampled")
