"""Device-side failure detection without a GPU fault: a GEMM whose first
pipeline stage waits for 16 bytes that never arrive (a host-injected
expect-tx surplus) must hit its bounded wait, report FP8Q_DEVSTATUS_TIMEOUT,
return, and leave the CUDA context usable for the next correct call."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_gemm_ok, to_f32

pytestmark = pytest.mark.gpu

FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


@pytest.fixture
def q():
    from fp8_fine_grained_25_b300 import fp8q as mod
    mod.fp8q_get_device_status()
    yield mod
    mod.fp8q_set_fault_injection(0)
    mod.fp8q_set_wait_timeout_ns(0)
    mod.fp8q_set_gemm_pairs(True)
    mod.fp8q_set_gemm_tile_n(0)


def _ops(M, N, K, seed):
    rng = np.random.default_rng(seed)
    t = lambda a: torch.from_numpy(a).to(DEV)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.uniform(0.01, 2, (M, -(-K // 128))).astype(np.float32)
    sb = rng.uniform(0.01, 2, (-(-N // 128), -(-K // 128))).astype(np.float32)
    return (qa, sa, qb, sb), (t(qa), t(sa), t(qb), t(sb))


@pytest.mark.parametrize("bn", [0, 224])
@pytest.mark.parametrize("pairs", [True, False])
def test_stalled_stage_times_out_and_context_survives(q, pairs, bn):
    q.fp8q_set_gemm_pairs(pairs)
    q.fp8q_set_gemm_tile_n(bn)
    host, dev = _ops(512, 512, 1024, 1)
    q.fp8q_set_wait_timeout_ns(20_000_000)  # 20 ms per wait
    q.fp8q_set_fault_injection(q.INJECT_STALLED_STAGE)
    q.fp8_block_gemm(*dev)
    status = q.fp8q_get_device_status()
    assert status & q.DEVSTATUS_TIMEOUT
    # the same context computes the next call correctly
    q.fp8q_set_fault_injection(0)
    q.fp8q_set_wait_timeout_ns(0)
    C = q.fp8_block_gemm(*dev)
    assert q.fp8q_get_device_status() == 0
    c32, S = oracle.gemm(*host)
    assert_gemm_ok(to_f32(C), c32, S, "GEMM after an injected timeout")


def test_grouped_stalled_stage_times_out(q):
    rng = np.random.default_rng(3)
    t = lambda a: torch.from_numpy(a).to(DEV)
    off = np.array([0, 100, 300], np.int32)
    qa = rng.choice(FINITE, size=(300, 256)).astype(np.uint8)
    sa = np.ones((300, 2), np.float32)
    qb = rng.choice(FINITE, size=(2, 256, 256)).astype(np.uint8)
    sb = np.ones((2, 2, 2), np.float32)
    q.fp8q_set_wait_timeout_ns(20_000_000)
    q.fp8q_set_fault_injection(q.INJECT_STALLED_STAGE)
    q.fp8_grouped_gemm(t(qa), t(sa), t(qb), t(sb), t(off))
    assert q.fp8q_get_device_status() & q.DEVSTATUS_TIMEOUT
    q.fp8q_set_fault_injection(0)
    q.fp8q_set_wait_timeout_ns(0)
    C = q.fp8_grouped_gemm(t(qa), t(sa), t(qb), t(sb), t(off))
    assert q.fp8q_get_device_status() == 0
    c32, S = oracle.grouped_gemm(qa, sa, qb, sb, off, rows=np.arange(300))
    assert_gemm_ok(to_f32(C), c32, S, "grouped GEMM after an injected timeout")


@pytest.mark.parametrize("pairs", [True, False])
def test_wgrad_stalled_stage_times_out(q, pairs):
    # the row-scaled (weight-gradient) kernel shares the bounded waits; its
    # scale ring holds a slot until the slot's last K block, so a stall
    # there must unwind as well
    q.fp8q_set_gemm_pairs(pairs)
    rng = np.random.default_rng(5)
    t = lambda a: torch.from_numpy(a).to(DEV)
    M, N, K = 384, 256, 1024
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.uniform(0.01, 2, (M, K // 128)).astype(np.float32)
    sb = rng.uniform(0.01, 2, (N, K // 128)).astype(np.float32)
    q.fp8q_set_wait_timeout_ns(20_000_000)
    q.fp8q_set_fault_injection(q.INJECT_STALLED_STAGE)
    q.fp8_wgrad_gemm(t(qa), t(sa), t(qb), t(sb))
    assert q.fp8q_get_device_status() & q.DEVSTATUS_TIMEOUT
    q.fp8q_set_fault_injection(0)
    q.fp8q_set_wait_timeout_ns(0)
    C = q.fp8_wgrad_gemm(t(qa), t(sa), t(qb), t(sb))
    assert q.fp8q_get_device_status() == 0
    c32, S = oracle.wgrad_gemm(qa, sa, qb, sb)
    assert_gemm_ok(to_f32(C), c32, S, "weight-gradient GEMM after an injected timeout")


@pytest.mark.parametrize("pairs", [True, False])
def test_ue8m0_gemm_stalled_stage_times_out(q, pairs):
    # the hardware-scaled GEMM has its own pipeline (scale-factor ring in
    # tensor memory): a stalled stage must unwind it as well
    q.fp8q_set_gemm_pairs(pairs)
    rng = np.random.default_rng(8)
    t = lambda a: torch.from_numpy(a).to(DEV)
    M, N, K = 512, 448, 1024
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.integers(118, 136, size=(M, K // 128)).astype(np.uint8)
    sb = rng.integers(118, 136, size=(-(-N // 128), K // 128)).astype(np.uint8)
    q.fp8q_set_wait_timeout_ns(20_000_000)
    q.fp8q_set_fault_injection(q.INJECT_STALLED_STAGE)
    q.fp8_block_gemm_ue8m0(t(qa), t(sa), t(qb), t(sb))
    assert q.fp8q_get_device_status() & q.DEVSTATUS_TIMEOUT
    q.fp8q_set_fault_injection(0)
    q.fp8q_set_wait_timeout_ns(0)
    C = q.fp8_block_gemm_ue8m0(t(qa), t(sa), t(qb), t(sb))
    assert q.fp8q_get_device_status() == 0
    c32, S = oracle.gemm_ue8m0(qa, sa, qb, sb)
    assert_gemm_ok(to_f32(C), c32, S, "UE8M0 GEMM after an injected timeout")
