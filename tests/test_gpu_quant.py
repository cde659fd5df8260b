"""GPU quantizers vs the CPU oracle: codes and scales bit-exact, on small
ragged shapes, on edge-case tiles, and on the full-size workloads."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_codes_equal, assert_scales_equal, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    from fp8_fine_grained_25_b300 import fp8q as mod
    mod.fp8q_get_device_status()
    return mod


def _edge_rows(M, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g)
    if M > 1:
        x[1] = 0.0                                   # all-zero tiles
    if M > 2:
        x[2] = -0.0                                  # negative zeros only
    if M > 3:
        x[3] = 0.0
        x[3, ::128] = 3.0                            # spike tiles
    if M > 4:
        x[4] *= 1e-35                                # tiny values (scale near fp32 min)
    if M > 5:
        x[5] *= 1e30                                 # huge values
    if M > 6:
        codes = torch.randint(0, 126, (K,), generator=g, dtype=torch.int32)
        x[6] = torch.from_numpy(oracle.e4m3_decode(codes.numpy().astype(np.uint8))).float() * 2.0 ** -5
        x[6, ::128] = 448 * 2.0 ** -5                # grid values x a power of two
    if M > 7:
        x[7] = torch.randn(K, generator=g) * 2.0 ** -130  # bf16 subnormals
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("M,K", [(1, 16), (3, 128), (8, 208), (9, 384), (129, 1040),
                                 (64, 7168), (33, 7184)])
def test_quant_act_small(q, M, K):
    x = _edge_rows(M, K, M * 7 + K).to(DEV)
    qg, sg = q.fp8q_quant_act(x)
    qo, so = oracle.quant_act(bits(x))
    assert_scales_equal(sg, so, f"act scales {M}x{K}")
    assert_codes_equal(qg, qo, f"act codes {M}x{K}")


@pytest.mark.parametrize("N,K", [(1, 16), (8, 128), (200, 336), (256, 512), (576, 7168),
                                 (130, 7184)])
def test_quant_weight_small(q, N, K):
    x = (_edge_rows(N, K, N * 3 + K).float() * 0.01).to(torch.bfloat16).to(DEV)
    qg, sg = q.fp8q_quant_weight(x)
    qo, so = oracle.quant_weight(bits(x))
    assert_scales_equal(sg, so, f"weight scales {N}x{K}")
    assert_codes_equal(qg, qo, f"weight codes {N}x{K}")


def test_quant_does_not_write_outside_outputs(q):
    M, K = 5, 208
    x = torch.randn(M, K).to(torch.bfloat16).to(DEV)
    qbuf = torch.full((M + 1, K), 0xA5, dtype=torch.uint8, device=DEV)
    sbuf = torch.full((M + 1, 2), -7.0, dtype=torch.float32, device=DEV)
    q.fp8q_quant_act(x, qbuf[:M], sbuf[:M])
    torch.cuda.synchronize()
    assert torch.all(qbuf[M] == 0xA5) and torch.all(sbuf[M] == -7.0)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_quant_act_full_size(q, cfg):
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.WORKLOADS[cfg](seed=0, device=DEV)
    qg, sg = q.fp8q_quant_act(w.A)
    qo, so = oracle.quant_act(bits(w.A))
    assert_scales_equal(sg, so, f"config {cfg} act scales")
    assert_codes_equal(qg, qo, f"config {cfg} act codes")
    for name, W in w.weights.items():
        qg, sg = q.fp8q_quant_weight(W)
        qo, so = oracle.quant_weight(bits(W))
        assert_scales_equal(sg, so, f"config {cfg} {name} scales")
        assert_codes_equal(qg, qo, f"config {cfg} {name} codes")


@pytest.mark.slow
def test_quant_moe_full_size(q):
    """MoE workload: the gathered activations in full; the whole expert stack
    quantized in one call as [E*N, K], checked on a sample of experts."""
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.moe_grouped(seed=0, device=DEV)
    qg, sg = q.fp8q_quant_act(w.A)
    qo, so = oracle.quant_act(bits(w.A))
    assert_scales_equal(sg, so, "moe act scales")
    assert_codes_equal(qg, qo, "moe act codes")
    W = w.weights["W"]
    qw, sw = q.fp8q_quant_weight(W)
    for e in (0, 1, 77, 128, 255):
        qo, so = oracle.quant_weight(bits(W[e]))
        assert_scales_equal(sw[e], so, f"moe expert {e} scales")
        assert_codes_equal(qw[e], qo, f"moe expert {e} codes")
