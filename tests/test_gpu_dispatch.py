"""FP8 dispatch: gathering quantized rows equals quantizing gathered rows, bit
for bit (1x128 tiles are row-local); the gather itself moves exactly the
selected rows; out-of-range indices are reported and give zero rows."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DEV, assert_codes_equal, assert_scales_equal, bits, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    from fp8_fine_grained_25_b300 import fp8q as mod
    mod.fp8q_get_device_status()
    return mod


@pytest.mark.parametrize("T,K,R", [(5, 16, 9), (64, 200 + 8, 300), (300, 7168, 1000), (7, 4096 + 16, 1)])
def test_gather_moves_the_selected_rows(q, T, K, R):
    g = torch.Generator().manual_seed(T + K + R)
    x = (torch.randn(T, K, generator=g)).to(torch.bfloat16).to(DEV)
    qx, sx = q.fp8q_quant_act(x)
    idx = torch.randint(0, T, (R,), generator=g, dtype=torch.int32).to(DEV)
    qd, sd = q.fp8q_gather_rows(qx, sx, idx)
    torch.cuda.synchronize()
    assert q.fp8q_get_device_status() == 0
    i = host(idx).astype(np.int64)
    assert np.array_equal(host(qd), host(qx)[i])
    assert np.array_equal(host(sd).view(np.uint32), host(sx).view(np.uint32)[i])


def test_bad_index_gives_zero_row_and_status(q):
    x = torch.randn(4, 256).to(torch.bfloat16).to(DEV)
    qx, sx = q.fp8q_quant_act(x)
    idx = torch.tensor([1, 4, -1, 3], dtype=torch.int32, device=DEV)
    qd, sd = q.fp8q_gather_rows(qx, sx, idx)
    assert q.fp8q_get_device_status() & q.DEVSTATUS_BAD_INDEX
    assert np.array_equal(host(qd[0]), host(qx[1])) and np.array_equal(host(qd[3]), host(qx[3]))
    assert not host(qd[1]).any() and not host(qd[2]).any() and not host(sd[1:3]).any()


@pytest.mark.slow
def test_moe_dispatch_equals_quantizing_gathered_rows(q):
    """The MoE workload (4096 tokens, 32768 routed rows): quantize-then-gather
    matches the oracle's quantization of the gathered bf16 rows."""
    from fp8_fine_grained_25_b300 import workloads
    w = workloads.moe_dispatch_fp8(seed=0, device=DEV)
    qx, sx = q.fp8q_quant_act(w.tokens)
    qd, sd = q.fp8q_gather_rows(qx, sx, w.index)
    torch.cuda.synchronize()
    qo, so = oracle.quant_act(bits(w.A))
    assert_scales_equal(sd, so, "dispatched scales")
    assert_codes_equal(qd, qo, "dispatched codes")
