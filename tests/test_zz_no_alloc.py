"""fp8_block_gemm_static: the split-K GEMM for callers that cannot allocate
device memory (they may not call cudaMalloc where they issue the GEMM, or
they only receive their input and output buffers). It keeps its scratch in
a fixed array inside the library instead of a caller workspace.

Called here through the C ABI (ctypes), twice in a row on the same shape so
that the second call runs on the scratch contents the first one left; its
output is compared with fp8_block_gemm_ws on a caller workspace within the
GEMM acceptance bound (1 bf16 ulp + 1e-5 * sum_k |a_k b_k|). This file is
collected last so that a failure here does not stop the rest of the suite
in a run that stops at the first failure."""
import ctypes

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
    for reset in (lambda: mod.fp8q_set_gemm_splits(0), lambda: mod.fp8q_set_gemm_tile_n(0),
                  lambda: mod.fp8q_set_gemm_pairs(True)):
        reset()
    mod.fp8q_get_device_status()
    yield mod
    mod.fp8q_set_gemm_splits(0)


def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    qa = rng.choice(FINITE, size=(M, K)).astype(np.uint8)
    qb = rng.choice(FINITE, size=(N, K)).astype(np.uint8)
    sa = rng.uniform(0.01, 4.0, size=(M, -(-K // 128))).astype(np.float32)
    sb = rng.uniform(0.01, 4.0, size=(-(-N // 128), -(-K // 128))).astype(np.float32)
    return qa, sa, qb, sb


def _call_static(lib, dev_ops, C):
    """One call of the C entry point with raw device pointers."""
    qa, sa, qb, sb = dev_ops
    f = lib.fp8_block_gemm_static
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
    f.restype = ctypes.c_int
    M, K = qa.shape
    N = qb.shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    return f(qa.data_ptr(), sa.data_ptr(), qb.data_ptr(), sb.data_ptr(), C.data_ptr(), M, N, K, stream)


def _within_bound(c_test, c_ref, S, what):
    """|c_test - c_ref| <= 1 bf16 ulp(c_ref) + 1e-5 * S, elementwise."""
    ref = to_f32(c_ref).astype(np.float64)
    test = to_f32(c_test).astype(np.float64)
    mag = np.abs(ref)
    ulp = np.where(mag > 0, np.exp2(np.floor(np.log2(np.where(mag > 0, mag, 1.0))) - 7), 2.0 ** -133)
    bad = np.abs(test - ref) > ulp + 1e-5 * S
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs differ from fp8_block_gemm_ws beyond the bound"


@pytest.mark.parametrize("M,N,K,splits", [(512, 576, 7168, 0), (300, 520, 2048, 3)])
def test_static_scratch_gemm_matches_workspace_gemm(q, M, N, K, splits):
    """Automatic split count (512 x 576 x 7168 splits) and a forced one."""
    q.fp8q_set_gemm_splits(splits)
    host_ops = _operands(M, N, K, M + N + K)
    dev_ops = [torch.from_numpy(a).to(DEV) for a in host_ops]
    assert q.fp8_block_gemm_workspace_size(M, N, K) > 0, "the shape should split K"
    ref = q.fp8_block_gemm_ws(*dev_ops)
    torch.cuda.synchronize()
    c32, S = oracle.gemm(*host_ops)
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert _call_static(q.lib, dev_ops, C) == q.OK
        torch.cuda.synchronize()
        assert q.fp8q_get_device_status() == 0
        _within_bound(C, ref, S, f"static scratch call {call + 1} ({M}x{N}x{K})")
        assert_gemm_ok(to_f32(C), c32, S, f"static scratch call {call + 1} vs oracle")


def test_static_scratch_rejects_oversize_requests(q):
    """A split count whose partial tiles exceed the built-in array: an error,
    and nothing is written."""
    M, N, K = 4096, 7168, 1024
    q.fp8q_set_gemm_splits(4)
    dev_ops = [torch.from_numpy(a).to(DEV) for a in _operands(M, N, K, 5)]
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    assert _call_static(q.lib, dev_ops, C) == q.ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(C))
