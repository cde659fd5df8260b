"""Shared pieces of the GPU parity tests: run the CUDA path through the
binding, run the oracle on the same bytes, compare.

Codes and scales must be bit-identical. GEMM outputs must satisfy
|C_gpu - C_oracle_fp32| <= 1 bf16 ulp(C_oracle_fp32) + 1e-5 * sum_k |a_k b_k|
(the acceptance bound of the method's accuracy target)."""
from __future__ import annotations

import numpy as np
import torch

import oracle

DEV = "cuda:0"


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_codes_equal(q_gpu: torch.Tensor, q_ref: np.ndarray, what: str):
    qg = host(q_gpu.view(torch.uint8))
    if not np.array_equal(qg, q_ref):
        bad = np.argwhere(qg != q_ref)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} codes differ; first at {i}: "
                             f"gpu {qg[i]:#04x} oracle {q_ref[i]:#04x}")


def assert_scales_equal(s_gpu: torch.Tensor, s_ref: np.ndarray, what: str):
    sg = host(s_gpu)
    if not np.array_equal(sg.view(np.uint32), s_ref.view(np.uint32)):
        bad = np.argwhere(sg.view(np.uint32) != s_ref.view(np.uint32))
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} scales differ; first at {i}: "
                             f"gpu {sg[i]!r} oracle {s_ref[i]!r}")


def assert_gemm_ok(c_gpu_rows: np.ndarray, c32: np.ndarray, S: np.ndarray, what: str):
    ok, worst, idx = oracle.gemm_check(c_gpu_rows.astype(np.float64), c32, S)
    if not ok:
        raise AssertionError(f"{what}: outside tolerance, worst |err|/bound = {worst:.3g} at {idx}: "
                             f"gpu {c_gpu_rows[idx]!r} oracle {c32[idx]!r} S {S[idx]!r}")
    return worst


def to_f32(c_bf16: torch.Tensor) -> np.ndarray:
    return host(c_bf16.float())
