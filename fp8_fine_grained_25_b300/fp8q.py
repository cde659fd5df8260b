"""Python binding of libfp8q.so: the C-ABI entry points of include/fp8q.h
under the same names, taking torch CUDA tensors.

This module only marshals arguments (shapes, pointers, the current CUDA
stream) and, where an output is not given, allocates it with torch. Every
step of the computation runs in the library's CUDA kernels; there is no
other implementation behind these names. Importing this module fails if
the library has not been built (``python -m fp8_fine_grained_25_b300.build``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfp8q.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with "
                      "`python -m fp8_fine_grained_25_b300.build` (nvcc, sm_103a)")

lib = ctypes.CDLL(_LIB_PATH)
_i64, _i32, _p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
lib.fp8q_quant_act.argtypes = [_p, _i64, _i64, _p, _p, _p]
lib.fp8q_quant_weight.argtypes = [_p, _i64, _i64, _p, _p, _p]
lib.fp8q_quant_act_t.argtypes = [_p, _i64, _i64, _p, _p, _p]
lib.fp8q_quant_act_ue8m0.argtypes = [_p, _i64, _i64, _p, _p, _p]
lib.fp8q_quant_weight_ue8m0.argtypes = [_p, _i64, _i64, _p, _p, _p]
lib.fp8q_quant_weight_t.argtypes = [_p, _i64, _i64, _p, _p, _p, _p, _p]
lib.fp8_block_gemm.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p]
lib.fp8_block_gemm_ws.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p, ctypes.c_size_t, _p]
lib.fp8_block_gemm_workspace_size.argtypes = [_i64, _i64, _i64, ctypes.POINTER(ctypes.c_size_t)]
lib.fp8_block_gemm_static.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p]
lib.fp8q_set_gemm_splits.argtypes = [ctypes.c_int]
lib.fp8q_set_gemm_splits.restype = ctypes.c_int
lib.fp8_wgrad_gemm.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p]
lib.fp8_block_gemm_ue8m0.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p]
lib.fp8_wgrad_gemm_ue8m0.argtypes = [_p, _p, _p, _p, _p, _i64, _i64, _i64, _p]
lib.fp8q_quant_act_t_ue8m0.argtypes = [_p, _i64, _i64, _p, _p, _p]
lib.fp8q_quant_weight_t_ue8m0.argtypes = [_p, _i64, _i64, _p, _p, _p, _p, _p]
lib.fp8q_gather_rows.argtypes = [_p, _p, _i64, _i64, _p, _i64, _p, _p, _p]
lib.fp8q_gather_rows.restype = ctypes.c_int
lib.fp8_grouped_gemm.argtypes = [_p, _p, _p, _p, _p, _p, _i32, _i64, _i64, _i64, _p]
lib.fp8q_get_device_status.argtypes = [_p, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
lib.fp8q_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
lib.fp8q_set_wait_timeout_ns.restype = None
lib.fp8q_set_gemm_tile_n.argtypes = [ctypes.c_int]
lib.fp8q_set_gemm_tile_n.restype = ctypes.c_int
lib.fp8q_set_gemm_pairs.argtypes = [ctypes.c_int]
lib.fp8q_set_gemm_pairs.restype = ctypes.c_int
lib.fp8q_set_fault_injection.argtypes = [ctypes.c_uint32]
lib.fp8q_set_fault_injection.restype = ctypes.c_int
lib.fp8q_status_string.argtypes = [ctypes.c_int]
lib.fp8q_status_string.restype = ctypes.c_char_p
for _f in ("fp8q_quant_act", "fp8q_quant_weight", "fp8q_quant_act_t", "fp8q_quant_weight_t",
           "fp8q_quant_act_ue8m0", "fp8q_quant_weight_ue8m0",
           "fp8_block_gemm", "fp8_block_gemm_ws", "fp8_block_gemm_workspace_size", "fp8_block_gemm_static",
           "fp8_wgrad_gemm", "fp8_block_gemm_ue8m0", "fp8_wgrad_gemm_ue8m0",
           "fp8q_quant_act_t_ue8m0", "fp8q_quant_weight_t_ue8m0", "fp8_grouped_gemm",
           "fp8q_get_device_status"):
    getattr(lib, _f).restype = ctypes.c_int

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DEVICE, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED, ERR_OFFSETS = range(9)
DEVSTATUS_TIMEOUT = 0x1
DEVSTATUS_BAD_OFFSETS = 0x2
DEVSTATUS_BAD_INDEX = 0x4
INJECT_STALLED_STAGE = 0x1

CODE_DTYPES = (torch.uint8, torch.float8_e4m3fn)


class FP8QError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fp8q_status_string(status)} (status {status})")


def fp8q_status_string(status: int) -> str:
    return lib.fp8q_status_string(int(status)).decode()


def _check(rc: int, where: str) -> None:
    if rc != OK:
        raise FP8QError(rc, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, dtypes, shape) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def fp8q_quant_act(x: torch.Tensor, q: torch.Tensor | None = None,
                   scales: torch.Tensor | None = None, stream=None):
    """1x128-tile quantization of bf16 activations x [M, K] -> (q uint8 [M, K],
    scales fp32 [M, ceil(K/128)])."""
    M, K = x.shape
    _need(x, "x", (torch.bfloat16,), None)
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((M, _cdiv(K, 128)), dtype=torch.float32, device=x.device)
    _need(q, "q", CODE_DTYPES, (M, K))
    _need(scales, "scales", (torch.float32,), (M, _cdiv(K, 128)))
    _check(lib.fp8q_quant_act(x.data_ptr(), M, K, q.data_ptr(), scales.data_ptr(), _stream(stream)),
           "fp8q_quant_act")
    return q, scales


def fp8q_quant_weight(w: torch.Tensor, q: torch.Tensor | None = None,
                      scales: torch.Tensor | None = None, stream=None):
    """128x128-block quantization of bf16 weights w [N, K] (or a stack
    [E, N, K] with N % 128 == 0) -> (q uint8, scales fp32 [.., ceil(N/128), ceil(K/128)])."""
    _need(w, "w", (torch.bfloat16,), None)
    shape = tuple(w.shape)
    if len(shape) == 3:
        E, N, K = shape
        if N % 128:
            raise ValueError("a weight stack needs N % 128 == 0")
        rows, sshape = E * N, (E, N // 128, _cdiv(K, 128))
    else:
        N, K = shape
        rows, sshape = N, (_cdiv(N, 128), _cdiv(K, 128))
    if q is None:
        q = torch.empty(shape, dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty(sshape, dtype=torch.float32, device=w.device)
    _need(q, "q", CODE_DTYPES, shape)
    _need(scales, "scales", (torch.float32,), sshape)
    _check(lib.fp8q_quant_weight(w.data_ptr(), rows, K, q.data_ptr(), scales.data_ptr(),
                                 _stream(stream)), "fp8q_quant_weight")
    return q, scales


def fp8q_quant_act_ue8m0(x: torch.Tensor, q: torch.Tensor | None = None,
                         scales: torch.Tensor | None = None, stream=None):
    """1x128 tiles with power-of-two (UE8M0) scales -> (q uint8 [M, K], scale
    bytes uint8 [M, ceil(K/128)]; the scale is 2^(byte - 127))."""
    M, K = x.shape
    _need(x, "x", (torch.bfloat16,), None)
    if q is None:
        q = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((M, _cdiv(K, 128)), dtype=torch.uint8, device=x.device)
    _need(q, "q", CODE_DTYPES, (M, K))
    _need(scales, "scales", (torch.uint8,), (M, _cdiv(K, 128)))
    _check(lib.fp8q_quant_act_ue8m0(x.data_ptr(), M, K, q.data_ptr(), scales.data_ptr(),
                                    _stream(stream)), "fp8q_quant_act_ue8m0")
    return q, scales


def fp8q_quant_weight_ue8m0(w: torch.Tensor, q: torch.Tensor | None = None,
                            scales: torch.Tensor | None = None, stream=None):
    """128x128 blocks with power-of-two (UE8M0) scales -> (q uint8 [N, K], scale
    bytes uint8 [ceil(N/128), ceil(K/128)])."""
    N, K = w.shape
    _need(w, "w", (torch.bfloat16,), None)
    if q is None:
        q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((_cdiv(N, 128), _cdiv(K, 128)), dtype=torch.uint8, device=w.device)
    _need(q, "q", CODE_DTYPES, (N, K))
    _need(scales, "scales", (torch.uint8,), (_cdiv(N, 128), _cdiv(K, 128)))
    _check(lib.fp8q_quant_weight_ue8m0(w.data_ptr(), N, K, q.data_ptr(), scales.data_ptr(),
                                       _stream(stream)), "fp8q_quant_weight_ue8m0")
    return q, scales


def fp8q_quant_act_t(x: torch.Tensor, qt: torch.Tensor | None = None,
                     st: torch.Tensor | None = None, stream=None):
    """128x1-tile quantization of bf16 activations x [M, K] (M tokens), written
    transposed -> (qt uint8 [K, M], st fp32 [K, ceil(M/128)]): the operand
    layout of fp8_wgrad_gemm."""
    M, K = x.shape
    _need(x, "x", (torch.bfloat16,), None)
    if qt is None:
        qt = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    if st is None:
        st = torch.empty((K, _cdiv(M, 128)), dtype=torch.float32, device=x.device)
    _need(qt, "qt", CODE_DTYPES, (K, M))
    _need(st, "st", (torch.float32,), (K, _cdiv(M, 128)))
    _check(lib.fp8q_quant_act_t(x.data_ptr(), M, K, qt.data_ptr(), st.data_ptr(), _stream(stream)),
           "fp8q_quant_act_t")
    return qt, st


def fp8q_quant_weight_t(w: torch.Tensor, q: torch.Tensor | None = None,
                        scales: torch.Tensor | None = None, qt: torch.Tensor | None = None,
                        st: torch.Tensor | None = None, with_forward: bool = True, stream=None):
    """128x128-block quantization of bf16 weights w [N, K] in both layouts ->
    (q [N, K], s [NB, KB], qt [K, N], st [KB, NB]); with_forward=False skips
    q and s (returned as None)."""
    _need(w, "w", (torch.bfloat16,), None)
    N, K = w.shape
    NB, KB = _cdiv(N, 128), _cdiv(K, 128)
    dev = w.device
    if with_forward:
        q = torch.empty((N, K), dtype=torch.uint8, device=dev) if q is None else q
        scales = torch.empty((NB, KB), dtype=torch.float32, device=dev) if scales is None else scales
        _need(q, "q", CODE_DTYPES, (N, K))
        _need(scales, "scales", (torch.float32,), (NB, KB))
    else:
        q = scales = None
    qt = torch.empty((K, N), dtype=torch.uint8, device=dev) if qt is None else qt
    st = torch.empty((KB, NB), dtype=torch.float32, device=dev) if st is None else st
    _need(qt, "qt", CODE_DTYPES, (K, N))
    _need(st, "st", (torch.float32,), (KB, NB))
    _check(lib.fp8q_quant_weight_t(w.data_ptr(), N, K, q.data_ptr() if q is not None else None,
                                   scales.data_ptr() if scales is not None else None,
                                   qt.data_ptr(), st.data_ptr(), _stream(stream)),
           "fp8q_quant_weight_t")
    return q, scales, qt, st


def fp8q_quant_act_t_ue8m0(x: torch.Tensor, qt: torch.Tensor | None = None,
                           st: torch.Tensor | None = None, stream=None):
    """128x1 tiles with UE8M0 scales, written transposed -> (qt uint8 [K, M],
    st uint8 [K, ceil(M/128)])."""
    M, K = x.shape
    _need(x, "x", (torch.bfloat16,), None)
    if qt is None:
        qt = torch.empty((K, M), dtype=torch.uint8, device=x.device)
    if st is None:
        st = torch.empty((K, _cdiv(M, 128)), dtype=torch.uint8, device=x.device)
    _need(qt, "qt", CODE_DTYPES, (K, M))
    _need(st, "st", (torch.uint8,), (K, _cdiv(M, 128)))
    _check(lib.fp8q_quant_act_t_ue8m0(x.data_ptr(), M, K, qt.data_ptr(), st.data_ptr(), _stream(stream)),
           "fp8q_quant_act_t_ue8m0")
    return qt, st


def fp8q_quant_weight_t_ue8m0(w: torch.Tensor, q: torch.Tensor | None = None,
                              scales: torch.Tensor | None = None, qt: torch.Tensor | None = None,
                              st: torch.Tensor | None = None, with_forward: bool = True, stream=None):
    """128x128 UE8M0 blocks in both layouts -> (q [N, K], s uint8 [NB, KB],
    qt [K, N], st uint8 [KB, NB]); with_forward=False skips q and s."""
    _need(w, "w", (torch.bfloat16,), None)
    N, K = w.shape
    NB, KB = _cdiv(N, 128), _cdiv(K, 128)
    dev = w.device
    if with_forward:
        q = torch.empty((N, K), dtype=torch.uint8, device=dev) if q is None else q
        scales = torch.empty((NB, KB), dtype=torch.uint8, device=dev) if scales is None else scales
        _need(q, "q", CODE_DTYPES, (N, K))
        _need(scales, "scales", (torch.uint8,), (NB, KB))
    else:
        q = scales = None
    qt = torch.empty((K, N), dtype=torch.uint8, device=dev) if qt is None else qt
    st = torch.empty((KB, NB), dtype=torch.uint8, device=dev) if st is None else st
    _need(qt, "qt", CODE_DTYPES, (K, N))
    _need(st, "st", (torch.uint8,), (KB, NB))
    _check(lib.fp8q_quant_weight_t_ue8m0(w.data_ptr(), N, K, q.data_ptr() if q is not None else None,
                                         scales.data_ptr() if scales is not None else None,
                                         qt.data_ptr(), st.data_ptr(), _stream(stream)),
           "fp8q_quant_weight_t_ue8m0")
    return q, scales, qt, st


def fp8q_gather_rows(q_src: torch.Tensor, s_src: torch.Tensor, index: torch.Tensor,
                     q_dst: torch.Tensor | None = None, s_dst: torch.Tensor | None = None,
                     stream=None):
    """Rows index[r] of quantized activations (codes [T, K], scales [T, KB])
    -> (codes [R, K], scales [R, KB]): the MoE dispatch in FP8."""
    T, K = q_src.shape
    R = index.shape[0]
    KB = _cdiv(K, 128)
    _need(q_src, "q_src", CODE_DTYPES, (T, K))
    _need(s_src, "s_src", (torch.float32,), (T, KB))
    _need(index, "index", (torch.int32,), (R,))
    if q_dst is None:
        q_dst = torch.empty((R, K), dtype=q_src.dtype, device=q_src.device)
    if s_dst is None:
        s_dst = torch.empty((R, KB), dtype=torch.float32, device=q_src.device)
    _need(q_dst, "q_dst", CODE_DTYPES, (R, K))
    _need(s_dst, "s_dst", (torch.float32,), (R, KB))
    _check(lib.fp8q_gather_rows(q_src.data_ptr(), s_src.data_ptr(), T, K, index.data_ptr(), R,
                                q_dst.data_ptr(), s_dst.data_ptr(), _stream(stream)),
           "fp8q_gather_rows")
    return q_dst, s_dst


def fp8_block_gemm(A: torch.Tensor, sa: torch.Tensor, B: torch.Tensor, sb: torch.Tensor,
                   C: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C[M, N] (bf16) = block-scaled A[M, K] * B[N, K]^T."""
    M, K = A.shape
    N = B.shape[0]
    _need(A, "A", CODE_DTYPES, (M, K))
    _need(B, "B", CODE_DTYPES, (N, K))
    _need(sa, "sa", (torch.float32,), (M, _cdiv(K, 128)))
    _need(sb, "sb", (torch.float32,), (_cdiv(N, 128), _cdiv(K, 128)))
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(C, "C", (torch.bfloat16,), (M, N))
    _check(lib.fp8_block_gemm(A.data_ptr(), sa.data_ptr(), B.data_ptr(), sb.data_ptr(),
                              C.data_ptr(), M, N, K, _stream(stream)), "fp8_block_gemm")
    return C


def fp8_block_gemm_workspace_size(M: int, N: int, K: int) -> int:
    """Bytes of workspace fp8_block_gemm_ws uses for an M x N x K call on the
    current device (0: it would not split K)."""
    n = ctypes.c_size_t(0)
    _check(lib.fp8_block_gemm_workspace_size(int(M), int(N), int(K), ctypes.byref(n)),
           "fp8_block_gemm_workspace_size")
    return int(n.value)


def fp8_block_gemm_ws(A: torch.Tensor, sa: torch.Tensor, B: torch.Tensor, sb: torch.Tensor,
                      C: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """fp8_block_gemm with split K through a caller-owned workspace (a uint8
    CUDA tensor; allocated here at the size fp8_block_gemm_workspace_size
    gives when not passed)."""
    M, K = A.shape
    N = B.shape[0]
    _need(A, "A", CODE_DTYPES, (M, K))
    _need(B, "B", CODE_DTYPES, (N, K))
    _need(sa, "sa", (torch.float32,), (M, _cdiv(K, 128)))
    _need(sb, "sb", (torch.float32,), (_cdiv(N, 128), _cdiv(K, 128)))
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(C, "C", (torch.bfloat16,), (M, N))
    if workspace is None:
        workspace = torch.empty(max(256, fp8_block_gemm_workspace_size(M, N, K)), dtype=torch.uint8,
                                device=A.device)
    _need(workspace, "workspace", (torch.uint8,), None)
    _check(lib.fp8_block_gemm_ws(A.data_ptr(), sa.data_ptr(), B.data_ptr(), sb.data_ptr(), C.data_ptr(),
                                 M, N, K, workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "fp8_block_gemm_ws")
    return C


def fp8_block_gemm_static(A: torch.Tensor, sa: torch.Tensor, B: torch.Tensor, sb: torch.Tensor,
                          C: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fp8_block_gemm_ws with the library's built-in scratch array instead of a
    workspace: for callers that cannot allocate device memory (the C entry
    point allocates nothing; only C is allocated here when not passed)."""
    M, K = A.shape
    N = B.shape[0]
    _need(A, "A", CODE_DTYPES, (M, K))
    _need(B, "B", CODE_DTYPES, (N, K))
    _need(sa, "sa", (torch.float32,), (M, _cdiv(K, 128)))
    _need(sb, "sb", (torch.float32,), (_cdiv(N, 128), _cdiv(K, 128)))
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(C, "C", (torch.bfloat16,), (M, N))
    _check(lib.fp8_block_gemm_static(A.data_ptr(), sa.data_ptr(), B.data_ptr(), sb.data_ptr(), C.data_ptr(),
                                     M, N, K, _stream(stream)), "fp8_block_gemm_static")
    return C


def fp8_wgrad_gemm(A: torch.Tensor, sa: torch.Tensor, B: torch.Tensor, sb: torch.Tensor,
                   C: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C[M, N] (bf16) = A[M, K] * B[N, K]^T with one scale per row of each
    operand per 128-wide K block (sa [M, KB], sb [N, KB]): the weight
    gradient dW = dY^T X from fp8q_quant_act_t(dY) and fp8q_quant_act_t(X)."""
    M, K = A.shape
    N = B.shape[0]
    _need(A, "A", CODE_DTYPES, (M, K))
    _need(B, "B", CODE_DTYPES, (N, K))
    _need(sa, "sa", (torch.float32,), (M, _cdiv(K, 128)))
    _need(sb, "sb", (torch.float32,), (N, _cdiv(K, 128)))
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(C, "C", (torch.bfloat16,), (M, N))
    _check(lib.fp8_wgrad_gemm(A.data_ptr(), sa.data_ptr(), B.data_ptr(), sb.data_ptr(),
                              C.data_ptr(), M, N, K, _stream(stream)), "fp8_wgrad_gemm")
    return C


def fp8_block_gemm_ue8m0(A: torch.Tensor, sa: torch.Tensor, B: torch.Tensor, sb: torch.Tensor,
                         C: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C[M, N] (bf16) = A[M, K] * B[N, K]^T with UE8M0 scale bytes (sa [M, KB],
    sb [NB, KB]) applied by the tensor core."""
    M, K = A.shape
    N = B.shape[0]
    _need(A, "A", CODE_DTYPES, (M, K))
    _need(B, "B", CODE_DTYPES, (N, K))
    _need(sa, "sa", (torch.uint8,), (M, _cdiv(K, 128)))
    _need(sb, "sb", (torch.uint8,), (_cdiv(N, 128), _cdiv(K, 128)))
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(C, "C", (torch.bfloat16,), (M, N))
    _check(lib.fp8_block_gemm_ue8m0(A.data_ptr(), sa.data_ptr(), B.data_ptr(), sb.data_ptr(),
                                    C.data_ptr(), M, N, K, _stream(stream)), "fp8_block_gemm_ue8m0")
    return C


def fp8_wgrad_gemm_ue8m0(A: torch.Tensor, sa: torch.Tensor, B: torch.Tensor, sb: torch.Tensor,
                         C: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C[M, N] (bf16) = A[M, K] * B[N, K]^T with one UE8M0 byte per row of A
    and of B per 128-wide K block (sa [M, KB], sb [N, KB])."""
    M, K = A.shape
    N = B.shape[0]
    _need(A, "A", CODE_DTYPES, (M, K))
    _need(B, "B", CODE_DTYPES, (N, K))
    _need(sa, "sa", (torch.uint8,), (M, _cdiv(K, 128)))
    _need(sb, "sb", (torch.uint8,), (N, _cdiv(K, 128)))
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(C, "C", (torch.bfloat16,), (M, N))
    _check(lib.fp8_wgrad_gemm_ue8m0(A.data_ptr(), sa.data_ptr(), B.data_ptr(), sb.data_ptr(),
                                    C.data_ptr(), M, N, K, _stream(stream)), "fp8_wgrad_gemm_ue8m0")
    return C


def fp8_grouped_gemm(A: torch.Tensor, sa: torch.Tensor, B: torch.Tensor, sb: torch.Tensor,
                     expert_offsets: torch.Tensor, C: torch.Tensor | None = None,
                     total_M: int | None = None, stream=None) -> torch.Tensor:
    """Grouped GEMM: rows [off[e], off[e+1]) of A use expert e of B [E, N, K].

    ``total_M`` defaults to A.shape[0] (the offsets stay on the device)."""
    M, K = A.shape
    E, N, Kb = B.shape
    if Kb != K:
        raise ValueError("A and B disagree on K")
    total_M = M if total_M is None else int(total_M)
    _need(A, "A", CODE_DTYPES, (M, K))
    _need(B, "B", CODE_DTYPES, (E, N, K))
    _need(sa, "sa", (torch.float32,), (M, _cdiv(K, 128)))
    _need(sb, "sb", (torch.float32,), (E, _cdiv(N, 128), _cdiv(K, 128)))
    _need(expert_offsets, "expert_offsets", (torch.int32,), (E + 1,))
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _need(C, "C", (torch.bfloat16,), (M, N))
    _check(lib.fp8_grouped_gemm(A.data_ptr(), sa.data_ptr(), B.data_ptr(), sb.data_ptr(),
                                C.data_ptr(), expert_offsets.data_ptr(), E, total_M, N, K,
                                _stream(stream)), "fp8_grouped_gemm")
    return C


def fp8q_get_device_status(stream=None, clear: bool = True) -> int:
    """Synchronize the stream and return (and by default clear) the device
    status word (DEVSTATUS_* bits)."""
    out = ctypes.c_uint32(0)
    _check(lib.fp8q_get_device_status(_stream(stream), ctypes.byref(out), int(bool(clear))),
           "fp8q_get_device_status")
    return out.value


def fp8q_set_wait_timeout_ns(ns: int) -> None:
    lib.fp8q_set_wait_timeout_ns(int(ns))


def fp8q_set_gemm_tile_n(bn: int) -> None:
    """Force the dense GEMM's output-tile width (128, 160, 224 or 256; 0 =
    automatic; 160 and 224 apply to the block-scaled GEMM, the weight-gradient
    GEMM runs 256; 160 to pair tiles only, without split K)."""
    _check(lib.fp8q_set_gemm_tile_n(int(bn)), "fp8q_set_gemm_tile_n")


def fp8q_set_gemm_splits(splits: int) -> None:
    """Force the number of K ranges of fp8_block_gemm_ws (1 .. 8; 0 = automatic)."""
    _check(lib.fp8q_set_gemm_splits(int(splits)), "fp8q_set_gemm_splits")


def fp8q_set_gemm_pairs(enable: bool) -> None:
    """Allow (default) or forbid 2-SM pair tiles in the dense GEMM."""
    _check(lib.fp8q_set_gemm_pairs(int(bool(enable))), "fp8q_set_gemm_pairs")


def fp8q_set_fault_injection(flags: int) -> None:
    """Test hook: INJECT_STALLED_STAGE makes every GEMM launch time out (see
    include/fp8q.h); 0 turns it off."""
    _check(lib.fp8q_set_fault_injection(int(flags)), "fp8q_set_fault_injection")
