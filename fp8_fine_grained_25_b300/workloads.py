"""Seeded synthetic inputs shaped like the layers the pages describe.

This module only draws random tensors (torch generators) and arranges them;
it holds none of the quantization or GEMM arithmetic. The same bytes feed
both the CUDA path and the CPU oracle in the tests.

Shapes come from the pages (news.qq.com/rain/a/20241229A05OQF00, "Multi-head
Latent Attention": KV compression 512, query compression 1536, decoupled key
dim 64; "DeepSeekMoE 架构": 256 routed experts, top-8; the aliyun article's
model table: hidden size 7168). The expert intermediate size (2048), the
value distributions, the outlier scheme and the token counts are synthetic
choices of this repository; no dataset or trained weight is involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

HIDDEN = 7168
MLA_Q_RANK = 1536
MLA_KV_RANK = 512
MLA_ROPE_DIM = 64
N_ROUTED = 256
TOP_K = 8
EXPERT_DIM = 2048


def _gen(device, seed: int) -> torch.Generator:
    return torch.Generator(device=device).manual_seed(int(seed))


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) samples drawn in fp32 and rounded to bf16."""
    x = torch.randn(*shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def activations_with_outliers(M: int, K: int, seed: int, device="cpu",
                              frac: float = 0.001, gain: float = 100.0) -> torch.Tensor:
    """N(0,1) activations where floor(frac * K) channels, chosen by a seeded
    permutation, are multiplied by `gain` (heavy-tailed outlier channels)."""
    g = _gen(device, seed)
    x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    n = int(frac * K)
    if n > 0:
        idx = torch.randperm(K, generator=g, device=device)[:n]
        x[:, idx] *= gain
    return x.to(torch.bfloat16)


def moe_routing(T: int, E: int, top_k: int, seed: int, device="cpu"):
    """Top-k routing from sigmoid(N(0,1) token-expert scores) plus a per-expert
    bias ~ U(-0.1, 0.1) (the bias only steers selection, as in the pages'
    auxiliary-loss-free balancing). Returns (token index of each routed row
    sorted stably by expert [T*top_k] int64, expert offsets [E+1] int32)."""
    g = _gen(device, seed)
    scores = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    bias = torch.rand(E, generator=g, device=device, dtype=torch.float32) * 0.2 - 0.1
    sel = torch.topk(torch.sigmoid(scores) + bias, top_k, dim=1).indices  # [T, k]
    expert = sel.reshape(-1)
    token = torch.arange(T, device=device).repeat_interleave(top_k)
    order = torch.sort(expert, stable=True).indices
    counts = torch.bincount(expert, minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int64, device=device)
    offsets[1:] = torch.cumsum(counts, 0)
    return token[order], offsets.to(torch.int32)


@dataclass
class Workload:
    name: str
    A: torch.Tensor                       # bf16 activations [M, K] (grouped: gathered rows)
    weights: dict = field(default_factory=dict)  # name -> bf16 [N, K] or [E, N, K]
    offsets: torch.Tensor | None = None   # int32 [E+1] for the grouped GEMM
    note: str = ""
    tokens: torch.Tensor | None = None    # MoE: the un-gathered token activations [T, K]
    index: torch.Tensor | None = None     # MoE: int32 token of each routed row (A = tokens[index])
    X: torch.Tensor | None = None         # backward: the layer input [T, K] (A holds dY [T, N])
    scales: str = "fp32"                  # "fp32" (amax / 448) or "ue8m0" (powers of two)


def tiny(seed: int = 0, device="cpu") -> Workload:
    """A [128, 512] ~ N(0,1), B [256, 512] ~ N(0, 0.02^2)."""
    return Workload("tiny 128x256x512",
                    normal_bf16((128, 512), 1.0, seed * 1000 + 1, device),
                    {"B": normal_bf16((256, 512), 0.02, seed * 1000 + 2, device)})


def mla_down(seed: int = 0, device="cpu", tokens: int = 4096) -> Workload:
    """MLA down-projections: A [tokens, 7168] ~ N(0,1); Wq [1536, 7168] and
    Wkv [576 = 512 + 64, 7168] ~ N(0, 0.006^2)."""
    return Workload(f"MLA down-proj {tokens}x{{1536,576}}x7168",
                    normal_bf16((tokens, HIDDEN), 1.0, seed * 1000 + 1, device),
                    {"Wq": normal_bf16((MLA_Q_RANK, HIDDEN), 0.006, seed * 1000 + 2, device),
                     "Wkv": normal_bf16((MLA_KV_RANK + MLA_ROPE_DIM, HIDDEN), 0.006,
                                        seed * 1000 + 3, device)})


def mla_down_fused(seed: int = 0, device="cpu", tokens: int = 4096) -> Workload:
    """The MLA down-projections as one GEMM: the same A and the same Wq, Wkv
    draws as mla_down, with the weights stacked row-wise into Wq‖Wkv
    [2112, 7168]. 1536 is a multiple of 128, so the 128x128 weight blocks and
    their scales are those of the two separate weights, and the output's
    columns [0, 1536) and [1536, 2112) are the two projections."""
    w = mla_down(seed, device, tokens)
    Wqkv = torch.cat([w.weights["Wq"], w.weights["Wkv"]], dim=0)
    return Workload(f"MLA down-proj fused {tokens}x2112x7168 (Wq||Wkv)", w.A, {"Wqkv": Wqkv})


def dense_square(seed: int = 0, device="cpu", M: int = 8192) -> Workload:
    """A [M, 7168] ~ N(0,1) with 0.1% outlier channels x100; B [7168, 7168]
    ~ N(0, 0.01^2)."""
    return Workload(f"dense {M}x7168x7168",
                    activations_with_outliers(M, HIDDEN, seed * 1000 + 1, device),
                    {"B": normal_bf16((HIDDEN, HIDDEN), 0.01, seed * 1000 + 2, device)})


def moe_grouped(seed: int = 0, device="cpu", T: int = 4096, E: int = N_ROUTED,
                N: int = EXPERT_DIM, top_k: int = TOP_K, K: int = HIDDEN) -> Workload:
    """T tokens X [T, K] ~ N(0,1), routed top-k over E experts; the routed rows
    are gathered in expert order into A [T*top_k, K]; expert weights
    W [E, N, K] ~ N(0, 0.01^2)."""
    X = normal_bf16((T, K), 1.0, seed * 1000 + 1, device)
    token, offsets = moe_routing(T, E, top_k, seed * 1000 + 2, device)
    W = torch.empty((E, N, K), dtype=torch.bfloat16, device=device)
    for e in range(E):  # per expert, to bound the fp32 scratch
        W[e] = normal_bf16((N, K), 0.01, seed * 1000 + 10 + e, device)
    return Workload(f"MoE grouped T={T} E={E} top{top_k} {N}x{K}", X[token], {"W": W},
                    offsets, note="rows gathered in expert order", tokens=X,
                    index=token.to(torch.int32))


def moe_dispatch_fp8(seed: int = 0, device="cpu", **kw) -> Workload:
    """The MoE workload run as quantize-then-dispatch: the step quantizes the
    T tokens once and gathers codes and scales into expert order (the same
    data as moe_grouped)."""
    w = moe_grouped(seed, device, **kw)
    w.name = w.name.replace("MoE grouped", "MoE FP8 dispatch")
    w.note = "tokens quantized once, FP8 rows gathered in expert order"
    return w


def large_m(seed: int = 0, device="cpu", M: int = 32768) -> Workload:
    """A [M, 7168] ~ N(0,1) with the outlier channels; B [18432, 7168] ~ N(0, 0.01^2)."""
    return Workload(f"large-M {M}x18432x7168",
                    activations_with_outliers(M, HIDDEN, seed * 1000 + 1, device),
                    {"B": normal_bf16((18432, HIDDEN), 0.01, seed * 1000 + 2, device)})


def dense_backward(seed: int = 0, device="cpu", T: int = 8192) -> Workload:
    """The backward pass of the dense 7168-square layer y = x W^T: layer input
    X [T, 7168] ~ N(0,1) with the outlier channels (as dense_square's A),
    output gradient dY [T, 7168] ~ N(0,1), W [7168, 7168] ~ N(0, 0.01^2)."""
    X = activations_with_outliers(T, HIDDEN, seed * 1000 + 1, device)
    W = normal_bf16((HIDDEN, HIDDEN), 0.01, seed * 1000 + 2, device)
    dY = normal_bf16((T, HIDDEN), 1.0, seed * 1000 + 3, device)
    return Workload(f"dense backward {T}x7168x7168 (dX and dW)", dY, {"W": W},
                    note="A holds dY; X is the layer input", X=X)


def dense_square_ue8m0(seed: int = 0, device="cpu", M: int = 8192) -> Workload:
    """dense_square's tensors, quantized with power-of-two (UE8M0) scales and
    multiplied by the hardware-scaled GEMM."""
    w = dense_square(seed, device, M)
    w.name = f"dense {M}x7168x7168, UE8M0 scales"
    w.scales = "ue8m0"
    return w


def dense_backward_ue8m0(seed: int = 0, device="cpu", T: int = 8192) -> Workload:
    """dense_backward's tensors with power-of-two (UE8M0) scales throughout."""
    w = dense_backward(seed, device, T)
    w.name = f"dense backward {T}x7168x7168 (dX and dW), UE8M0 scales"
    w.scales = "ue8m0"
    return w


WORKLOADS = {1: tiny, 2: mla_down, 3: dense_square, 4: moe_grouped, 5: large_m, 6: mla_down_fused,
           7: moe_dispatch_fp8, 8: dense_backward, 9: dense_square_ue8m0, 10: dense_backward_ue8m0}
