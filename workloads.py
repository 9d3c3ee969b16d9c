"""Seeded synthetic inputs for MXFP4 block quantization.

This module only draws and shapes input tensors; it holds none of the
method's arithmetic (no scale, rounding or layout logic).  Both the GPU
library's tests/benchmark and the CPU oracle's tests take their inputs from
here.  It sits outside the library package and imports only torch, so a
process that draws inputs for the oracle alone maps no part of the CUDA
library.  Every generator is deterministic for a given seed and device; values
are drawn as float32 with ``torch.Generator`` and rounded to BF16 by torch's
round-to-nearest-even cast.

The shapes mirror the workloads the method serves (MoE activations and
expert weights of the models named on the pages: Kimi-K2 style 384 experts
with top-8 routing and hidden size 7168; Qwen3-30B-A3B style 128 experts with
hidden 2048 and expert width 768).  No dataset or trained weight is used.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    """N(0, std^2) values rounded to BF16."""
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def small_matrix(seed: int = 0, M: int = 128, K: int = 256, device="cpu") -> torch.Tensor:
    """One BF16 matrix of N(0,1) values (default 128 x 256: 8 scale columns,
    2 k-tiles)."""
    return normal_bf16((M, K), seed, device=device)


def dense_activation(seed: int = 1, M: int = 4096, K: int = 7168, device="cpu") -> torch.Tensor:
    """Dense activation: N(0,1) * row_scale with row_scale = 2^U(-8, 8) per
    row (log-uniform in [2^-8, 2^8])."""
    g = _gen(seed, device)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    e = torch.rand((M, 1), generator=g, device=device, dtype=torch.float32) * 16.0 - 8.0
    return (x * torch.exp2(e)).to(torch.bfloat16)


@dataclass
class GroupedInput:
    x: torch.Tensor          # BF16 [tokens * top_k, K], rows sorted by expert
    offsets: torch.Tensor    # int32 [E + 1], segment e = rows [o[e], o[e+1])
    token_of_row: torch.Tensor  # int64 [tokens * top_k], source token of each row (CPU)
    num_experts: int
    x_tokens: torch.Tensor   # BF16 [tokens, K], the token rows before dispatch
    row_index: torch.Tensor  # int32 [tokens * top_k] on `device`: token of each row
    dest_rows: torch.Tensor  # int32 [tokens, top_k] on `device`: row of route j of token t


def moe_grouped(seed: int = 2, tokens: int = 16384, top_k: int = 8, num_experts: int = 384,
                K: int = 7168, device="cpu") -> GroupedInput:
    """MoE expert-sorted activations: every token is routed to ``top_k``
    distinct experts drawn uniformly (the first ``top_k`` of a random
    ordering); its N(0,1) hidden row is duplicated once per route; rows are
    stable-sorted by expert (then token); int32 offsets delimit the experts'
    segments.  ``row_index`` (row -> token) and ``dest_rows`` (token, route ->
    row) are the two directions of the same dispatch permutation."""
    g_route = _gen(seed, "cpu")
    keys = torch.rand((tokens, num_experts), generator=g_route)
    experts = torch.topk(keys, top_k, dim=1).indices.reshape(-1)          # [T*k]
    token_ids = torch.arange(tokens).repeat_interleave(top_k)             # [T*k]
    order = torch.sort(experts, stable=True).indices
    token_of_row = token_ids[order]
    counts = torch.bincount(experts, minlength=num_experts)
    offsets = torch.zeros(num_experts + 1, dtype=torch.int64)
    offsets[1:] = torch.cumsum(counts, 0)
    x_tok = normal_bf16((tokens, K), seed + 1000, device=device)
    row_index = token_of_row.to(torch.int32).to(device)
    dest = torch.empty(tokens * top_k, dtype=torch.int64)
    dest[order] = torch.arange(tokens * top_k)
    dest_rows = dest.view(tokens, top_k).to(torch.int32).to(device)
    x = x_tok.index_select(0, token_of_row.to(device))
    return GroupedInput(x=x, offsets=offsets.to(torch.int32).to(device),
                        token_of_row=token_of_row, num_experts=num_experts, x_tokens=x_tok,
                        row_index=row_index, dest_rows=dest_rows)


@dataclass
class ExpertWeights:
    w13: torch.Tensor       # BF16 [E, 2N, H]  ([w1; w3] along dim 1)
    w2: torch.Tensor        # BF16 [E, H, N]
    w13_bias: torch.Tensor  # FP32 [E, 2N]
    w2_bias: torch.Tensor   # FP32 [E, H]


def expert_weights(seed: int = 3, E: int = 128, N: int = 768, H: int = 2048,
                   device="cpu") -> ExpertWeights:
    """MoE expert weights: w13 [E, 2N, H] and w2 [E, H, N] with N(0, 0.02^2)
    values, FP32 biases with N(0, 0.01^2)."""
    w13 = normal_bf16((E, 2 * N, H), seed, std=0.02, device=device)
    w2 = normal_bf16((E, H, N), seed + 1, std=0.02, device=device)
    g = _gen(seed + 2, device)
    b13 = torch.randn((E, 2 * N), generator=g, device=device) * 0.01
    b2 = torch.randn((E, H), generator=g, device=device) * 0.01
    return ExpertWeights(w13=w13, w2=w2, w13_bias=b13, w2_bias=b2)


def edge_cases(seed: int = 4, M: int = 1000, K: int = 2880, frac: float = 0.01) -> torch.Tensor:
    """Edge-case stress matrix (always drawn on the CPU): Student-t (nu = 2)
    values, plus three disjoint sets of ``frac`` of the 32-element blocks:
    (i) all zero; (ii) N(0,1) * 2^-130 (BF16 subnormals); (iii) blocks whose
    largest magnitude is set to exactly 1.5 * 2^e or 1.75 * 2^e (alternating;
    e = floor(log2) of the block's original largest magnitude, random sign)
    with every other element clamped to at most that magnitude.  No +-Inf."""
    g = _gen(seed, "cpu")
    z = torch.randn((3, M, K), generator=g, dtype=torch.float32)
    t = z[0] / torch.sqrt((z[1] * z[1] + z[2] * z[2]) / 2.0)      # Student-t, nu = 2
    x = t.to(torch.bfloat16).to(torch.float32)                      # BF16-exact values
    nb = K // 32
    blocks = x.view(M, nb, 32)
    n_special = int(round(frac * M * nb))
    perm = torch.randperm(M * nb, generator=g)
    zero_ids = perm[:n_special]
    sub_ids = perm[n_special:2 * n_special]
    mant_ids = perm[2 * n_special:3 * n_special]
    flat = blocks.reshape(M * nb, 32)
    flat[zero_ids] = 0.0
    sub = torch.randn((n_special, 32), generator=g, dtype=torch.float32) * (2.0 ** -130)
    flat[sub_ids] = sub.to(torch.bfloat16).to(torch.float32)
    signs = torch.where(torch.rand(n_special, generator=g) < 0.5, -1.0, 1.0)
    for i, b in enumerate(mant_ids.tolist()):
        row = flat[b]
        j = int(torch.argmax(row.abs()))
        amax = float(row[j].abs())
        if amax == 0.0 or not math.isfinite(amax):
            continue
        e = math.floor(math.log2(amax))
        m = 1.5 if i % 2 == 0 else 1.75
        target = m * 2.0 ** e
        row.clamp_(-target, target)
        row[j] = float(signs[i]) * target
    return flat.reshape(M, K).to(torch.bfloat16)


def bf16_bits(x: torch.Tensor):
    """BF16 tensor -> numpy uint16 bit patterns (host copy)."""
    return x.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def from_bits(bits, device="cpu") -> torch.Tensor:
    """numpy uint16 BF16 bit patterns -> BF16 tensor."""
    import numpy as np
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
