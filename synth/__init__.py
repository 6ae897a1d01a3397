"""Seeded synthetic inputs for the triangle-attention forward and its varlen form.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so the oracle and the CUDA path can both be fed from it
without sharing any of the method's computation.

Recipe (the same for every workload):
  * one ``torch.Generator('cpu')`` seeded with the workload's seed;
  * draws in a fixed order: q, k, v, bias, then the mask / lengths
    (varlen: lengths first, because they fix the packed shapes);
  * ``randn`` in fp32, scaled by the stated standard deviation, then cast to
    the storage dtype with round-to-nearest-even (``Tensor.to``).  The same
    bytes go to the GPU and, widened exactly to fp64, to the oracle.

Workload shapes follow the cuEquivariance ``triangle_attention`` API page
(Parameters: q, k, v, bias, mask, kv_lengths; Example) and, for the packed
form, the Transformer Engine ``fused_attn.h`` page (NVTE_NOT_INTERLEAVED
layout, ``cu_seqlens``) with the tensorplay ``BlockMask`` format.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class TriangleCase:
    """One triangle-attention problem, all tensors on the CPU."""

    name: str
    B: int
    N: int
    H: int
    Q: int
    K: int
    D: int
    dtype: str
    bias_dtype: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    bias: torch.Tensor
    mask: Optional[torch.Tensor]  # (B,N,1,1,K) uint8, nonzero = valid
    kv_lengths: Optional[torch.Tensor]  # (B,N) int32
    scale: float
    meta: dict = field(default_factory=dict)


@dataclass
class VarlenCase:
    """Packed sequences with a 128x128 block-sparse mask, all on the CPU."""

    name: str
    H: int
    D: int
    dtype: str
    lengths: torch.Tensor  # (S,) int32
    cu_seqlens: torch.Tensor  # (S+1,) int32
    q: torch.Tensor  # (total, H, D)
    k: torch.Tensor
    v: torch.Tensor
    kv_num_blocks: Optional[torch.Tensor]  # (S, mask_heads, max_q_blocks) int32
    kv_indices: Optional[torch.Tensor]  # (S, mask_heads, max_q_blocks, max_kv_blocks)
    full_kv_num_blocks: Optional[torch.Tensor]
    full_kv_indices: Optional[torch.Tensor]
    mask_mod: str  # "none" | "causal"
    block: int
    scale: float
    max_seqlen: int
    # key side; the same as the query side unless drawn with lengths_k
    lengths_k: Optional[torch.Tensor] = None
    cu_seqlens_k: Optional[torch.Tensor] = None
    max_seqlen_k: int = 0

    def __post_init__(self):
        if self.lengths_k is None:
            self.lengths_k = self.lengths
            self.cu_seqlens_k = self.cu_seqlens
            self.max_seqlen_k = self.max_seqlen


def _randn(gen, shape, std, dtype):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(TORCH_DTYPES[dtype]).contiguous()


def make_triangle(
    name: str,
    B: int,
    N: int,
    H: int,
    Q: int,
    K: int,
    D: int,
    dtype: str,
    bias_dtype: str,
    seed: int,
    bias_std: float = 1.0,
    mask: str = "none",
    kv_range: tuple[int, int] | None = None,
    kv_const: int | None = None,
    forced_kv: dict[int, int] | None = None,
    mask_p: float = 0.5,
    scale: float | None = None,
    qkv_std: float = 1.0,
) -> TriangleCase:
    """Draw a triangle-attention case.

    mask: "none" | "kvlen" (int32 lengths) | "dense" (Bernoulli key mask).
    kv_range (lo, hi) draws lengths uniformly in [lo, hi]; kv_const sets every
    row to one length; forced_kv pins a few flat (b*N+n) rows afterwards.
    """
    g = torch.Generator("cpu").manual_seed(seed)
    q = _randn(g, (B, N, H, Q, D), qkv_std, dtype)
    k = _randn(g, (B, N, H, K, D), qkv_std, dtype)
    v = _randn(g, (B, N, H, K, D), qkv_std, dtype)
    bias = _randn(g, (B, 1, H, Q, K), bias_std, bias_dtype)
    m = None
    kvl = None
    if mask == "kvlen":
        if kv_const is not None:
            kvl = torch.full((B, N), kv_const, dtype=torch.int32)
        else:
            lo, hi = kv_range
            kvl = torch.randint(lo, hi + 1, (B, N), generator=g, dtype=torch.int64).to(torch.int32)
        if forced_kv:
            flat = kvl.view(-1)
            for idx, val in forced_kv.items():
                flat[idx] = val
    elif mask == "dense":
        m = (torch.rand(B, N, 1, 1, K, generator=g) < mask_p).to(torch.uint8)
    elif mask != "none":
        raise ValueError(mask)
    s = 1.0 / math.sqrt(D) if scale is None else scale
    return TriangleCase(name, B, N, H, Q, K, D, dtype, bias_dtype, q, k, v, bias, m, kvl, s)


def grad_out(case: TriangleCase, seed: int, std: float = 1.0) -> torch.Tensor:
    """A seeded dL/dO for a triangle case: standard normal (times std) in the case's dtype, q's shape."""
    g = torch.Generator("cpu").manual_seed(seed)
    return _randn(g, tuple(case.q.shape), std, case.dtype)


def page_example_kv_lengths(seq_len: int = 128, valid: int = 96) -> torch.Tensor:
    """The key mask of the triangle_attention API page's example (row_valid & col_valid).

    Returned as the (1, seq_len, 1, 1, seq_len) bool mask the example builds:
    rows n < valid keep keys j < valid, rows n >= valid keep none.
    """
    pos = torch.arange(seq_len)
    row_valid = pos.view(1, seq_len) < valid
    col_valid = pos.view(1, seq_len) < valid
    return row_valid.view(1, seq_len, 1, 1, 1) & col_valid.view(1, 1, 1, 1, seq_len)


# ---------------------------------------------------------------------------
# The five workloads (sizes and distributions as stated for each)
# ---------------------------------------------------------------------------

def tiny_fp32() -> TriangleCase:
    """B=1,N=32,H=2,Q=K=32,D=32 fp32, bias fp32, scale 1/sqrt(32), no mask."""
    return make_triangle("tiny_fp32", 1, 32, 2, 32, 32, 32, "f32", "f32", seed=1001)


def fp16_kvlen() -> TriangleCase:
    """B=1,N=128,H=2,Q=K=128,D=32 fp16, bias fp32, kv_lengths=96 on every row."""
    return make_triangle("fp16_kvlen", 1, 128, 2, 128, 128, 32, "f16", "f32", seed=1002,
                         mask="kvlen", kv_const=96)


def fp16_dense() -> TriangleCase:
    """Same q/k/v/bias as fp16_kvlen, with a dense Bernoulli(0.5) key mask."""
    return make_triangle("fp16_dense", 1, 128, 2, 128, 128, 32, "f16", "f32", seed=1002,
                         mask="dense", mask_p=0.5)


def fp16_page_example() -> TriangleCase:
    """Same q/k/v/bias as fp16_kvlen with the page example's lengths (96 for n<96, else 0)."""
    c = make_triangle("fp16_page_example", 1, 128, 2, 128, 128, 32, "f16", "f32", seed=1002,
                      mask="kvlen", kv_const=96)
    c.kv_lengths[:, 96:] = 0
    return c


def bf16_pairstack() -> TriangleCase:
    """B=1,N=384,H=4,Q=K=384,D=32 bf16, bias ~N(0,2^2) bf16, kv_lengths uniform in [192,384]."""
    return make_triangle("bf16_pairstack", 1, 384, 4, 384, 384, 32, "bf16", "bf16", seed=1003,
                         bias_std=2.0, mask="kvlen", kv_range=(192, 384))


def bf16_long() -> TriangleCase:
    """B=1,N=768,H=4,Q=K=768,D=64 bf16, bias bf16, kv_lengths uniform in [0,768].

    Rows 0 and 1 are pinned to 0 (all keys masked) and 768 (all keys valid) so
    both extremes are always present.
    """
    return make_triangle("bf16_long", 1, 768, 4, 768, 768, 64, "bf16", "bf16", seed=1004,
                         mask="kvlen", kv_range=(0, 768), forced_kv={0: 0, 1: 768})


def bf16_long_d128() -> TriangleCase:
    """bf16_long with a head dimension of 128: B=1,N=768,H=4,Q=K=768,D=128 bf16, bias bf16,
    kv_lengths uniform in [0,768] (rows 0 and 1 pinned to 0 and 768)."""
    return make_triangle("bf16_long_d128", 1, 768, 4, 768, 768, 128, "bf16", "bf16", seed=1005,
                         mask="kvlen", kv_range=(0, 768), forced_kv={0: 0, 1: 768})


def bf16_d256() -> TriangleCase:
    """The widest head dimension the forward takes: B=1,N=64,H=4,Q=K=384,D=256 bf16, bias bf16,
    kv_lengths uniform in [0,384]."""
    return make_triangle("bf16_d256", 1, 64, 4, 384, 384, 256, "bf16", "bf16", seed=1006,
                         mask="kvlen", kv_range=(0, 384))


TRIANGLE_WORKLOADS = {
    "tiny_fp32": tiny_fp32,
    "fp16_kvlen": fp16_kvlen,
    "fp16_dense": fp16_dense,
    "fp16_page_example": fp16_page_example,
    "bf16_pairstack": bf16_pairstack,
    "bf16_long": bf16_long,
    "bf16_d256": bf16_d256,
}


# ---------------------------------------------------------------------------
# Packed (varlen) sequences and block-sparse masks
# ---------------------------------------------------------------------------

def causal_block_lists(lengths: list[int], block: int = 128, mask_heads: int = 1):
    """Block lists of a causal mask over equal-length q/k sequences.

    q-block i lists kv-block i as partial (the diagonal, where the causal
    predicate must be applied) and kv-blocks 0..i-1 as full.  Indices are
    sequence-local.  Returns int32 tensors
    (kv_num_blocks, kv_indices, full_kv_num_blocks, full_kv_indices)
    shaped (S, mask_heads, MQ) and (S, mask_heads, MQ, MK).
    """
    S = len(lengths)
    nbs = [(L + block - 1) // block for L in lengths]
    MQ = max(1, max(nbs))
    MK = MQ
    kv_num = torch.zeros(S, mask_heads, MQ, dtype=torch.int32)
    kv_idx = torch.zeros(S, mask_heads, MQ, MK, dtype=torch.int32)
    full_num = torch.zeros(S, mask_heads, MQ, dtype=torch.int32)
    full_idx = torch.zeros(S, mask_heads, MQ, MK, dtype=torch.int32)
    for s, nb in enumerate(nbs):
        for i in range(nb):
            kv_num[s, :, i] = 1
            kv_idx[s, :, i, 0] = i
            full_num[s, :, i] = i
            if i:
                full_idx[s, :, i, :i] = torch.arange(i, dtype=torch.int32)
    return kv_num, kv_idx, full_num, full_idx


def make_varlen(
    name: str,
    num_seqs: int,
    lmin: int,
    lmax: int,
    H: int,
    D: int,
    dtype: str,
    seed: int,
    mask_mod: str = "causal",
    lengths: list[int] | None = None,
    block_lists: str = "causal",
    scale: float | None = None,
    lengths_k: list[int] | None = None,
) -> VarlenCase:
    """Draw packed sequences and their block mask.

    q and k share lengths unless lengths_k gives the key lengths (then
    block_lists must be "none": the causal lists assume equal lengths).
    block_lists: "causal" (full + partial lists of a causal mask), "window<W>" (the
    lists of a sliding window of W keys, `window_block_lists`), "none" (no lists:
    every block visited, mask_mod applied everywhere).
    """
    g = torch.Generator("cpu").manual_seed(seed)
    if lengths is None:
        lengths = torch.randint(lmin, lmax + 1, (num_seqs,), generator=g, dtype=torch.int64).tolist()

    def offsets(ls):
        t = torch.tensor(ls, dtype=torch.int32)
        cu = torch.zeros(len(ls) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(t, 0).to(torch.int32)
        return t, cu

    lens, cu = offsets(lengths)
    lens_k, cu_k = offsets(lengths_k) if lengths_k is not None else (lens, cu)
    if lengths_k is not None and (len(lengths_k) != len(lengths) or block_lists != "none"):
        raise ValueError("lengths_k needs one key length per sequence and block_lists='none'")
    total, total_k = int(cu[-1]), int(cu_k[-1])
    q = _randn(g, (total, H, D), 1.0, dtype)
    k = _randn(g, (total_k, H, D), 1.0, dtype)
    v = _randn(g, (total_k, H, D), 1.0, dtype)
    kv_num = kv_idx = full_num = full_idx = None
    if block_lists == "causal":
        kv_num, kv_idx, full_num, full_idx = causal_block_lists(lengths)
    elif block_lists.startswith("window"):  # "window<W>": the lists of a sliding window of W keys
        kv_num, kv_idx, full_num, full_idx = window_block_lists(lengths, int(block_lists[6:]))
    elif block_lists != "none":
        raise ValueError(block_lists)
    s = 1.0 / math.sqrt(D) if scale is None else scale
    if lengths_k is None:
        return VarlenCase(name, H, D, dtype, lens, cu, q, k, v, kv_num, kv_idx, full_num, full_idx,
                          mask_mod, 128, s, max(lengths))
    return VarlenCase(name, H, D, dtype, lens, cu, q, k, v, kv_num, kv_idx, full_num, full_idx,
                      mask_mod, 128, s, max(lengths), lens_k, cu_k, max(lengths_k))


def window_block_lists(lengths: list[int], window: int, block: int = 128, mask_heads: int = 1):
    """Block lists of a causal sliding-window mask (keys q - window < k <= q) over equal-length
    q/k sequences, in the layout of `causal_block_lists`: kv-block j of q-block i is full when
    every (q, k) pair of the two blocks' extents is kept, partial when some pair is, unlisted
    otherwise."""
    if window < 1:
        raise ValueError("window must be >= 1")
    S = len(lengths)
    nbs = [(L + block - 1) // block for L in lengths]
    MQ = max(1, max(nbs))
    MK = MQ
    kv_num = torch.zeros(S, mask_heads, MQ, dtype=torch.int32)
    kv_idx = torch.zeros(S, mask_heads, MQ, MK, dtype=torch.int32)
    full_num = torch.zeros(S, mask_heads, MQ, dtype=torch.int32)
    full_idx = torch.zeros(S, mask_heads, MQ, MK, dtype=torch.int32)
    for s, nb in enumerate(nbs):
        for i in range(nb):
            a0, a1 = i * block, i * block + block - 1  # query rows of block i
            part, full = [], []
            for j in range(i + 1):
                b0, b1 = j * block, j * block + block - 1  # keys of block j
                if not (b0 <= a1 and b1 > a0 - window):
                    continue
                (full if (b1 <= a0 and b0 > a1 - window) else part).append(j)
            kv_num[s, :, i] = len(part)
            full_num[s, :, i] = len(full)
            if part:
                kv_idx[s, :, i, :len(part)] = torch.tensor(part, dtype=torch.int32)
            if full:
                full_idx[s, :, i, :len(full)] = torch.tensor(full, dtype=torch.int32)
    return kv_num, kv_idx, full_num, full_idx


def bf16_varlen() -> VarlenCase:
    """8 sequences, lengths uniform in [256,2048], H=8, D=128 bf16, no bias, causal BlockMask."""
    return make_varlen("bf16_varlen", 8, 256, 2048, 8, 128, "bf16", seed=1005)


def bf16_varlen_window512() -> VarlenCase:
    """The bf16_varlen sequences under a sliding window of 512 keys (mask_mod sliding_window,
    the window's block lists)."""
    return make_varlen("bf16_varlen_window512", 8, 256, 2048, 8, 128, "bf16", seed=1005,
                       mask_mod="sliding_window", block_lists="window512")


WORKLOADS = dict(TRIANGLE_WORKLOADS)
WORKLOADS["bf16_varlen"] = bf16_varlen
WORKLOADS["bf16_varlen_window512"] = bf16_varlen_window512
