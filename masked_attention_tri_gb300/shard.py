"""Split of the triangle-attention forward across ranks, one GPU per rank.

Every (b, n) slab of the triangle form is independent (the formula of the
cuEquivariance triangle_attention page has no term that couples two n), and
the bias (B, 1, H, Q, K) is shared over N.  So each rank takes a contiguous
range of the flattened (b, n) slabs, holds its slabs of q / k / v / mask /
kv_lengths and a replica of the bias, and runs the same kernels on them.
There is no exchange on the data path: a rank's outputs are exactly the rows
of the whole problem's outputs that belong to its slabs.
"""
from __future__ import annotations

from typing import Iterator


def slab_range(units: int, world: int, rank: int) -> tuple[int, int]:
    """[u0, u1) of `units` slabs for `rank` of `world`: contiguous, sizes differing by at most one,
    every slab in exactly one range."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    base, extra = divmod(units, world)
    u0 = rank * base + min(rank, extra)
    return u0, u0 + base + (1 if rank < extra else 0)


def per_batch_pieces(u0: int, u1: int, N: int) -> Iterator[tuple[int, int, int]]:
    """Split the flattened slab range [u0, u1) into (b, n0, n1) pieces that stay inside one b,
    so each piece is a contiguous (1, n1 - n0, ...) view with its own bias[b]."""
    u = u0
    while u < u1:
        b, n0 = divmod(u, N)
        n1 = min(N, n0 + (u1 - u))
        yield b, n0, n1
        u += n1 - n0


def triangle_attention_shard(q, k, v, bias, world: int, rank: int, mask=None, kv_lengths=None, scale=None,
                             return_aux=False):
    """This rank's share of ``triangle_attention`` on full-size (B, N, ...) inputs.

    Returns a list of ``(b, n0, n1, result)`` with ``result`` as returned by
    ``triangle_attention`` for slabs b, n0..n1-1 (O, or (O, lse, max)).
    Views of the inputs are passed in place; nothing is copied.
    """
    from .api import triangle_attention
    B, N = q.shape[0], q.shape[1]
    u0, u1 = slab_range(B * N, world, rank)
    out = []
    for b, n0, n1 in per_batch_pieces(u0, u1, N):
        kl = None if kv_lengths is None else kv_lengths.reshape(B, N)[b:b + 1, n0:n1]
        m = None if mask is None else mask[b:b + 1, n0:n1]
        res = triangle_attention(q[b:b + 1, n0:n1], k[b:b + 1, n0:n1], v[b:b + 1, n0:n1], bias[b:b + 1],
                                 mask=m, scale=scale, return_aux=return_aux, kv_lengths=kl)
        out.append((b, n0, n1, res))
    return out
