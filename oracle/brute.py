"""Pure-Python brute force of the triangle-attention forward, for tiny shapes.

TEST INFRASTRUCTURE ONLY.  Written independently of ``triattn_oracle.c``
(nested lists, ``math.fsum`` / ``math.exp``) so the two can be checked
against each other.  Follows the cuEquivariance ``triangle_attention`` API
page, formula: the logit of a masked key is replaced by -1e9.
"""
from __future__ import annotations

import math
import struct


def attention_rows(qs, ks, vs, bias_rows, valid, scale):
    """qs: list of query vectors; ks, vs: key / value vectors; bias_rows[i][j];
    valid[j] (or valid[i][j] when nested) -> list of (out vector, lse, max)."""
    res = []
    for i, qv in enumerate(qs):
        logits = []
        for j, kv in enumerate(ks):
            ok = valid[i][j] if isinstance(valid[0], (list, tuple)) else valid[j]
            if ok:
                dot = math.fsum(a * b for a, b in zip(qv, kv))
                logits.append(scale * dot + (bias_rows[i][j] if bias_rows is not None else 0.0))
            else:
                logits.append(-1e9)
        mx = max(logits)
        ws = [math.exp(x - mx) for x in logits]
        tot = math.fsum(ws)
        out = [math.fsum(w * vv[d] for w, vv in zip(ws, vs)) / tot for d in range(len(vs[0]))]
        res.append((out, mx + math.log(tot), mx))
    return res


def tri_fwd(q, k, v, bias, mask=None, kv_lengths=None, scale=None):
    """Nested-list inputs shaped like the page's (B,N,H,Q,D) etc.; returns nested O, lse, max."""
    B, N, H, Q, D = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0]), len(q[0][0][0][0])
    K = len(k[0][0][0])
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    # the scale reaches the kernel as a binary32 value
    scale = struct.unpack("f", struct.pack("f", scale))[0]
    O = [[[[None] * Q for _ in range(H)] for _ in range(N)] for _ in range(B)]
    L = [[[[None] * Q for _ in range(H)] for _ in range(N)] for _ in range(B)]
    M = [[[[None] * Q for _ in range(H)] for _ in range(N)] for _ in range(B)]
    for b in range(B):
        for n in range(N):
            if mask is not None:
                valid = [bool(mask[b][n][0][0][j]) for j in range(K)]
            elif kv_lengths is not None:
                ln = max(0, min(K, int(kv_lengths[b][n])))
                valid = [j < ln for j in range(K)]
            else:
                valid = [True] * K
            for h in range(H):
                rows = attention_rows(q[b][n][h], k[b][n][h], v[b][n][h], bias[b][0][h], valid, scale)
                for i, (o, lse, mx) in enumerate(rows):
                    O[b][n][h][i], L[b][n][h][i], M[b][n][h][i] = o, lse, mx
    return O, L, M
