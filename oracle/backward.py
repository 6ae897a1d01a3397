"""CPU oracle for the triangle-attention backward (fp64, plain definition).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: the product path never
imports it and it shares no code with the CUDA library.

The forward is the cuEquivariance ``triangle_attention`` API page's formula
(x = s Q.K + bias at valid keys, the constant -1e9 at masked keys; O = softmax(x) V;
the bias (B,1,H,Q,K) is shared over N).  The page notes that the function saves
its context for backward; the gradients are the chain rule through that
formula, for a loss L whose gradient with respect to O is ``d_out``:

    P      = softmax_k(x)                        (per query row)
    dV[k]  = sum_q P[q,k] dO[q]
    dP[q,k]= dO[q] . V[k]
    dx[q,k]= P[q,k] (dP[q,k] - sum_k' P[q,k'] dP[q,k'])   at valid keys,
             0 at masked keys (their logit is a constant)
    dQ[q]  = s sum_k dx[q,k] K[k]
    dK[k]  = s sum_q dx[q,k] Q[q]
    dBias[b,0,h,q,k] = sum_n dx[b,n,h,q,k]

(sum_k' P dP equals dO[q] . O[q].)  Written per (b, n, h) slab with numpy
matrix products, no blocking or reordering beyond the definition.
"""
from __future__ import annotations

import numpy as np

from . import widen

MASKED = -1.0e9


def _valid_keys(B, N, K, mask, kv_lengths):
    """(B, N, K) bool: key k of row (b, n) takes part (mask nonzero / k < clamped kv_lengths)."""
    if mask is not None:
        m = np.asarray(mask.detach().cpu().numpy() if hasattr(mask, "detach") else mask).reshape(B, N, K)
        return m != 0
    if kv_lengths is not None:
        kl = np.asarray(kv_lengths.detach().cpu().numpy() if hasattr(kv_lengths, "detach") else kv_lengths)
        kl = np.clip(kl.reshape(B, N).astype(np.int64), 0, K)
        return np.arange(K)[None, None, :] < kl[:, :, None]
    return np.ones((B, N, K), dtype=bool)


def tri_bwd(q, k, v, bias, d_out, mask=None, kv_lengths=None, scale=None):
    """Gradients (dQ, dK, dV, dBias) in fp64 numpy of L with dL/dO = d_out.

    q (B,N,H,Q,D), k/v (B,N,H,K,D), bias (B,1,H,Q,K) as stored tensors (widened
    exactly); d_out (B,N,H,Q,D) any float tensor or array (used in fp64).
    dBias has the bias's shape (B,1,H,Q,K): the sum over n of each slab's dx.
    """
    Qa, Ka, Va, Ba = widen(q), widen(k), widen(v), widen(bias)
    dO = np.asarray(d_out.detach().cpu().double().numpy() if hasattr(d_out, "detach") else d_out, dtype=np.float64)
    B, N, H, Qn, D = Qa.shape
    K = Ka.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    s = float(np.float32(scale))  # the forward receives the scale as a float
    valid = _valid_keys(B, N, K, mask, kv_lengths)
    dQ = np.zeros_like(Qa)
    dK = np.zeros_like(Ka)
    dV = np.zeros_like(Va)
    dBias = np.zeros_like(Ba)
    for b in range(B):
        for n in range(N):
            vk = valid[b, n]
            for h in range(H):
                qm, km, vm, do = Qa[b, n, h], Ka[b, n, h], Va[b, n, h], dO[b, n, h]
                x = s * (qm @ km.T) + Ba[b, 0, h]
                x[:, ~vk] = MASKED
                e = np.exp(x - x.max(axis=1, keepdims=True))
                P = e / e.sum(axis=1, keepdims=True)
                dV[b, n, h] = P.T @ do
                dP = do @ vm.T
                dx = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                dx[:, ~vk] = 0.0
                dQ[b, n, h] = s * (dx @ km)
                dK[b, n, h] = s * (dx.T @ qm)
                dBias[b, 0, h] += dx
    return dQ, dK, dV, dBias


def _np(t, dtype=np.int64):
    return None if t is None else np.asarray(t.detach().cpu().numpy() if hasattr(t, "detach") else t, dtype=dtype)


def varlen_bwd(q, k, v, cu_seqlens_q, cu_seqlens_k, d_out, scale=None, kv_num_blocks=None, kv_indices=None,
               full_kv_num_blocks=None, full_kv_indices=None, block=128, mask_mod="none", window=0,
               prefix_lengths=None, bias=None):
    """Gradients (dQ, dK, dV, dBias or None) of the packed-sequence forward, fp64 numpy.

    Inputs as for ``oracle.varlen_fwd``; d_out (total_q, H, D).  Per sequence and
    head the element mask follows the BlockMask page: the block lists rebuilt by
    the page's reconstruction loop (full blocks win over partial ones, mask_mod
    applies to partial blocks; without lists every block is partial), mask_mod
    on local indices (causal k <= q; sliding window q - window < k <= q; prefix
    LM k <= q or k < the prefix).  Masked keys have the constant logit -1e9, so
    their dx is 0; keys past a sequence's end take no part.  dBias (H,
    max_seqlen_q, max_seqlen_k) sums each sequence's dx at local positions.
    """
    from . import to_dense
    Qa, Ka, Va = widen(q), widen(k), widen(v)
    dO = np.asarray(d_out.detach().cpu().double().numpy() if hasattr(d_out, "detach") else d_out, dtype=np.float64)
    total_q, H, D = Qa.shape
    cq, ck = _np(cu_seqlens_q), _np(cu_seqlens_k)
    S = len(cq) - 1
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    s = float(np.float32(scale))
    Ba = widen(bias) if bias is not None else None
    kn, ki, fn, fi = _np(kv_num_blocks), _np(kv_indices), _np(full_kv_num_blocks), _np(full_kv_indices)
    dQ, dK, dV = np.zeros_like(Qa), np.zeros_like(Ka), np.zeros_like(Va)
    dBias = np.zeros_like(Ba) if Ba is not None else None
    for si in range(S):
        q0, q1, k0, k1 = int(cq[si]), int(cq[si + 1]), int(ck[si]), int(ck[si + 1])
        Lq, Lk = q1 - q0, k1 - k0
        if Lq <= 0 or Lk <= 0:
            continue
        if prefix_lengths is None:
            pre = 0
        elif isinstance(prefix_lengths, int):
            pre = prefix_lengths
        else:
            pre = int(_np(prefix_lengths)[si])
        qi, kj = np.arange(Lq)[:, None], np.arange(Lk)[None, :]
        if mask_mod == "causal":
            mod = kj <= qi
        elif mask_mod == "sliding_window":
            mod = (kj <= qi) & (kj > qi - window)
        elif mask_mod == "prefix_lm":
            mod = (kj <= qi) | (kj < pre)
        else:
            mod = np.ones((Lq, Lk), dtype=bool)
        nqb, nkb = (Lq + block - 1) // block, (Lk + block - 1) // block
        for h in range(H):
            if kn is None:
                part = np.ones((nqb, nkb), dtype=bool)
                full = np.zeros((nqb, nkb), dtype=bool)
            else:
                hm = 0 if kn.shape[1] == 1 else h
                MQ = kn.shape[2]
                part = np.zeros((nqb, nkb), dtype=bool)
                full = np.zeros((nqb, nkb), dtype=bool)
                rows = min(nqb, MQ)
                part[:rows] = to_dense(kn[si, hm, :rows], ki[si, hm, :rows], nkb).astype(bool)
                if fn is not None:
                    full[:rows] = to_dense(fn[si, hm, :rows], fi[si, hm, :rows], nkb).astype(bool)
                part &= ~full
            bf = np.repeat(np.repeat(full, block, 0), block, 1)[:Lq, :Lk]
            bp = np.repeat(np.repeat(part, block, 0), block, 1)[:Lq, :Lk]
            valid = bf | (bp & mod)
            qm, km, vm, do = Qa[q0:q1, h], Ka[k0:k1, h], Va[k0:k1, h], dO[q0:q1, h]
            x = s * (qm @ km.T)
            if Ba is not None:
                x = x + Ba[h, :Lq, :Lk]
            x[~valid] = MASKED
            e = np.exp(x - x.max(axis=1, keepdims=True))
            P = e / e.sum(axis=1, keepdims=True)
            dV[k0:k1, h] += P.T @ do
            dP = do @ vm.T
            dx = P * (dP - (P * dP).sum(axis=1, keepdims=True))
            dx[~valid] = 0.0
            dQ[q0:q1, h] += s * (dx @ km)
            dK[k0:k1, h] += s * (dx.T @ qm)
            if dBias is not None:
                dBias[h, :Lq, :Lk] += dx
    return dQ, dK, dV, dBias
