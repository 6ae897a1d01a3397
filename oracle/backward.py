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
