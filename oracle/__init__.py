"""CPU oracle for the triangle-attention forward (fp64, plain definition).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may use it; the product path
(``masked_attention_tri_gb300``) never imports it.  It shares no code with the
CUDA library.

``triattn_oracle.c`` holds the arithmetic (one query row at a time, every key,
index order, double precision); this module compiles it with gcc/OpenMP on
first use and wraps it for numpy / torch CPU tensors.  ``brute`` holds an
independent pure-Python restatement for tiny shapes; ``backward`` the
gradients of the triangle form (fp64 numpy, chain rule through the formula).

Each function follows the cuEquivariance ``triangle_attention`` API page
(formula; Parameters: bias, mask, scale, kv_lengths) or, for the packed form,
the Transformer Engine ``fused_attn.h`` page (NVTE_NOT_INTERLEAVED,
cu_seqlens) and the tensorplay ``BlockMask`` page (reconstruction loop,
full_kv_* lists).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "triattn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DT = {"f32": 0, "f16": 1, "bf16": 2}
MASK_MOD = {"none": 0, "causal": 1, "sliding_window": 2, "prefix_lm": 3}


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            LL = ctypes.c_longlong
            lib.oracle_tri_fwd.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, I, ctypes.c_double,
                                           P, LL, P, P, P, I]
            lib.oracle_tri_fwd.restype = I
            lib.oracle_varlen_fwd.argtypes = [P, P, P, I, P, P, I, I, I, ctypes.c_double,
                                              P, P, P, P, I, I, I, I, I, I, P, I, P, I, I, I, P, P, P, I]
            lib.oracle_varlen_fwd.restype = I
            lib.oracle_mask_to_kv_lengths.argtypes = [P, LL, I, P, P]
            lib.oracle_mask_to_kv_lengths.restype = None
            lib.oracle_widen.argtypes = [P, I, LL]
            lib.oracle_widen.restype = ctypes.c_double
            _lib = lib
    return _lib


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def _dtname(t: torch.Tensor) -> str:
    return {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[t.dtype]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cpu(t):
    return None if t is None else t.detach().to("cpu").contiguous()


def widen(t: torch.Tensor) -> np.ndarray:
    """Widen a stored f32/f16/bf16 tensor to fp64 with the oracle's own decoder."""
    lib = _load()
    t = _cpu(t)
    flat = t.reshape(-1)
    out = np.empty(flat.numel(), dtype=np.float64)
    for i in range(flat.numel()):
        out[i] = lib.oracle_widen(_ptr(flat), DT[_dtname(flat)], i)
    return out.reshape(tuple(t.shape))


def tri_fwd(q, k, v, bias, mask=None, kv_lengths=None, scale=None, rows=None, threads=None):
    """Triangle-attention forward in fp64.

    q (B,N,H,Q,D), k/v (B,N,H,K,D), bias (B,1,H,Q,K) in their stored dtypes;
    mask (B,N,1,1,K) any integer/bool (nonzero = valid) or kv_lengths (B,N)
    / (B,N,1,1,1) int.  rows: optional 1-D array of flat (b,n,h,q) indices to
    compute.  Returns numpy (O, lse, max) in fp64: O shaped like q (or
    (len(rows), D)), lse / max shaped (B,N,H,Q) (or (len(rows),)).
    """
    lib = _load()
    q, k, v, bias = _cpu(q), _cpu(k), _cpu(v), _cpu(bias)
    B, N, H, Q, D = q.shape
    K = k.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    s = float(np.float32(scale))  # the kernel receives the scale as a float
    m8 = None
    if mask is not None:
        m8 = (_cpu(mask).reshape(B, N, K) != 0).to(torch.uint8).contiguous()
    kl = None
    if kv_lengths is not None:
        kl = _cpu(kv_lengths).reshape(B, N).to(torch.int32).contiguous()
    if rows is not None:
        rows_t = torch.as_tensor(np.asarray(rows, dtype=np.int64)).contiguous()
        nrows = rows_t.numel()
        out = np.zeros((nrows, D), np.float64)
        lse = np.zeros(nrows, np.float64)
        mx = np.zeros(nrows, np.float64)
    else:
        rows_t = None
        nrows = 0
        out = np.zeros((B, N, H, Q, D), np.float64)
        lse = np.zeros((B, N, H, Q), np.float64)
        mx = np.zeros((B, N, H, Q), np.float64)
    rc = lib.oracle_tri_fwd(_ptr(q), _ptr(k), _ptr(v), DT[_dtname(q)], _ptr(bias), DT[_dtname(bias)],
                            _ptr(m8), _ptr(kl), B, N, H, Q, K, D, s, _ptr(rows_t), nrows,
                            out.ctypes.data_as(ctypes.c_void_p), lse.ctypes.data_as(ctypes.c_void_p),
                            mx.ctypes.data_as(ctypes.c_void_p), int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_tri_fwd: bad arguments")
    return out, lse, mx


def mask_to_kv_lengths(mask):
    """(B,N,1,1,K) mask -> (int32 (B,N) leading-valid counts, bool (B,N) is-prefix)."""
    lib = _load()
    m = _cpu(mask)
    B, N, K = m.shape[0], m.shape[1], m.shape[-1]
    m8 = (m.reshape(B * N, K) != 0).to(torch.uint8).contiguous()
    kl = torch.zeros(B * N, dtype=torch.int32)
    pre = torch.zeros(B * N, dtype=torch.uint8)
    lib.oracle_mask_to_kv_lengths(_ptr(m8), B * N, K, _ptr(kl), _ptr(pre))
    return kl.view(B, N), pre.view(B, N).bool()


def varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, scale=None, kv_num_blocks=None, kv_indices=None,
               full_kv_num_blocks=None, full_kv_indices=None, block=128, mask_mod="none",
               threads=None, window=0, prefix_lengths=None, bias=None):
    """Packed-sequence forward in fp64 with a BlockMask.

    q (total_q,H,D), k/v (total_k,H,D); cu_seqlens (S+1,) int.  Block lists are
    (S, mask_heads, MQ) / (S, mask_heads, MQ, MK) int, sequence-local.
    mask_mod on partial blocks: "none", "causal" (k <= q), "sliding_window"
    (q - window < k <= q) or "prefix_lm" (k <= q or k < the sequence's prefix
    length; prefix_lengths is an int or one int per sequence).  bias: optional
    (H, max_seqlen_q, max_seqlen_k) post-scale bias indexed by local positions.
    Returns numpy (O (total_q,H,D), lse (H,total_q), max (H,total_q)).
    """
    lib = _load()
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    total_q, H, D = q.shape
    cq = _cpu(cu_seqlens_q).to(torch.int32).contiguous()
    ck = _cpu(cu_seqlens_k).to(torch.int32).contiguous()
    S = cq.numel() - 1
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    s = float(np.float32(scale))

    def i32(t):
        return None if t is None else _cpu(t).to(torch.int32).contiguous()

    kn, ki, fn, fi = i32(kv_num_blocks), i32(kv_indices), i32(full_kv_num_blocks), i32(full_kv_indices)
    mask_heads, MQ, MK = 1, 1, 1
    if kn is not None:
        mask_heads, MQ = kn.shape[1], kn.shape[2]
        MK = ki.shape[3]
    bias_t = _cpu(bias)
    bq = bias_t.shape[1] if bias_t is not None else 0
    bk = bias_t.shape[2] if bias_t is not None else 0
    pl, p_all = None, 0
    if prefix_lengths is not None:
        if isinstance(prefix_lengths, int):
            p_all = prefix_lengths
        else:
            pl = torch.as_tensor(prefix_lengths).to(torch.int32).contiguous()
    out = np.zeros((total_q, H, D), np.float64)
    lse = np.zeros((H, total_q), np.float64)
    mx = np.zeros((H, total_q), np.float64)
    rc = lib.oracle_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), DT[_dtname(q)], _ptr(cq), _ptr(ck), S, H, D, s,
                               _ptr(kn), _ptr(ki), _ptr(fn), _ptr(fi), mask_heads, MQ, MK, block,
                               MASK_MOD[mask_mod], int(window), _ptr(pl), int(p_all),
                               _ptr(bias_t), DT[_dtname(bias_t)] if bias_t is not None else 0, bq, bk,
                               out.ctypes.data_as(ctypes.c_void_p),
                               lse.ctypes.data_as(ctypes.c_void_p), mx.ctypes.data_as(ctypes.c_void_p),
                               int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_varlen_fwd: bad arguments")
    return out, lse, mx


def to_dense(kv_num_blocks, kv_indices, cols):
    """The BlockMask page's reconstruction loop, for one (ROWS,) / (ROWS, MAX) pair.

    dense[row, kv_indices[row, t]] = 1 for t < kv_num_blocks[row]; later
    entries are never read.  Out-of-range column indices are ignored.
    """
    num = np.asarray(kv_num_blocks)
    idx = np.asarray(kv_indices)
    rows = num.shape[0]
    dense = np.zeros((rows, cols), np.uint8)
    for r in range(rows):
        for t in range(int(num[r])):
            c = int(idx[r, t])
            if 0 <= c < cols:
                dense[r, c] = 1
    return dense
