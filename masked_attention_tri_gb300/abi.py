"""ctypes binding of libtriattn.so: one Python function per C entry point, same names.

Argument marshalling only (pointers and sizes in, status code out); every step
of the computation runs in the library's CUDA kernels.  A non-OK status is
raised: TA_ERR_INVALID_ARG as ValueError, TA_ERR_UNSUPPORTED as
NotImplementedError, anything else as RuntimeError.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtriattn.so")

TA_OK, TA_ERR_INVALID_ARG, TA_ERR_UNSUPPORTED, TA_ERR_CUDA, TA_ERR_TIMEOUT, TA_ERR_DEVICE = range(6)
TA_F32, TA_F16, TA_BF16 = 0, 1, 2
TA_MASK_NONE, TA_MASK_CAUSAL, TA_MASK_SLIDING_WINDOW, TA_MASK_PREFIX_LM = 0, 1, 2, 3

# Every symbol include/triattn.h declares.
EXPORTS = ("tri_attn_fwd", "tri_attn_fwd_strided", "tri_attn_varlen_fwd", "tri_attn_varlen_fwd_strided", "tri_attn_varlen_fwd_masked",
           "tri_attn_bwd", "tri_attn_bwd_workspace_size", "tri_attn_bwd_noalloc", "tri_attn_varlen_bwd",
           "tri_attn_varlen_bwd_workspace_size",
           "tri_attn_mask_to_kv_lengths", "tri_attn_get_status", "tri_attn_error_string", "tri_attn_version")

_lock = threading.Lock()
_lib = None


class TriAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def load() -> ctypes.CDLL:
    """Load the built library; raise loudly if it is missing (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run masked_attention_tri_gb300.build.build() "
                              "(nvcc, sm_103a) first")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.tri_attn_fwd.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, I, F, P, P, P, P]
        lib.tri_attn_fwd.restype = I
        lib.tri_attn_fwd_strided.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, I, F, P, P, P, P, P, P, P]
        lib.tri_attn_fwd_strided.restype = I
        lib.tri_attn_varlen_fwd.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, F, P, P, P, P, I, I, I, I, I, I,
                                            P, P, P, P]
        lib.tri_attn_varlen_fwd.restype = I
        L = ctypes.c_longlong
        lib.tri_attn_varlen_fwd_strided.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, F, P, P, P, P, I, I, I, I,
                                                    I, I, L, L, L, P, P, P, P]
        lib.tri_attn_varlen_fwd_strided.restype = I
        lib.tri_attn_varlen_fwd_masked.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, F, P, P, P, P, I, I, I, I,
                                                   I, I, I, P, I, P, I, L, L, L, P, P, P, P]
        lib.tri_attn_varlen_fwd_masked.restype = I
        Z = ctypes.c_size_t
        lib.tri_attn_bwd.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, I, F, P, P, P, P, P, P, P, P, Z, P]
        lib.tri_attn_bwd.restype = I
        lib.tri_attn_bwd_noalloc.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, I, F, P, P, P, P, P, P, P, P]
        lib.tri_attn_bwd_noalloc.restype = I
        lib.tri_attn_varlen_bwd.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, F, P, P, P, P, I, I, I, I, I, I,
                                            I, P, I, P, I, P, P, P, P, P, P, P, P, Z, P]
        lib.tri_attn_varlen_bwd.restype = I
        lib.tri_attn_varlen_bwd_workspace_size.argtypes = [I, I, I, I, I, I]
        lib.tri_attn_varlen_bwd_workspace_size.restype = Z
        lib.tri_attn_bwd_workspace_size.argtypes = [I, I, I, I, I, I]
        lib.tri_attn_bwd_workspace_size.restype = Z
        lib.tri_attn_mask_to_kv_lengths.argtypes = [P, I, I, I, P, P, P]
        lib.tri_attn_mask_to_kv_lengths.restype = I
        lib.tri_attn_get_status.argtypes = [P]
        lib.tri_attn_get_status.restype = I
        lib.tri_attn_error_string.argtypes = [I]
        lib.tri_attn_error_string.restype = ctypes.c_char_p
        lib.tri_attn_version.argtypes = []
        lib.tri_attn_version.restype = I
        _lib = lib
        return lib


def tri_attn_error_string(status: int) -> str:
    return load().tri_attn_error_string(int(status)).decode()


def _check(status: int, fn: str) -> None:
    if status == TA_OK:
        return
    msg = f"{fn}: {tri_attn_error_string(status)} (status {status})"
    if status == TA_ERR_INVALID_ARG:
        raise ValueError(msg)
    if status == TA_ERR_UNSUPPORTED:
        raise NotImplementedError(msg)
    raise TriAttnError(status, msg)


def tri_attn_fwd(q, k, v, qkv_dtype, bias, bias_dtype, mask, kv_lengths, B, N, H, Q, K, D, scale, out, lse, max_,
                 stream) -> None:
    """Pointers are ints (0 = NULL); stream is a cudaStream_t handle as int."""
    st = load().tri_attn_fwd(q, k, v, qkv_dtype, bias, bias_dtype, mask or None, kv_lengths or None, B, N, H, Q, K,
                             D, float(scale), out, lse or None, max_ or None, stream or None)
    _check(st, "tri_attn_fwd")


def tri_attn_bwd(q, k, v, qkv_dtype, bias, bias_dtype, mask, kv_lengths, B, N, H, Q, K, D, scale, lse, out, d_out,
                 dq, dk, dv, dbias, workspace, workspace_bytes, stream) -> None:
    """Gradients of tri_attn_fwd; pointers are ints (0 = NULL), workspace_bytes an int."""
    st = load().tri_attn_bwd(q, k, v, qkv_dtype, bias, bias_dtype, mask or None, kv_lengths or None, B, N, H, Q, K, D,
                             float(scale), lse, out or None, d_out, dq, dk, dv, dbias or None, workspace,
                             int(workspace_bytes), stream or None)
    _check(st, "tri_attn_bwd")


def tri_attn_bwd_noalloc(q, k, v, qkv_dtype, bias, bias_dtype, mask, kv_lengths, B, N, H, Q, K, D, scale, lse, out,
                         d_out, dq, dk, dv, dbias, stream) -> None:
    """tri_attn_bwd in the library's own static scratch (no workspace, no allocation)."""
    st = load().tri_attn_bwd_noalloc(q, k, v, qkv_dtype, bias, bias_dtype, mask or None, kv_lengths or None, B, N, H,
                                     Q, K, D, float(scale), lse, out or None, d_out, dq, dk, dv, dbias or None,
                                     stream or None)
    _check(st, "tri_attn_bwd_noalloc")


# Bytes of the static scratch tri_attn_bwd_noalloc works in (TRI_ATTN_BWD_NOALLOC_SCRATCH_BYTES).
BWD_NOALLOC_SCRATCH_BYTES = 16 << 20


def tri_attn_varlen_bwd(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                        max_seqlen_k, H, D, scale, kv_num_blocks, kv_indices, full_kv_num_blocks, full_kv_indices,
                        mask_heads, max_q_blocks, max_kv_blocks, block_q, block_k, mask_mod, window,
                        prefix_lengths, prefix_length, bias, bias_dtype, lse, out, d_out, dq, dk, dv, dbias,
                        workspace, workspace_bytes, stream) -> None:
    st = load().tri_attn_varlen_bwd(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                                    max_seqlen_q, max_seqlen_k, H, D, float(scale), kv_num_blocks or None,
                                    kv_indices or None, full_kv_num_blocks or None, full_kv_indices or None,
                                    mask_heads, max_q_blocks, max_kv_blocks, block_q, block_k, mask_mod, window,
                                    prefix_lengths or None, prefix_length, bias or None, bias_dtype, lse, out,
                                    d_out, dq, dk, dv, dbias or None, workspace, int(workspace_bytes),
                                    stream or None)
    _check(st, "tri_attn_varlen_bwd")


def tri_attn_varlen_bwd_workspace_size(total_q, H, D, max_seqlen_q, max_seqlen_k, with_bias) -> int:
    return int(load().tri_attn_varlen_bwd_workspace_size(total_q, H, D, max_seqlen_q, max_seqlen_k,
                                                         1 if with_bias else 0))


def tri_attn_bwd_workspace_size(B, N, H, Q, K, D) -> int:
    return int(load().tri_attn_bwd_workspace_size(B, N, H, Q, K, D))


def _strides4(st):
    """A host array of 4 element strides (b, n, h, row) for the C call, or None (contiguous)."""
    return None if st is None else (ctypes.c_longlong * 4)(*[int(x) for x in st])


def tri_attn_fwd_strided(q, k, v, qkv_dtype, bias, bias_dtype, mask, kv_lengths, B, N, H, Q, K, D, scale, q_strides,
                         k_strides, v_strides, out, lse, max_, stream) -> None:
    """q_strides / k_strides / v_strides: 4 element strides (b, n, h, row) each, or None."""
    qs, ks, vs = _strides4(q_strides), _strides4(k_strides), _strides4(v_strides)
    st = load().tri_attn_fwd_strided(q, k, v, qkv_dtype, bias, bias_dtype, mask or None, kv_lengths or None, B, N, H,
                                     Q, K, D, float(scale), qs, ks, vs, out, lse or None, max_ or None,
                                     stream or None)
    _check(st, "tri_attn_fwd_strided")


def tri_attn_varlen_fwd(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                        max_seqlen_k, H, D, scale, kv_num_blocks, kv_indices, full_kv_num_blocks, full_kv_indices, mask_heads,
                        max_q_blocks, max_kv_blocks, block_q, block_k, mask_mod, out, lse, max_, stream) -> None:
    st = load().tri_attn_varlen_fwd(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                                    max_seqlen_q, max_seqlen_k, H, D, float(scale), kv_num_blocks or None, kv_indices or None,
                                    full_kv_num_blocks or None, full_kv_indices or None, mask_heads, max_q_blocks,
                                    max_kv_blocks, block_q, block_k, mask_mod, out, lse or None, max_ or None,
                                    stream or None)
    _check(st, "tri_attn_varlen_fwd")


def tri_attn_varlen_fwd_strided(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                                max_seqlen_q, max_seqlen_k, H, D, scale, kv_num_blocks, kv_indices, full_kv_num_blocks,
                                full_kv_indices, mask_heads, max_q_blocks, max_kv_blocks, block_q, block_k, mask_mod,
                                q_row_stride, k_row_stride, v_row_stride, out, lse, max_, stream) -> None:
    st = load().tri_attn_varlen_fwd_strided(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                                            max_seqlen_q, max_seqlen_k, H, D, float(scale), kv_num_blocks or None,
                                            kv_indices or None, full_kv_num_blocks or None, full_kv_indices or None,
                                            mask_heads, max_q_blocks, max_kv_blocks, block_q, block_k, mask_mod,
                                            int(q_row_stride), int(k_row_stride), int(v_row_stride), out,
                                            lse or None, max_ or None, stream or None)
    _check(st, "tri_attn_varlen_fwd_strided")


def tri_attn_varlen_fwd_masked(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                               max_seqlen_q, max_seqlen_k, H, D, scale, kv_num_blocks, kv_indices, full_kv_num_blocks,
                               full_kv_indices, mask_heads, max_q_blocks, max_kv_blocks, block_q, block_k, mask_mod,
                               window, prefix_lengths, prefix_length, bias, bias_dtype, q_row_stride, k_row_stride,
                               v_row_stride, out, lse, max_, stream) -> None:
    st = load().tri_attn_varlen_fwd_masked(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                                           max_seqlen_q, max_seqlen_k, H, D, float(scale), kv_num_blocks or None,
                                           kv_indices or None, full_kv_num_blocks or None, full_kv_indices or None,
                                           mask_heads, max_q_blocks, max_kv_blocks, block_q, block_k, mask_mod,
                                           int(window), prefix_lengths or None, int(prefix_length), bias or None,
                                           int(bias_dtype), int(q_row_stride), int(k_row_stride), int(v_row_stride), out,
                                           lse or None, max_ or None, stream or None)
    _check(st, "tri_attn_varlen_fwd_masked")


def tri_attn_mask_to_kv_lengths(mask, B, N, K, kv_lengths, nonprefix_count, stream) -> None:
    st = load().tri_attn_mask_to_kv_lengths(mask, B, N, K, kv_lengths, nonprefix_count or None, stream or None)
    _check(st, "tri_attn_mask_to_kv_lengths")


def tri_attn_get_status(stream) -> int:
    """Synchronize the stream and return (and clear) the device status word."""
    return int(load().tri_attn_get_status(stream or None))


def tri_attn_version() -> int:
    return int(load().tri_attn_version())
