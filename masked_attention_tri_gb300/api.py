"""PyTorch-facing API over the C ABI.

Mirrors the cuEquivariance ``triangle_attention`` signature (with its
backward through ``triangle_attention_autograd`` / ``triangle_attention_backward``)
and adds the packed-sequence entry with a tensorplay-style ``BlockMask``.
PyTorch provides device memory and the current stream; the work is done by
libtriattn.so's kernels.  Inputs are used in place (no casts or copies): they
must be contiguous CUDA tensors of the documented dtypes.
"""
from __future__ import annotations

import math
from typing import Optional

import torch

from . import abi

_DT = {torch.float32: abi.TA_F32, torch.float16: abi.TA_F16, torch.bfloat16: abi.TA_BF16}
_MASK_MODS = {None: abi.TA_MASK_NONE, "none": abi.TA_MASK_NONE, "causal": abi.TA_MASK_CAUSAL,
              "sliding_window": abi.TA_MASK_SLIDING_WINDOW, "prefix_lm": abi.TA_MASK_PREFIX_LM}


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, device: torch.device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_out(out, shape, dtype) -> None:
    """A preallocated output must be exactly what the kernels write: they store whole rows of
    `shape` in `dtype`, so a smaller or differently typed buffer would be overrun."""
    if not isinstance(out, torch.Tensor):
        raise TypeError("out must be a torch.Tensor")
    if tuple(out.shape) != tuple(shape) or out.dtype != dtype:
        raise ValueError(f"out must be {tuple(shape)} of {dtype}, got {tuple(out.shape)} of {out.dtype}")


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def triangle_attention(q, k, v, bias, mask=None, scale=None, return_aux=False, *, kv_lengths=None, out=None,
                       lse=None, mx=None):
    """Triangle-attention forward (cuEquivariance triangle_attention page: formula, Parameters).

    q (B,N,H,Q,D), k/v (B,N,H,K,D), bias (B,1,H,Q,K); for B=1 the 4-D forms
    (N,H,Q,D) / (1,H,Q,K) / (N,1,1,K) are accepted.  q, k, v may be strided
    views whose last dimension is contiguous (e.g. a (B,N,Q,H,D) buffer
    transposed to (B,N,H,Q,D)); they are read in place.  mask: bool/uint8
    (B,N,1,1,K); kv_lengths: int32 (B,N,1,1,1) or (B,N); at most one of them.
    scale defaults to 1/sqrt(D).  Returns O, or (O, lse, max) with
    return_aux (lse / max fp32 shaped (B,N,H,Q,1)).  out, lse, mx may be given
    preallocated (contiguous, on q's device); lse / mx are written only with
    return_aux.
    """
    if mask is not None and kv_lengths is not None:
        raise ValueError("pass either mask or kv_lengths, not both")
    four_d = q.dim() == 4
    if four_d:
        q, k, v = q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0)
        if bias.dim() == 4:
            bias = bias.unsqueeze(0)
        if mask is not None and mask.dim() == 4:
            mask = mask.unsqueeze(0)
    if q.dim() != 5 or k.dim() != 5 or v.dim() != 5 or bias.dim() != 5:
        raise ValueError("expected q/k/v (B,N,H,Q|K,D) and bias (B,1,H,Q,K)")
    B, N, H, Q, D = q.shape
    K = k.shape[3]
    if tuple(k.shape) != (B, N, H, K, D) or tuple(v.shape) != (B, N, H, K, D):
        raise ValueError(f"k/v must be {(B, N, H, K, D)}, got {tuple(k.shape)} / {tuple(v.shape)}")
    if tuple(bias.shape) != (B, 1, H, Q, K):
        raise ValueError(f"bias must be {(B, 1, H, Q, K)}, got {tuple(bias.shape)}")
    if out is not None:
        _check_out(out, tuple(q.shape), q.dtype)
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("triangle_attention runs on CUDA tensors only")
    _need(bias, "bias", dev)
    strides = []
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        if not isinstance(t, torch.Tensor) or t.device != dev:
            raise ValueError(f"{nm} must be a tensor on {dev}")
        if t.stride(4) != 1:
            raise ValueError(f"{nm}: the last dimension (D) must be contiguous")
        # None = contiguous (the plain entry point)
        strides.append(None if t.is_contiguous() else tuple(t.stride(i) for i in range(4)))
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype among float32 / float16 / bfloat16")
    if bias.dtype not in (torch.float32, q.dtype):
        raise TypeError("bias must be float32 or q's dtype")
    m8 = None
    if mask is not None:
        if tuple(mask.shape) != (B, N, 1, 1, K):
            raise ValueError(f"mask must be {(B, N, 1, 1, K)}, got {tuple(mask.shape)}")
        if mask.dtype not in (torch.bool, torch.uint8, torch.int8):
            raise TypeError("mask must be bool, uint8 or int8 (nonzero = valid)")
        _need(mask, "mask", dev)
        m8 = mask.view(torch.uint8)
    kl = None
    if kv_lengths is not None:
        if kv_lengths.dtype != torch.int32 or kv_lengths.numel() != B * N:
            raise ValueError("kv_lengths must be int32 with B*N elements ((B,N,1,1,1) or (B,N))")
        _need(kv_lengths, "kv_lengths", dev)
        kl = kv_lengths
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=dev)
    else:
        _need(out, "out", dev)
    if return_aux:
        for name, t in (("lse", lse), ("mx", mx)):
            if t is not None:
                _need(t, name, dev)
                if t.dtype != torch.float32 or t.numel() != B * N * H * Q:
                    raise ValueError(f"{name} must be float32 with B*N*H*Q elements")
        if lse is None:
            lse = torch.empty(B, N, H, Q, 1, device=dev, dtype=torch.float32)
        if mx is None:
            mx = torch.empty(B, N, H, Q, 1, device=dev, dtype=torch.float32)
    else:
        lse = mx = None
    with torch.cuda.device(dev):
        if strides == [None, None, None]:
            abi.tri_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(bias), _DT[bias.dtype], _ptr(m8),
                             _ptr(kl), B, N, H, Q, K, D, s, _ptr(out), _ptr(lse), _ptr(mx), _stream(dev))
        else:
            full = [st if st is not None else tuple(t.stride(i) for i in range(4)) for st, t in zip(strides, (q, k, v))]
            abi.tri_attn_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(bias), _DT[bias.dtype], _ptr(m8),
                                     _ptr(kl), B, N, H, Q, K, D, s, full[0], full[1], full[2], _ptr(out), _ptr(lse),
                                     _ptr(mx), _stream(dev))
    if four_d:
        out = out.squeeze(0)
        if return_aux:
            lse, mx = lse.squeeze(0), mx.squeeze(0)
    return (out, lse, mx) if return_aux else out


def triangle_attention_backward(q, k, v, bias, lse, d_out, mask=None, scale=None, *, kv_lengths=None,
                                need_dbias=True, out=None):
    """Gradients (dq, dk, dv, dbias) of triangle_attention for dL/dO = d_out.

    q, k, v, bias, mask / kv_lengths and scale as given to the forward
    (contiguous 5-D tensors); lse: the forward's lse (return_aux), fp32 with
    B*N*H*Q elements; d_out like q; out, optional, the forward's O (then the
    per-row sum of P dP is the row sum of dO * O, else it is formed exactly).
    dbias has the bias's shape and dtype (the sum over n), or is None without
    need_dbias.  The fp32 workspace is taken
    from PyTorch's allocator on q's device.
    """
    if mask is not None and kv_lengths is not None:
        raise ValueError("pass either mask or kv_lengths, not both")
    if q.dim() != 5 or k.dim() != 5 or v.dim() != 5 or bias.dim() != 5:
        raise ValueError("expected q/k/v (B,N,H,Q|K,D) and bias (B,1,H,Q,K)")
    B, N, H, Q, D = q.shape
    K = k.shape[3]
    if tuple(k.shape) != (B, N, H, K, D) or tuple(v.shape) != (B, N, H, K, D):
        raise ValueError(f"k/v must be {(B, N, H, K, D)}")
    if tuple(bias.shape) != (B, 1, H, Q, K):
        raise ValueError(f"bias must be {(B, 1, H, Q, K)}")
    if tuple(d_out.shape) != tuple(q.shape) or d_out.dtype != q.dtype:
        raise ValueError("d_out must have q's shape and dtype")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("triangle_attention_backward runs on CUDA tensors only")
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (bias, "bias"), (lse, "lse"), (d_out, "d_out")):
        _need(t, nm, dev)
    if out is not None:
        _need(out, "out", dev)
        if tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype:
            raise ValueError("out must have q's shape and dtype")
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype among float32 / float16 / bfloat16")
    if bias.dtype not in (torch.float32, q.dtype):
        raise TypeError("bias must be float32 or q's dtype")
    if lse.dtype != torch.float32 or lse.numel() != B * N * H * Q:
        raise ValueError("lse must be float32 with B*N*H*Q elements")
    m8 = kl = None
    if mask is not None:
        if tuple(mask.shape) != (B, N, 1, 1, K) or mask.dtype not in (torch.bool, torch.uint8, torch.int8):
            raise ValueError(f"mask must be bool/uint8/int8 {(B, N, 1, 1, K)}")
        _need(mask, "mask", dev)
        m8 = mask.view(torch.uint8)
    if kv_lengths is not None:
        if kv_lengths.dtype != torch.int32 or kv_lengths.numel() != B * N:
            raise ValueError("kv_lengths must be int32 with B*N elements")
        _need(kv_lengths, "kv_lengths", dev)
        kl = kv_lengths
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dbias = torch.empty_like(bias) if need_dbias else None
    nbytes = abi.tri_attn_bwd_workspace_size(B, N, H, Q, K, D)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        abi.tri_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(bias), _DT[bias.dtype], _ptr(m8), _ptr(kl),
                         B, N, H, Q, K, D, s, _ptr(lse), _ptr(out), _ptr(d_out), _ptr(dq), _ptr(dk), _ptr(dv),
                         _ptr(dbias),
                         _ptr(ws), nbytes, _stream(dev))
    return dq, dk, dv, dbias


class _TriangleAttentionFn(torch.autograd.Function):
    """Autograd node: the forward saves q, k, v, bias, the mask and lse; the
    backward runs tri_attn_bwd (the page's Notes 1: context saved for backward)."""

    @staticmethod
    def forward(ctx, q, k, v, bias, mask, kv_lengths, scale):
        o, lse, mx = triangle_attention(q, k, v, bias, mask, scale, True, kv_lengths=kv_lengths)
        ctx.save_for_backward(q, k, v, bias, mask, kv_lengths, lse, o)
        ctx.scale = scale
        ctx.mark_non_differentiable(lse, mx)
        return o, lse, mx

    @staticmethod
    def backward(ctx, d_out, _d_lse, _d_mx):
        q, k, v, bias, mask, kv_lengths, lse, o = ctx.saved_tensors
        dq, dk, dv, dbias = triangle_attention_backward(q, k, v, bias, lse, d_out.contiguous(), mask, ctx.scale,
                                                        kv_lengths=kv_lengths, need_dbias=ctx.needs_input_grad[3],
                                                        out=o)
        return dq, dk, dv, dbias, None, None, None


def triangle_attention_autograd(q, k, v, bias, mask=None, scale=None, return_aux=False, *, kv_lengths=None):
    """triangle_attention with gradients for q, k, v and bias (contiguous 5-D inputs, or the
    B=1 4-D forms).  Returns O, or (O, lse, max) with return_aux."""
    four_d = q.dim() == 4
    if four_d:
        q, k, v = q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0)
        if bias.dim() == 4:
            bias = bias.unsqueeze(0)
        if mask is not None and mask.dim() == 4:
            mask = mask.unsqueeze(0)
    o, lse, mx = _TriangleAttentionFn.apply(q, k, v, bias, mask, kv_lengths, scale)
    if four_d:
        o, lse, mx = o.squeeze(0), lse.squeeze(0), mx.squeeze(0)
    return (o, lse, mx) if return_aux else o


def mask_to_kv_lengths(mask: torch.Tensor, return_nonprefix: bool = False):
    """(B,N,1,1,K) key mask -> int32 (B,N,1,1,1) counts of leading valid keys.

    The triangle_attention page's Example uses this to turn a right-padded
    mask into kv_lengths.  With return_nonprefix, also returns a 1-element
    int32 tensor counting rows that are not a prefix mask.
    """
    if mask.dim() == 4:
        mask = mask.unsqueeze(0)
    B, N, K = mask.shape[0], mask.shape[1], mask.shape[-1]
    if mask.numel() != B * N * K:
        raise ValueError("mask must be (B,N,1,1,K)")
    if mask.dtype not in (torch.bool, torch.uint8, torch.int8):
        raise TypeError("mask must be bool, uint8 or int8")
    dev = mask.device
    _need(mask, "mask", dev)
    kl = torch.empty(B, N, 1, 1, 1, device=dev, dtype=torch.int32)
    cnt = torch.zeros(1, device=dev, dtype=torch.int32) if return_nonprefix else None
    with torch.cuda.device(dev):
        abi.tri_attn_mask_to_kv_lengths(_ptr(mask.view(torch.uint8)), B, N, K, _ptr(kl), _ptr(cnt), _stream(dev))
    return (kl, cnt) if return_nonprefix else kl


class BlockMask:
    """Block-sparse mask in the tensorplay BlockMask format (kv side, forward only).

    kv_num_blocks (S, Hm, MQ) and kv_indices (S, Hm, MQ, MK): partial blocks
    of each q block, where mask_mod applies; full_kv_* (optional, same shapes):
    blocks where every key is valid.  Indices are sequence-local 128-row
    blocks.  mask_mod is None, "causal", "sliding_window" or "prefix_lm" (a C
    ABI cannot take a callable; the last two take their parameter from
    ``varlen_attention``'s ``window`` / ``prefix_lengths``).
    seq_lengths (q_len, kv_len), as on the page's from_kv_blocks, fixes the
    number of kv blocks, i.e. the columns of ``to_dense``; without it the
    columns are the larger of MK and the highest listed block index + 1.
    """

    def __init__(self, kv_num_blocks, kv_indices, full_kv_num_blocks=None, full_kv_indices=None, BLOCK_SIZE=128,
                 mask_mod=None, seq_lengths=None):
        self.kv_num_blocks = kv_num_blocks
        self.kv_indices = kv_indices
        self.full_kv_num_blocks = full_kv_num_blocks
        self.full_kv_indices = full_kv_indices
        self.BLOCK_SIZE = (BLOCK_SIZE, BLOCK_SIZE) if isinstance(BLOCK_SIZE, int) else tuple(BLOCK_SIZE)
        self.mask_mod = mask_mod
        self.seq_lengths = None if seq_lengths is None else (int(seq_lengths[0]), int(seq_lengths[1]))

    @classmethod
    def from_kv_blocks(cls, kv_num_blocks, kv_indices, full_kv_num_blocks=None, full_kv_indices=None,
                       BLOCK_SIZE=128, mask_mod=None, seq_lengths=None):
        """Same error rules as the BlockMask page's from_kv_blocks (Raises)."""
        if kv_indices.dim() < 2:
            raise RuntimeError("BlockMask must have at least 2 dimensions")
        assert (full_kv_num_blocks is None) == (full_kv_indices is None), \
            "full_kv_num_blocks and full_kv_indices must be both provided or omitted"
        if mask_mod not in _MASK_MODS:
            raise ValueError(f"mask_mod must be one of {sorted(k for k in _MASK_MODS if k)} or None")
        return cls(kv_num_blocks, kv_indices, full_kv_num_blocks, full_kv_indices, BLOCK_SIZE, mask_mod,
                   seq_lengths)

    @property
    def mask_mod_code(self) -> int:
        return _MASK_MODS[self.mask_mod]

    def _lists(self):
        pairs = [(self.kv_num_blocks.cpu(), self.kv_indices.cpu())]
        if self.full_kv_num_blocks is not None:
            pairs.append((self.full_kv_num_blocks.cpu(), self.full_kv_indices.cpu()))
        return pairs

    def num_kv_blocks(self) -> int:
        """Columns of the dense block mask (kv blocks per row)."""
        if self.seq_lengths is not None:
            kb = self.BLOCK_SIZE[1] if len(self.BLOCK_SIZE) > 1 else self.BLOCK_SIZE[0]
            return (self.seq_lengths[1] + kb - 1) // kb
        cols = int(self.kv_indices.shape[-1])
        for nb, ix in self._lists():
            flat_n = nb.reshape(-1)
            flat_i = ix.reshape(flat_n.numel(), -1)
            for r in range(flat_n.numel()):
                n = min(max(int(flat_n[r]), 0), flat_i.shape[1])
                if n:
                    cols = max(cols, int(flat_i[r, :n].max()) + 1)
        return cols

    def numel(self) -> int:
        """Blocks in the mask, not accounting for sparsity (q blocks x kv blocks x leading dims)."""
        n = 1
        for x in self.kv_num_blocks.shape:
            n *= int(x)
        return n * self.num_kv_blocks()

    def to_dense(self) -> torch.Tensor:
        """Dense (..., MQ, num_kv_blocks) block mask: 1 where a block is listed (partial or full).

        The page's reconstruction loop: for each row, the first kv_num_blocks[row]
        entries of kv_indices[row] are set; later entries are never read."""
        cols = self.num_kv_blocks()
        num = self.kv_num_blocks.cpu()
        dense = torch.zeros(*num.shape, cols, dtype=torch.int32)
        flat_d = dense.view(-1, cols)
        for nb, ix in self._lists():
            flat_n = nb.reshape(-1)
            flat_i = ix.reshape(flat_n.numel(), -1)
            for r in range(flat_n.numel()):
                for t in range(min(int(flat_n[r]), flat_i.shape[1])):
                    c = int(flat_i[r, t])
                    if 0 <= c < cols:
                        flat_d[r, c] = 1
        return dense

    def sparsity(self) -> float:
        """Percentage of blocks that are not computed."""
        dense = self.to_dense()
        return 100.0 * (1.0 - float(dense.sum()) / max(1, dense.numel()))


def _row_stride(t: torch.Tensor, name: str, device: torch.device) -> int:
    """Row stride (elements) of a (total, H, D) view whose heads and elements are contiguous."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    rows, H, D = t.shape
    if t.stride(2) != 1 or (H > 1 and t.stride(1) != D):
        raise ValueError(f"{name} must have contiguous heads and elements (strides (*, D, 1))")
    if rows <= 1:
        return H * D
    if t.stride(0) < H * D:
        # Rows that overlap (an expanded or otherwise aliased view, stride 0 included) would make
        # the kernels read rows*H*D elements from a smaller allocation.
        raise ValueError(f"{name} rows overlap (row stride {t.stride(0)} < H*D = {H * D}); pass a "
                         "contiguous tensor")
    return t.stride(0)


def _mask_args(block_mask, mask_mod, dev):
    """The C ABI's block-mask arguments of a BlockMask (or none) and a mask_mod name."""
    kn = ki = fn = fi = None
    mask_heads = MQ = MK = 0
    bq = bk = 128
    if mask_mod not in _MASK_MODS:
        raise ValueError(f"mask_mod must be one of {sorted(k for k in _MASK_MODS if k)} or None")
    mm = _MASK_MODS[mask_mod]
    if block_mask is not None:
        kn, ki = block_mask.kv_num_blocks, block_mask.kv_indices
        fn, fi = block_mask.full_kv_num_blocks, block_mask.full_kv_indices
        for t, nm in ((kn, "kv_num_blocks"), (ki, "kv_indices"), (fn, "full_kv_num_blocks"),
                      (fi, "full_kv_indices")):
            if t is not None:
                _need(t, nm, dev)
                if t.dtype != torch.int32:
                    raise TypeError(f"{nm} must be int32")
        if kn.dim() != 3 or ki.dim() != 4:
            raise ValueError("kv_num_blocks must be (S, Hm, MQ) and kv_indices (S, Hm, MQ, MK)")
        mask_heads, MQ, MK = kn.shape[1], kn.shape[2], ki.shape[3]
        if fn is not None and (tuple(fn.shape) != tuple(kn.shape) or tuple(fi.shape) != tuple(ki.shape)):
            raise ValueError("full_kv_* must have the shapes of kv_*")
        bq, bk = block_mask.BLOCK_SIZE
        mm = block_mask.mask_mod_code
    return kn, ki, fn, fi, mask_heads, MQ, MK, bq, bk, mm


def _prefix_args(prefix_lengths, S, dev):
    """(per-sequence tensor or None, one length for all) for the prefix-LM mask_mod."""
    if isinstance(prefix_lengths, torch.Tensor):
        _need(prefix_lengths, "prefix_lengths", dev)
        if prefix_lengths.dtype != torch.int32 or prefix_lengths.numel() != S:
            raise ValueError("prefix_lengths must be int32 with one entry per sequence")
        return prefix_lengths, 0
    return None, (0 if prefix_lengths is None else int(prefix_lengths))


def varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, block_mask=None, scale=None,
                     return_aux=False, *, mask_mod=None, out=None, window=0, prefix_lengths=None, bias=None):
    """Packed-sequence forward with an optional BlockMask.

    q (total_q,H,D), k/v (total_k,H,D), cu_seqlens int32 (S+1,).  q, k, v may
    be row-strided views (heads and elements contiguous), e.g. the slices of
    an interleaved QKV or KV buffer (see ``varlen_attention_qkvpacked`` /
    ``varlen_attention_kvpacked``); ``out`` is contiguous.  Without a
    block_mask every block is visited and ``mask_mod`` applies everywhere.
    mask_mod: None, "causal" (k <= q), "sliding_window" (q - window < k <= q)
    or "prefix_lm" (k <= q or k < the sequence's prefix; ``prefix_lengths`` is
    an int or an int32 CUDA tensor with one length per sequence).  bias: an
    optional post-scale bias (H, max_seqlen_q, max_seqlen_k), float32 or q's
    dtype, indexed by each sequence's local positions.
    Returns O, or (O, lse, max) with lse/max (H, total_q).
    """
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("expected q (total_q,H,D), k/v (total_k,H,D)")
    total_q, H, D = q.shape
    if tuple(k.shape[1:]) != (H, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be (total_k, H, D) with q's H and D")
    if out is not None:
        _check_out(out, (total_q, H, D), q.dtype)
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("varlen_attention runs on CUDA tensors only")
    q_rs, k_rs, v_rs = (_row_stride(t, nm, dev) for t, nm in ((q, "q"), (k, "k"), (v, "v")))
    for t, nm in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _need(t, nm, dev)
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype among float32 / float16 / bfloat16")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    S = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != S + 1 or S <= 0:
        raise ValueError("cu_seqlens_q / cu_seqlens_k must both have num_seqs + 1 entries")
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    kn, ki, fn, fi, mask_heads, MQ, MK, bq, bk, mm = _mask_args(block_mask, mask_mod, dev)
    if out is None:
        out = torch.empty(total_q, H, D, device=dev, dtype=q.dtype)
    else:
        _need(out, "out", dev)
    lse = mx = None
    if return_aux:
        lse = torch.empty(H, total_q, device=dev, dtype=torch.float32)
        mx = torch.empty(H, total_q, device=dev, dtype=torch.float32)
    if bias is not None:
        _need(bias, "bias", dev)
        if tuple(bias.shape) != (H, int(max_seqlen_q), int(max_seqlen_k)):
            raise ValueError(f"bias must be (H, max_seqlen_q, max_seqlen_k) = {(H, int(max_seqlen_q), int(max_seqlen_k))}")
        if bias.dtype not in (torch.float32, q.dtype):
            raise TypeError("bias must be float32 or q's dtype")
    pl, p_all = _prefix_args(prefix_lengths, S, dev)
    with torch.cuda.device(dev):
        abi.tri_attn_varlen_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(cu_seqlens_q),
                                       _ptr(cu_seqlens_k), S, total_q, k.shape[0], int(max_seqlen_q),
                                       int(max_seqlen_k), H, D, s, _ptr(kn), _ptr(ki), _ptr(fn), _ptr(fi),
                                       mask_heads, MQ, MK, bq, bk, mm, int(window), _ptr(pl), p_all, _ptr(bias),
                                       _DT[bias.dtype] if bias is not None else abi.TA_F32, q_rs, k_rs, v_rs,
                                       _ptr(out), _ptr(lse), _ptr(mx), _stream(dev))
    return (out, lse, mx) if return_aux else out


def varlen_attention_qkvpacked(qkv, cu_seqlens, max_seqlen, block_mask=None, scale=None, return_aux=False, *,
                               mask_mod=None, out=None, window=0, prefix_lengths=None):
    """NVTE_QKV_INTERLEAVED (Transformer Engine fused_attn.h): one (total, 3, H, D) buffer, q and k sharing
    cu_seqlens.  The kernels read q, k, v in place through row strides; no copy is made."""
    if qkv.dim() != 4 or qkv.shape[1] != 3:
        raise ValueError("expected qkv (total, 3, H, D)")
    q, k, v = qkv.unbind(1)
    return varlen_attention(q, k, v, cu_seqlens, cu_seqlens, max_seqlen, max_seqlen, block_mask, scale, return_aux,
                            mask_mod=mask_mod, out=out, window=window, prefix_lengths=prefix_lengths)


def varlen_attention_kvpacked(q, kv, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, block_mask=None,
                              scale=None, return_aux=False, *, mask_mod=None, out=None, window=0,
                              prefix_lengths=None):
    """NVTE_KV_INTERLEAVED (Transformer Engine fused_attn.h): q (total_q, H, D) and one (total_k, 2, H, D)
    buffer for k and v, read in place through row strides."""
    if kv.dim() != 4 or kv.shape[1] != 2:
        raise ValueError("expected kv (total_k, 2, H, D)")
    k, v = kv.unbind(1)
    return varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, block_mask, scale,
                            return_aux, mask_mod=mask_mod, out=out, window=window, prefix_lengths=prefix_lengths)


def varlen_attention_backward(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, out, lse, d_out,
                              block_mask=None, scale=None, *, mask_mod=None, window=0, prefix_lengths=None,
                              bias=None, need_dbias=True):
    """Gradients (dq, dk, dv, dbias) of ``varlen_attention`` for dL/dO = d_out.

    Arguments as given to the forward (q / k / v contiguous (total, H, D)), plus
    its O (``out``) and lse (H, total_q).  dbias (bias's shape and dtype, the sum
    over sequences) is returned when a bias is given and need_dbias, else None.
    """
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("expected q (total_q,H,D), k/v (total_k,H,D)")
    total_q, H, D = q.shape
    if tuple(k.shape[1:]) != (H, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be (total_k, H, D) with q's H and D")
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("varlen_attention_backward runs on CUDA tensors only")
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (lse, "lse"), (d_out, "d_out"),
                  (cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _need(t, nm, dev)
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype among float32 / float16 / bfloat16")
    for t, nm in ((out, "out"), (d_out, "d_out")):
        if tuple(t.shape) != tuple(q.shape) or t.dtype != q.dtype:
            raise ValueError(f"{nm} must have q's shape and dtype")
    if lse.dtype != torch.float32 or lse.numel() != H * total_q:
        raise ValueError("lse must be float32 (H, total_q)")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    S = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != S + 1 or S <= 0:
        raise ValueError("cu_seqlens_q / cu_seqlens_k must both have num_seqs + 1 entries")
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    kn, ki, fn, fi, mask_heads, MQ, MK, bq, bk, mm = _mask_args(block_mask, mask_mod, dev)
    pl, p_all = _prefix_args(prefix_lengths, S, dev)
    if bias is not None:
        _need(bias, "bias", dev)
        if tuple(bias.shape) != (H, int(max_seqlen_q), int(max_seqlen_k)):
            raise ValueError(f"bias must be (H, max_seqlen_q, max_seqlen_k) = {(H, int(max_seqlen_q), int(max_seqlen_k))}")
        if bias.dtype not in (torch.float32, q.dtype):
            raise TypeError("bias must be float32 or q's dtype")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dbias = torch.empty_like(bias) if (bias is not None and need_dbias) else None
    nbytes = abi.tri_attn_varlen_bwd_workspace_size(total_q, H, D, int(max_seqlen_q), int(max_seqlen_k),
                                                    dbias is not None)
    ws = torch.empty(max(nbytes // 4, 1), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        abi.tri_attn_varlen_bwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), S,
                                total_q, k.shape[0], int(max_seqlen_q), int(max_seqlen_k), H, D, s, _ptr(kn),
                                _ptr(ki), _ptr(fn), _ptr(fi), mask_heads, MQ, MK, bq, bk, mm, int(window),
                                _ptr(pl), p_all, _ptr(bias), _DT[bias.dtype] if bias is not None else abi.TA_F32,
                                _ptr(lse), _ptr(out), _ptr(d_out), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias),
                                _ptr(ws), nbytes, _stream(dev))
    return dq, dk, dv, dbias


def get_status(device=None) -> int:
    """Synchronize the current stream and return/clear the device status word (0 = OK)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return abi.tri_attn_get_status(_stream(dev))
