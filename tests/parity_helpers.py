"""Shared helpers for the GPU parity tests: run a synth case through the
library and compare with the oracle on the same stored inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances (max-abs): fp32 inputs O 1e-4 / lse 1e-5; fp16/bf16 inputs O 2e-2 / lse 5e-3.
TOL = {"f32": (1e-4, 1e-5), "f16": (2e-2, 5e-3), "bf16": (2e-2, 5e-3)}


def to_gpu(t):
    return None if t is None else t.cuda()


def run_triangle(case, return_aux=True):
    import masked_attention_tri_gb300 as ta
    q, k, v, bias = (to_gpu(x) for x in (case.q, case.k, case.v, case.bias))
    res = ta.triangle_attention(q, k, v, bias, mask=to_gpu(case.mask), scale=case.scale, return_aux=return_aux,
                                kv_lengths=to_gpu(case.kv_lengths))
    torch.cuda.synchronize()
    assert ta.get_status() == 0
    return res


def f32_round(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def compare(name, dtype, got_o, got_lse, got_max, ref_o, ref_lse, ref_max):
    """Element-wise max-abs comparison; lse/max are compared with the oracle rounded to fp32."""
    to, tl = TOL[dtype]
    go = got_o.detach().float().cpu().double().numpy().reshape(ref_o.shape)
    err_o = np.abs(go - ref_o)
    assert np.isfinite(go).all(), f"{name}: non-finite output"
    assert err_o.max() <= to, f"{name}: O max-abs {err_o.max():.3e} > {to} at {np.unravel_index(err_o.argmax(), err_o.shape)}"
    if got_lse is not None:
        gl = got_lse.detach().cpu().double().numpy().reshape(ref_lse.shape)
        gm = got_max.detach().cpu().double().numpy().reshape(ref_max.shape)
        el = np.abs(gl - f32_round(ref_lse))
        em = np.abs(gm - f32_round(ref_max))
        assert el.max() <= tl, f"{name}: lse max-abs {el.max():.3e} > {tl} at {np.unravel_index(el.argmax(), el.shape)}"
        assert em.max() <= tl, f"{name}: max max-abs {em.max():.3e} > {tl}"
    return float(err_o.max())


def check_triangle(case, rows=None):
    """Run the library on the case and compare with the oracle (all rows, or a sample)."""
    O, L, M = run_triangle(case)
    rO, rL, rM = oracle.tri_fwd(case.q, case.k, case.v, case.bias, mask=case.mask, kv_lengths=case.kv_lengths,
                                scale=case.scale, rows=rows)
    if rows is not None:
        D = case.D
        O = O.reshape(-1, D)[torch.as_tensor(rows, device=O.device)]
        L = L.reshape(-1)[torch.as_tensor(rows, device=L.device)]
        M = M.reshape(-1)[torch.as_tensor(rows, device=M.device)]
    return compare(case.name, case.dtype, O, L, M, rO, rL, rM)


def run_varlen(case, return_aux=True, window=0, prefix=None, bias=None):
    import masked_attention_tri_gb300 as ta
    bm = None
    if case.kv_num_blocks is not None:
        bm = ta.BlockMask.from_kv_blocks(to_gpu(case.kv_num_blocks), to_gpu(case.kv_indices),
                                         to_gpu(case.full_kv_num_blocks), to_gpu(case.full_kv_indices),
                                         BLOCK_SIZE=case.block, mask_mod=case.mask_mod)
    cu, cuk = case.cu_seqlens.cuda(), case.cu_seqlens_k.cuda()
    res = ta.varlen_attention(case.q.cuda(), case.k.cuda(), case.v.cuda(), cu, cuk, case.max_seqlen,
                              case.max_seqlen_k, block_mask=bm, scale=case.scale, return_aux=return_aux,
                              mask_mod=case.mask_mod if bm is None else None, window=window,
                              prefix_lengths=prefix if not isinstance(prefix, list) else
                              torch.tensor(prefix, dtype=torch.int32, device="cuda"),
                              bias=None if bias is None else bias.cuda())
    torch.cuda.synchronize()
    assert ta.get_status() == 0
    return res


def check_varlen(case, window=0, prefix=None, bias=None):
    O, L, M = run_varlen(case, window=window, prefix=prefix, bias=bias)
    rO, rL, rM = oracle.varlen_fwd(case.q, case.k, case.v, case.cu_seqlens, case.cu_seqlens_k, case.scale,
                                   case.kv_num_blocks, case.kv_indices, case.full_kv_num_blocks,
                                   case.full_kv_indices, block=case.block, mask_mod=case.mask_mod,
                                   window=window, prefix_lengths=prefix, bias=bias)
    return compare(case.name, case.dtype, O, L, M, rO, rL, rM)
