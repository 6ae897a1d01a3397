"""GPU parity of the backward (tri_attn_bwd) with the fp64 backward oracle.

The oracle (oracle/backward.py) is the chain rule through the triangle_attention
page's formula, pinned on the CPU by finite differences, torch autograd and
closed forms.  The library recomputes P from the forward's own lse; the per-key-tile
gradients run on tensor cores (16-bit inputs, D up to 128) or in fp32 on CUDA cores; dQ and
dBias are summed in fp32.

Tolerance, per gradient g against the oracle r (element-wise):
    |g - r| <= atol * max|r| + rtol * |r|
with (atol, rtol) = (1e-4, 1e-3) for fp32 inputs (fp32 arithmetic, summation
order varies) and (1e-2, 1e-2) for fp16 / bf16 inputs (one rounding of each
output to the 16-bit type, 2^-9 relative for bf16, on top of fp32 arithmetic).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.backward as obwd
import synth
from parity_helpers import to_gpu

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-4, 1e-3), "f16": (1e-2, 1e-2), "bf16": (1e-2, 1e-2)}


def _close(name, dtype, got, ref):
    atol, rtol = TOL[dtype]
    g = got.detach().float().cpu().double().numpy().reshape(ref.shape)
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    scale = max(float(np.abs(ref).max()), 1e-30)
    err = np.abs(g - ref)
    bound = atol * scale + rtol * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (f"{name}: |g - r| = {err[worst]:.3e} > {bound[worst]:.3e} at {worst} "
                                  f"(g {g[worst]:.6e}, r {ref[worst]:.6e}, max|r| {scale:.3e})")


def _run(case, seed, need_dbias=True, use_autograd=False, with_out=False):
    import masked_attention_tri_gb300 as ta
    d_out = synth.grad_out(case, seed)
    q, k, v, bias = (to_gpu(x) for x in (case.q, case.k, case.v, case.bias))
    mask, kl = to_gpu(case.mask), to_gpu(case.kv_lengths)
    if use_autograd:
        q, k, v, bias = (t.clone().requires_grad_(True) for t in (q, k, v, bias))
        o = ta.triangle_attention_autograd(q, k, v, bias, mask, case.scale, kv_lengths=kl)
        o.backward(d_out.cuda())
        torch.cuda.synchronize()
        grads = (q.grad, k.grad, v.grad, bias.grad)
    else:
        o, lse, _ = ta.triangle_attention(q, k, v, bias, mask, case.scale, True, kv_lengths=kl)
        grads = ta.triangle_attention_backward(q, k, v, bias, lse, d_out.cuda(), mask, case.scale, kv_lengths=kl,
                                               need_dbias=need_dbias, out=o if with_out else None)
        torch.cuda.synchronize()
    assert ta.get_status() == 0
    ref = obwd.tri_bwd(case.q, case.k, case.v, case.bias, d_out, mask=case.mask, kv_lengths=case.kv_lengths,
                       scale=case.scale)
    return grads, ref


def _check(case, seed, **kw):
    grads, ref = _run(case, seed, **kw)
    for nm, g, r in zip(("dq", "dk", "dv", "dbias"), grads, ref):
        if g is None:
            continue
        assert g.dtype == (case.bias.dtype if nm == "dbias" else case.q.dtype), nm
        _close(f"{case.name}:{nm}", case.dtype, g, r)


# dtypes x bias dtypes x masks; ragged Q and K (not multiples of the 32-row tiles), N > 1 for
# the sum of dBias over n, kv_lengths extremes (0: every key masked, K, beyond K).  16-bit
# inputs with D in {16, 32, 64}, or a multiple of 16 in (64, 128], take the
# tensor-core gradients, the others the CUDA-core kernel; with_out: sum_k P dP from the
# forward's O instead of the exact pass.
@pytest.mark.parametrize("with_out", [False, True])
@pytest.mark.parametrize("dtype,bias_dtype,mask,D", [
    ("bf16", "bf16", "kvlen", 64), ("bf16", "f32", "dense", 32), ("f16", "f32", "none", 128),
    ("f16", "f16", "kvlen", 16), ("f32", "f32", "kvlen", 40), ("f32", "f32", "dense", 8),
    ("bf16", "bf16", "kvlen", 128), ("f16", "f16", "dense", 96), ("bf16", "bf16", "none", 80),
])
def test_backward_matches_oracle(dtype, bias_dtype, mask, D, with_out):
    K = 70 if dtype == "f32" else 72  # 16-bit inputs need K % 8 == 0 (the forward's rule)
    c = synth.make_triangle(f"bwd_{dtype}_{bias_dtype}_{mask}_{D}", 2, 3, 2, 45, K, D, dtype, bias_dtype,
                            seed=700 + D, mask=mask, kv_range=(0, K))
    if mask == "kvlen":
        c.kv_lengths.view(-1)[:3] = torch.tensor([0, K, 1000], dtype=torch.int32)
    if mask == "dense":
        c.mask[0, 1] = 0  # a row block with every key masked
    _check(c, 710 + D, with_out=with_out)


@pytest.mark.parametrize("D", [136, 256])
def test_backward_wide_head_dims(D):
    c = synth.make_triangle(f"bwd_wide_{D}", 1, 2, 2, 33, 40, D, "bf16", "f32", seed=720 + D, mask="kvlen",
                            kv_range=(1, 40))
    _check(c, 730 + D)


@pytest.mark.parametrize("with_out", [False, True])
def test_backward_without_dbias_and_large_logits(with_out):
    c = synth.make_triangle("bwd_large", 1, 2, 2, 64, 96, 64, "bf16", "bf16", seed=740, bias_std=8.0, scale=0.5,
                            mask="kvlen", kv_range=(10, 96))
    _check(c, 741, need_dbias=False, with_out=with_out)


@pytest.mark.parametrize("D,bias_dtype", [(64, "bf16"), (128, "bf16"), (128, "f32")])
def test_backward_several_tiles(D, bias_dtype):
    """Several 128-key and 128-row tiles per slab (ragged), tensor-core gradients (D = 128: the
    tiles' two column boxes, one S^T / dP^T buffer for both query halves; with an fp32 bias its
    two halves take turns in one shared-memory slot), both delta forms."""
    c = synth.make_triangle(f"bwd_tiles_{D}_{bias_dtype}", 1, 2, 2, 300, 264, D, "bf16", bias_dtype, seed=745 + D,
                            mask="kvlen", kv_range=(100, 264))
    _check(c, 746 + D)
    _check(c, 747 + D, with_out=True)


@pytest.mark.parametrize("dtype,D,bias_dtype", [("bf16", 32, "f32"), ("f16", 64, "f32"), ("bf16", 128, "bf16"),
                                                ("f16", 96, "f32")])
def test_backward_padded_key_tiles(dtype, D, bias_dtype):
    """kv_lengths that leave whole 128-key tiles past the valid prefix (their dK / dV are zero and
    they add nothing to dQ or dBias), next to 0 (every key weighted 1 / K), 1, tile edges, K and
    beyond K, and a negative value."""
    K = 264
    lens = [0, 1, 127, 128, 129, 256, 264, 300, -3]
    c = synth.make_triangle(f"bwd_pad_{dtype}_{D}", 1, len(lens), 2, 140, K, D, dtype, bias_dtype, seed=760 + D,
                            mask="kvlen", kv_range=(0, K))
    c.kv_lengths.view(-1)[:] = torch.tensor(lens, dtype=torch.int32)
    _check(c, 761 + D)
    _check(c, 762 + D, with_out=True)


@pytest.mark.parametrize("workload", ["bf16_long", "bf16_long_d128"])
def test_backward_full_size_sampled_slabs(workload):
    """The benchmark's backward launch at full size (B=1, N=768, H=4, Q=K=768, D = 64 or 128,
    the forward's O given, dBias requested): dQ, dK and dV of sampled (b, n) slabs against the
    oracle run on those slabs alone (each slab's dQ / dK / dV depends on that slab only; dBias,
    a sum over all 768 slabs, is checked by the smaller cases).  The samples take kv_length 0
    (every key masked), 768 (every key valid) and values in between."""
    import masked_attention_tri_gb300 as ta
    c = getattr(synth, workload)()
    d_out = synth.grad_out(c, 790 + c.D)
    q, k, v, bias, kl = (to_gpu(x) for x in (c.q, c.k, c.v, c.bias, c.kv_lengths))
    o, lse, _ = ta.triangle_attention(q, k, v, bias, None, c.scale, True, kv_lengths=kl)
    dq, dk, dv, db = ta.triangle_attention_backward(q, k, v, bias, lse, d_out.cuda(), None, c.scale, kv_lengths=kl,
                                                    need_dbias=True, out=o)
    torch.cuda.synchronize()
    assert ta.get_status() == 0
    assert db is not None and torch.isfinite(db.float()).all()
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    del q, k, v, o, lse, db
    for n in (0, 1, 2, 385, 767):
        sl = slice(n, n + 1)
        rq, rk, rv, _ = obwd.tri_bwd(c.q[:, sl], c.k[:, sl], c.v[:, sl], c.bias, d_out[:, sl],
                                     kv_lengths=c.kv_lengths[:, sl], scale=c.scale)
        _close(f"{workload}:dq[n={n}]", c.dtype, dq[:, sl], rq)
        _close(f"{workload}:dk[n={n}]", c.dtype, dk[:, sl], rk)
        _close(f"{workload}:dv[n={n}]", c.dtype, dv[:, sl], rv)


def test_autograd_wrapper():
    """torch autograd through triangle_attention_autograd gives the same gradients (it passes the
    forward's O, so the per-row sums come from dO . O)."""
    c = synth.make_triangle("bwd_autograd", 1, 2, 3, 50, 64, 32, "bf16", "f32", seed=750, mask="dense")
    _check(c, 751, use_autograd=True)


def test_backward_page_example_shape():
    """The page's Example shapes at a smaller sequence length: fp16, bias and mask from kv_lengths."""
    c = synth.make_triangle("bwd_page", 1, 4, 2, 64, 64, 32, "f16", "f16", seed=760, mask="kvlen", kv_range=(48, 64))
    _check(c, 761)


# ---------------------------------------------------------------------------
# Packed sequences (tri_attn_varlen_bwd), against oracle.backward.varlen_bwd
# ---------------------------------------------------------------------------

def _check_varlen(case, seed, window=0, prefix=None, bias=None):
    import masked_attention_tri_gb300 as ta
    bm = None
    if case.kv_num_blocks is not None:
        bm = ta.BlockMask.from_kv_blocks(to_gpu(case.kv_num_blocks), to_gpu(case.kv_indices),
                                         to_gpu(case.full_kv_num_blocks), to_gpu(case.full_kv_indices),
                                         BLOCK_SIZE=case.block, mask_mod=case.mask_mod)
    mm = case.mask_mod if bm is None else None
    pl = None if prefix is None else torch.tensor(prefix, dtype=torch.int32, device="cuda")
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    cu, cuk = case.cu_seqlens.cuda(), case.cu_seqlens_k.cuda()
    bg = None if bias is None else bias.cuda()
    o, lse, _ = ta.varlen_attention(q, k, v, cu, cuk, case.max_seqlen, case.max_seqlen_k, block_mask=bm,
                                    scale=case.scale, return_aux=True, mask_mod=mm, window=window,
                                    prefix_lengths=pl, bias=bg)
    g = torch.Generator().manual_seed(seed)
    d_out = torch.randn(tuple(case.q.shape), generator=g).to(case.q.dtype)
    grads = ta.varlen_attention_backward(q, k, v, cu, cuk, case.max_seqlen, case.max_seqlen_k, o, lse,
                                         d_out.cuda(), block_mask=bm, scale=case.scale, mask_mod=mm,
                                         window=window, prefix_lengths=pl, bias=bg)
    torch.cuda.synchronize()
    assert ta.get_status() == 0
    ref = obwd.varlen_bwd(case.q, case.k, case.v, case.cu_seqlens, case.cu_seqlens_k, d_out, scale=case.scale,
                          kv_num_blocks=case.kv_num_blocks, kv_indices=case.kv_indices,
                          full_kv_num_blocks=case.full_kv_num_blocks, full_kv_indices=case.full_kv_indices,
                          block=case.block, mask_mod=case.mask_mod, window=window,
                          prefix_lengths=prefix, bias=bias)
    for nm, gr, r in zip(("dq", "dk", "dv", "dbias"), grads, ref):
        if r is None:
            assert gr is None
            continue
        _close(f"{case.name}:{nm}", case.dtype, gr, r)


@pytest.mark.parametrize("dtype,D,lists", [("bf16", 64, "causal"), ("f16", 32, "none"), ("f32", 16, "causal")])
def test_varlen_backward_matches_oracle(dtype, D, lists):
    c = synth.make_varlen(f"vbwd_{dtype}_{D}_{lists}", 4, 0, 0, 2, D, dtype, seed=770 + D, lengths=[300, 129, 64, 1],
                          block_lists=lists, mask_mod="causal")
    _check_varlen(c, 771 + D)


def test_varlen_backward_random_lists_and_unlisted_blocks():
    """Random full / partial lists, a q block with no listed block (its rows all masked), D = 128."""
    c = synth.make_varlen("vbwd_rand", 2, 0, 0, 2, 128, "bf16", seed=785, lengths=[400, 260])
    g = np.random.default_rng(3)
    S, MQ = 2, 4
    kn = torch.zeros(S, 1, MQ, dtype=torch.int32)
    ki = torch.full((S, 1, MQ, MQ), 77, dtype=torch.int32)
    fn = torch.zeros(S, 1, MQ, dtype=torch.int32)
    fi = torch.full((S, 1, MQ, MQ), 77, dtype=torch.int32)
    for s_, L in enumerate([400, 260]):
        nb = (L + 127) // 128
        for qb in range(nb):
            if qb == 1:
                continue
            perm = g.permutation(nb).tolist()
            nf = int(g.integers(0, nb + 1))
            fn[s_, 0, qb] = nf
            fi[s_, 0, qb, :nf] = torch.tensor(perm[:nf], dtype=torch.int32)
            kn[s_, 0, qb] = nb - nf
            ki[s_, 0, qb, :nb - nf] = torch.tensor(perm[nf:], dtype=torch.int32)
    c.kv_num_blocks, c.kv_indices, c.full_kv_num_blocks, c.full_kv_indices = kn, ki, fn, fi
    _check_varlen(c, 786)


def test_varlen_backward_lq_ne_lk_window_and_bias():
    c = synth.make_varlen("vbwd_lqlk", 3, 0, 0, 2, 64, "bf16", seed=780, lengths=[200, 70, 129],
                          lengths_k=[90, 300, 129], block_lists="none", mask_mod="sliding_window")
    c.max_seqlen, c.max_seqlen_k = 208, 304
    g = torch.Generator().manual_seed(781)
    bias = torch.randn(2, 208, 304, generator=g).to(torch.bfloat16)
    _check_varlen(c, 782, window=40, bias=bias)


def test_varlen_backward_prefix_lm_fp32_bias():
    c = synth.make_varlen("vbwd_prefix", 3, 0, 0, 1, 32, "f16", seed=790, lengths=[150, 40, 260],
                          block_lists="none", mask_mod="prefix_lm")
    c.max_seqlen = c.max_seqlen_k = 264
    g = torch.Generator().manual_seed(791)
    bias = torch.randn(1, 264, 264, generator=g)
    _check_varlen(c, 792, prefix=[20, 0, 300], bias=bias)


# Packed sequences run on the tensor cores (16-bit, D <= 128; a bias too, 16-bit at D > 64): one CTA per
# (sequence, head, 128-key block) over the q blocks whose lists hold the key block.

def test_varlen_backward_lq_ne_lk_window_no_bias():
    """Lq != Lk (top-left aligned), a sliding window on every block (no lists), keys past the
    queries' reach and sequences shorter than one block."""
    c = synth.make_varlen("vbwd_lqlk_nb", 3, 0, 0, 2, 64, "bf16", seed=783, lengths=[200, 70, 129],
                          lengths_k=[90, 300, 129], block_lists="none", mask_mod="sliding_window")
    c.max_seqlen, c.max_seqlen_k = 208, 304
    _check_varlen(c, 784, window=40)


def test_varlen_backward_prefix_lm_no_bias():
    """Prefix-LM on every block, per-sequence prefixes 20, 0 and beyond the sequence."""
    c = synth.make_varlen("vbwd_prefix_nb", 3, 0, 0, 2, 32, "f16", seed=793, lengths=[150, 40, 260],
                          block_lists="none", mask_mod="prefix_lm")
    c.max_seqlen = c.max_seqlen_k = 264
    _check_varlen(c, 794, prefix=[20, 0, 300])


@pytest.mark.parametrize("D", [64, 128])
def test_varlen_backward_many_blocks(D):
    """Causal lists over several q and key blocks per sequence (full blocks below the diagonal,
    partial ones on it), three heads, a one-token sequence."""
    c = synth.make_varlen(f"vbwd_many_{D}", 3, 0, 0, 3, D, "bf16", seed=795 + D, lengths=[700, 300, 1],
                          block_lists="causal", mask_mod="causal")
    _check_varlen(c, 796 + D)


def test_varlen_backward_full_size_sampled_sequences():
    """The bf16_varlen packed sequences at full size (8 causal sequences of 256-2048 tokens, H=8,
    D=128), as the benchmark runs them; dQ, dK and dV of the shortest and the longest sequence
    against the oracle run on that sequence alone (without a bias a sequence's gradients depend
    on its own rows only)."""
    import masked_attention_tri_gb300 as ta
    c = synth.bf16_varlen()
    bm = ta.BlockMask.from_kv_blocks(to_gpu(c.kv_num_blocks), to_gpu(c.kv_indices), to_gpu(c.full_kv_num_blocks),
                                     to_gpu(c.full_kv_indices), BLOCK_SIZE=c.block, mask_mod=c.mask_mod)
    q, k, v, cu = c.q.cuda(), c.k.cuda(), c.v.cuda(), c.cu_seqlens.cuda()
    o, lse, _ = ta.varlen_attention(q, k, v, cu, cu, c.max_seqlen, c.max_seqlen, block_mask=bm, scale=c.scale,
                                    return_aux=True)
    g = torch.Generator().manual_seed(799)
    d_out = torch.randn(tuple(c.q.shape), generator=g).to(c.q.dtype)
    dq, dk, dv, db = ta.varlen_attention_backward(q, k, v, cu, cu, c.max_seqlen, c.max_seqlen, o, lse, d_out.cuda(),
                                                  block_mask=bm, scale=c.scale)
    torch.cuda.synchronize()
    assert ta.get_status() == 0 and db is None
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    L = c.lengths.tolist()
    for s in sorted({L.index(min(L)), L.index(max(L))}):
        a, b = int(c.cu_seqlens[s]), int(c.cu_seqlens[s + 1])
        cu1 = torch.tensor([0, b - a], dtype=torch.int32)
        sl = slice(s, s + 1)
        ref = obwd.varlen_bwd(c.q[a:b], c.k[a:b], c.v[a:b], cu1, cu1, d_out[a:b], scale=c.scale,
                              kv_num_blocks=c.kv_num_blocks[sl], kv_indices=c.kv_indices[sl],
                              full_kv_num_blocks=c.full_kv_num_blocks[sl], full_kv_indices=c.full_kv_indices[sl],
                              block=c.block, mask_mod=c.mask_mod)
        for nm, gr, r in zip(("dq", "dk", "dv"), (dq[a:b], dk[a:b], dv[a:b]), ref[:3]):
            _close(f"bf16_varlen[seq {s}, {b - a} tokens]:{nm}", c.dtype, gr, r)


@pytest.mark.parametrize("bias_dtype", [torch.bfloat16, torch.float32])
def test_varlen_backward_wide_bias_and_dbias(bias_dtype):
    """D = 128 with a post-scale bias (H, max_seqlen_q, max_seqlen_k), bf16 or fp32 (its halves
    sharing one slot), and its gradient summed over the sequences, causal lists over several
    blocks."""
    c = synth.make_varlen("vbwd_wide_bias", 2, 0, 0, 2, 128, "bf16", seed=801, lengths=[300, 129],
                          block_lists="causal", mask_mod="causal")
    c.max_seqlen = c.max_seqlen_k = 304
    g = torch.Generator().manual_seed(802)
    bias = torch.randn(2, 304, 304, generator=g).to(bias_dtype)
    _check_varlen(c, 803, bias=bias)


def test_varlen_backward_per_head_lists():
    """Per-head lists (mask_heads = H): head 0 causal lists, head 1 only the diagonal blocks
    (partial) and, for sequence 0, no block at all for q block 1 (its rows have no valid key and
    weigh every key 1 / Lk); every key block derives its own q-block list per head."""
    c = synth.make_varlen("vbwd_heads", 2, 0, 0, 2, 64, "bf16", seed=805, lengths=[384, 200])
    kn, ki, fn, fi = synth.causal_block_lists([384, 200], mask_heads=2)
    fn[:, 1] = 0
    kn[0, 1, 1] = 0
    c.kv_num_blocks, c.kv_indices, c.full_kv_num_blocks, c.full_kv_indices = kn, ki, fn, fi
    _check_varlen(c, 806)
