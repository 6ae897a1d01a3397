"""Pins of the backward oracle (``oracle.backward.tri_bwd``), CPU only.

The gradients are checked against things other than their own formula:
central finite differences of the independent pure-Python forward
(``oracle.brute``, fp64), torch autograd through a separate torch restatement
of the cuEquivariance triangle_attention formula, closed forms (one valid
key, an all-masked row) and the shift invariance of the softmax (each row of
dx sums to zero).
"""
import numpy as np
import pytest
import torch

from oracle import brute
from oracle.backward import tri_bwd


def _case(seed, B=1, N=2, H=2, Q=3, K=4, D=3, mask_kind="none"):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, N, H, Q, D, generator=g)
    k = torch.randn(B, N, H, K, D, generator=g)
    v = torch.randn(B, N, H, K, D, generator=g)
    bias = torch.randn(B, 1, H, Q, K, generator=g)
    d_out = torch.randn(B, N, H, Q, D, generator=g, dtype=torch.float64)
    mask = kvl = None
    if mask_kind == "kvlen":
        kvl = torch.tensor([[2, 0][:N]] * B, dtype=torch.int32)  # a partial prefix and an all-masked row
    elif mask_kind == "dense":
        mask = (torch.rand(B, N, 1, 1, K, generator=g) < 0.6).to(torch.uint8)
        mask[0, 0, 0, 0, 0] = 1
    return q, k, v, bias, d_out, mask, kvl


def _loss_brute(q, k, v, bias, d_out, mask, kvl, scale):
    O, _, _ = brute.tri_fwd(q.tolist(), k.tolist(), v.tolist(), bias.tolist(),
                            mask=None if mask is None else mask.tolist(),
                            kv_lengths=None if kvl is None else kvl.tolist(), scale=scale)
    return float((torch.tensor(O, dtype=torch.float64) * d_out).sum())


@pytest.mark.parametrize("mask_kind", ["none", "kvlen", "dense"])
def test_gradients_match_finite_differences(mask_kind):
    q, k, v, bias, d_out, mask, kvl = _case(11, mask_kind=mask_kind)
    scale = 0.7
    grads = tri_bwd(q, k, v, bias, d_out, mask=mask, kv_lengths=kvl, scale=scale)
    eps = 1e-6
    for t, g in zip((q, k, v, bias), grads):
        base = t.double()
        flat = base.reshape(-1)
        fd = np.zeros(flat.numel())
        for i in range(flat.numel()):
            plus, minus = flat.clone(), flat.clone()
            plus[i] += eps
            minus[i] -= eps
            args = [q.double(), k.double(), v.double(), bias.double()]
            idx = [id(x) for x in (q, k, v, bias)].index(id(t))
            args[idx] = plus.reshape(base.shape)
            lp = _loss_brute(*args, d_out, mask, kvl, scale)
            args[idx] = minus.reshape(base.shape)
            lm = _loss_brute(*args, d_out, mask, kvl, scale)
            fd[i] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g.reshape(-1), fd, atol=2e-6, rtol=1e-5)


def _torch_grads(q, k, v, bias, d_out, valid, scale):
    s = float(np.float32(scale))
    qd, kd, vd, bd = (t.double().clone().requires_grad_(True) for t in (q, k, v, bias))
    x = s * torch.einsum("bnhqd,bnhkd->bnhqk", qd, kd) + bd  # bias broadcast over n
    x = x.masked_fill(~valid[:, :, None, None, :], -1e9)
    O = torch.einsum("bnhqk,bnhkd->bnhqd", torch.softmax(x, dim=-1), vd)
    (O * d_out).sum().backward()
    return [t.grad.numpy() for t in (qd, kd, vd, bd)]


@pytest.mark.parametrize("mask_kind", ["none", "kvlen", "dense"])
def test_gradients_match_torch_autograd(mask_kind):
    q, k, v, bias, d_out, mask, kvl = _case(21, B=2, N=3, H=2, Q=5, K=6, D=8, mask_kind=mask_kind)
    if kvl is not None:
        kvl = torch.tensor([[3, 0, 6], [1, 7, 4]], dtype=torch.int32)
    B, N, K = q.shape[0], q.shape[1], k.shape[3]
    if mask is not None:
        valid = mask.reshape(B, N, K) != 0
    elif kvl is not None:
        valid = torch.arange(K)[None, None, :] < kvl.clamp(0, K)[:, :, None]
    else:
        valid = torch.ones(B, N, K, dtype=torch.bool)
    got = tri_bwd(q, k, v, bias, d_out, mask=mask, kv_lengths=kvl, scale=None)
    ref = _torch_grads(q, k, v, bias, d_out, valid, 1.0 / np.sqrt(q.shape[-1]))
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, atol=1e-10, rtol=1e-9)


def test_single_valid_key_passes_no_gradient_to_logits():
    q, k, v, bias, d_out, _, _ = _case(31)
    kvl = torch.ones(1, 2, dtype=torch.int32)
    dQ, dK, dV, dB = tri_bwd(q, k, v, bias, d_out, kv_lengths=kvl)
    assert np.abs(dQ).max() == 0 and np.abs(dK).max() == 0 and np.abs(dB).max() == 0
    # all weight on key 0: dV[key 0] = sum over queries of dO, other keys 0
    np.testing.assert_allclose(dV[:, :, :, 0], d_out.numpy().sum(axis=3), rtol=1e-14, atol=1e-14)
    assert np.abs(dV[:, :, :, 1:]).max() == 0


def test_all_masked_row_spreads_dv_uniformly():
    q, k, v, bias, d_out, _, _ = _case(41)
    kvl = torch.zeros(1, 2, dtype=torch.int32)
    dQ, dK, dV, dB = tri_bwd(q, k, v, bias, d_out, kv_lengths=kvl)
    assert np.abs(dQ).max() == 0 and np.abs(dK).max() == 0 and np.abs(dB).max() == 0
    K = k.shape[3]
    expect = d_out.numpy().sum(axis=3, keepdims=True) / K
    np.testing.assert_allclose(dV, np.broadcast_to(expect, dV.shape), rtol=1e-13, atol=1e-14)


def test_bias_gradient_rows_sum_to_zero():
    q, k, v, bias, d_out, _, _ = _case(51, B=1, N=3, H=2, Q=4, K=7, D=5)
    _, _, _, dB = tri_bwd(q, k, v, bias, d_out)
    assert np.abs(dB.sum(axis=-1)).max() < 1e-12


# ---------------------------------------------------------------------------
# Packed sequences (oracle.backward.varlen_bwd)
# ---------------------------------------------------------------------------

from oracle.backward import varlen_bwd  # noqa: E402


def test_varlen_bwd_one_sequence_is_the_triangle_backward():
    """One sequence, no lists, mask_mod none: the (B=N=1) triangle problem."""
    g = torch.Generator().manual_seed(41)
    Lq, Lk, H, D = 37, 29, 2, 8
    q, k, v = (torch.randn(L, H, D, generator=g) for L in (Lq, Lk, Lk))
    bias = torch.randn(H, Lq, Lk, generator=g)
    do = torch.randn(Lq, H, D, generator=g, dtype=torch.float64)
    r = varlen_bwd(q, k, v, torch.tensor([0, Lq]), torch.tensor([0, Lk]), do, scale=0.3, bias=bias)
    tri = lambda t: t.permute(1, 0, 2)[None, None].contiguous()
    t = tri_bwd(tri(q), tri(k), tri(v), bias[None, None].contiguous(), tri(do), scale=0.3)
    for a, b in zip(r[:3], t[:3]):
        np.testing.assert_allclose(a, b[0, 0].transpose(1, 0, 2), atol=1e-12)
    np.testing.assert_allclose(r[3], t[3][0, 0], atol=1e-12)


def _element_mask(Lq, Lk, block, part_sets, full_sets, mod, window, prefix):
    """(Lq, Lk) bool built key by key from block sets (dicts qb -> set of kb) and the
    mask_mod rule, written out directly; no lists (part_sets None) = every block partial."""
    m = torch.zeros(Lq, Lk, dtype=torch.bool)
    for qq in range(Lq):
        for kk in range(Lk):
            qb, kb = qq // block, kk // block
            if part_sets is None:
                full, part = False, True
            else:
                full = kb in full_sets.get(qb, set())
                part = (kb in part_sets.get(qb, set())) and not full
            keep = {"none": True, "causal": kk <= qq, "sliding_window": qq - window < kk <= qq,
                    "prefix_lm": kk <= qq or kk < prefix}[mod]
            m[qq, kk] = full or (part and keep)
    return m


@pytest.mark.parametrize("mod", ["none", "causal", "sliding_window", "prefix_lm"])
@pytest.mark.parametrize("lists", [False, True])
def test_varlen_bwd_matches_torch_autograd(mod, lists):
    """Several sequences (Lq != Lk, one of them all masked when lists skip its blocks), block
    size 4, a post-scale bias: fp64 autograd through a masked softmax with the element
    mask of `_element_mask`."""
    g = torch.Generator().manual_seed(51)
    lq, lk, H, D, block, window = [9, 6, 5], [7, 10, 5], 2, 4, 4, 3
    cq = torch.tensor([0, 9, 15, 20]); ck = torch.tensor([0, 7, 17, 22])
    q, k, v = torch.randn(20, H, D, generator=g), torch.randn(22, H, D, generator=g), torch.randn(22, H, D, generator=g)
    bias = torch.randn(H, 9, 10, generator=g)
    do = torch.randn(20, H, D, generator=g, dtype=torch.float64)
    prefix = [2, 0, 4]
    kn = ki = fn = fi = None
    part_sets = full_sets = None
    if lists:
        MQ, MK = 3, 3
        # per sequence (mask_heads 1): q block -> partial / full kv blocks (entries past the count unread)
        P = [{0: [0], 1: [1, 0], 2: [1]}, {0: [0, 2], 1: []}, {0: [], 1: [1]}]
        F = [{1: [0]}, {0: [1]}, {}]
        kn = torch.zeros(3, 1, MQ, dtype=torch.int32); ki = torch.full((3, 1, MQ, MK), 7, dtype=torch.int32)
        fn = torch.zeros(3, 1, MQ, dtype=torch.int32); fi = torch.full((3, 1, MQ, MK), 7, dtype=torch.int32)
        for s_ in range(3):
            for qb, kbs in P[s_].items():
                kn[s_, 0, qb] = len(kbs)
                ki[s_, 0, qb, :len(kbs)] = torch.tensor(kbs, dtype=torch.int32) if kbs else ki[s_, 0, qb, :0]
            for qb, kbs in F[s_].items():
                fn[s_, 0, qb] = len(kbs)
                fi[s_, 0, qb, :len(kbs)] = torch.tensor(kbs, dtype=torch.int32)
        part_sets = [{qb: set(v_) for qb, v_ in P[s_].items()} for s_ in range(3)]
        full_sets = [{qb: set(v_) for qb, v_ in F[s_].items()} for s_ in range(3)]
    scale = 0.375  # exact in fp32 (the oracle takes the scale as the kernels' float)
    got = varlen_bwd(q, k, v, cq, ck, do, scale=scale, kv_num_blocks=kn, kv_indices=ki, full_kv_num_blocks=fn,
                     full_kv_indices=fi, block=block, mask_mod=mod, window=window,
                     prefix_lengths=torch.tensor(prefix), bias=bias)
    qd, kd, vd, bd = (t.double().clone().requires_grad_(True) for t in (q, k, v, bias))
    loss = 0.0
    for s_ in range(3):
        q0, k0, Lq, Lk = int(cq[s_]), int(ck[s_]), lq[s_], lk[s_]
        m = _element_mask(Lq, Lk, block, None if part_sets is None else part_sets[s_],
                          None if full_sets is None else full_sets[s_], mod, window, prefix[s_])
        for h in range(H):
            x = scale * (qd[q0:q0 + Lq, h] @ kd[k0:k0 + Lk, h].T) + bd[h, :Lq, :Lk]
            x = torch.where(m, x, torch.full_like(x, -1e9))
            o = torch.softmax(x, dim=-1) @ vd[k0:k0 + Lk, h]
            loss = loss + (o * do[q0:q0 + Lq, h]).sum()
    loss.backward()
    for a, t in zip(got, (qd, kd, vd, bd)):
        np.testing.assert_allclose(a, t.grad.numpy(), atol=1e-10, rtol=1e-9)


def test_varlen_bwd_per_head_lists_match_torch_autograd():
    """Per-head lists (mask_heads = H = 2, the lists' second axis): head 0 and head 1 list different
    blocks (head 1 leaves one q block with no block at all, so its rows have no valid key), causal
    mask_mod; fp64 autograd with each head's element mask from `_element_mask`."""
    g = torch.Generator().manual_seed(61)
    lq, H, D, block = [9, 7], 2, 4, 4
    cu = torch.tensor([0, 9, 16])
    q, k, v = (torch.randn(16, H, D, generator=g) for _ in range(3))
    do = torch.randn(16, H, D, generator=g, dtype=torch.float64)
    MQ = MK = 3
    # [sequence][head]: q block -> partial / full kv blocks
    P = [[{0: [0], 1: [1], 2: [2]}, {0: [0], 1: [], 2: [0, 2]}], [{0: [0], 1: [1]}, {0: [0], 1: [0, 1]}]]
    F = [[{1: [0], 2: [0, 1]}, {2: [1]}], [{1: [0]}, {}]]
    kn = torch.zeros(2, H, MQ, dtype=torch.int32); ki = torch.full((2, H, MQ, MK), 7, dtype=torch.int32)
    fn = torch.zeros(2, H, MQ, dtype=torch.int32); fi = torch.full((2, H, MQ, MK), 7, dtype=torch.int32)
    for s_ in range(2):
        for h in range(H):
            for qb, kbs in P[s_][h].items():
                kn[s_, h, qb] = len(kbs)
                if kbs:
                    ki[s_, h, qb, :len(kbs)] = torch.tensor(kbs, dtype=torch.int32)
            for qb, kbs in F[s_][h].items():
                fn[s_, h, qb] = len(kbs)
                fi[s_, h, qb, :len(kbs)] = torch.tensor(kbs, dtype=torch.int32)
    scale = 0.375
    got = varlen_bwd(q, k, v, cu, cu, do, scale=scale, kv_num_blocks=kn, kv_indices=ki, full_kv_num_blocks=fn,
                     full_kv_indices=fi, block=block, mask_mod="causal")
    qd, kd, vd = (t.double().clone().requires_grad_(True) for t in (q, k, v))
    loss = 0.0
    for s_ in range(2):
        c0, L = int(cu[s_]), lq[s_]
        for h in range(H):
            m = _element_mask(L, L, block, {qb: set(x) for qb, x in P[s_][h].items()},
                              {qb: set(x) for qb, x in F[s_][h].items()}, "causal", 0, 0)
            x = scale * (qd[c0:c0 + L, h] @ kd[c0:c0 + L, h].T)
            x = torch.where(m, x, torch.full_like(x, -1e9))
            o = torch.softmax(x, dim=-1) @ vd[c0:c0 + L, h]
            loss = loss + (o * do[c0:c0 + L, h]).sum()
    loss.backward()
    assert got[3] is None
    for a, t in zip(got[:3], (qd, kd, vd)):
        np.testing.assert_allclose(a, t.grad.numpy(), atol=1e-10, rtol=1e-9)
