"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the fp64 oracle against brute force, a closed form, an
invariant of the cuEquivariance triangle_attention formula, a library
routine (torch SDPA in fp64), or the triangle_attention page's worked
example.  Together they are chosen so a dropped term, a wrong sign, a
transposed operand, additive instead of replacing masking, or a wrong mask
index fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _f64(t):
    return t.to(torch.float64)


def _nested(t):
    return _f64(t).tolist()


# ---------------------------------------------------------------------------
# Widening of stored inputs
# ---------------------------------------------------------------------------

def test_widen_fp16_all_patterns():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    h = bits.view(torch.float16)
    got = oracle.widen(h)
    ref = h.numpy().astype(np.float64)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_widen_bf16_all_patterns():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    b = bits.view(torch.bfloat16)
    got = oracle.widen(b)
    ref = b.to(torch.float64).numpy()
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


# ---------------------------------------------------------------------------
# Brute force on tiny inputs (the two restatements are independent)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,bias_dtype", [("f32", "f32"), ("f16", "f32"), ("bf16", "bf16"), ("f16", "f16")])
@pytest.mark.parametrize("mask", ["none", "kvlen", "dense"])
def test_oracle_matches_brute_force(dtype, bias_dtype, mask):
    c = synth.make_triangle("t", 2, 3, 2, 5, 7, 8, dtype, bias_dtype, seed=7, bias_std=1.5,
                            mask=mask, kv_range=(0, 7) if mask == "kvlen" else None)
    if mask == "kvlen":
        c.kv_lengths.view(-1)[:4] = torch.tensor([0, 9, -3, 3], dtype=torch.int32)
    O, L, M = oracle.tri_fwd(c.q, c.k, c.v, c.bias, mask=c.mask, kv_lengths=c.kv_lengths, scale=c.scale)
    bO, bL, bM = brute.tri_fwd(_nested(c.q), _nested(c.k), _nested(c.v), _nested(c.bias),
                               mask=None if c.mask is None else c.mask.tolist(),
                               kv_lengths=None if c.kv_lengths is None else c.kv_lengths.tolist(),
                               scale=c.scale)
    np.testing.assert_allclose(O, np.array(bO), rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, np.array(bL), rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(M, np.array(bM), rtol=1e-13, atol=1e-12)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def test_two_key_hand_case():
    """One query, two keys, D=1: q=1, k=(1,2), v=(1,3), bias 0, s=1.

    Logits (1, 2): softmax weights 1/(1+e), e/(1+e); O = (1+3e)/(1+e);
    lse = log(e + e^2); max = 2.
    """
    q = torch.ones(1, 1, 1, 1, 1)
    k = torch.tensor([1.0, 2.0]).view(1, 1, 1, 2, 1)
    v = torch.tensor([1.0, 3.0]).view(1, 1, 1, 2, 1)
    bias = torch.zeros(1, 1, 1, 1, 2)
    O, L, M = oracle.tri_fwd(q, k, v, bias, scale=1.0)
    e = math.e
    assert O.item() == pytest.approx((1 + 3 * e) / (1 + e), abs=1e-14)
    assert L.item() == pytest.approx(math.log(e + e * e), abs=1e-14)
    assert M.item() == 2.0


def test_constant_v_gives_constant():
    c = synth.make_triangle("t", 1, 3, 2, 9, 11, 16, "f32", "f32", seed=11, bias_std=3.0,
                            mask="kvlen", kv_range=(0, 11))
    v = torch.full_like(c.v, 0.75)
    O, _, _ = oracle.tri_fwd(c.q, c.k, v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale)
    np.testing.assert_allclose(O, 0.75, rtol=0, atol=1e-14)


def test_zero_query_zero_bias_is_mean_of_valid_values():
    c = synth.make_triangle("t", 1, 4, 2, 3, 10, 8, "f32", "f32", seed=12, mask="kvlen", kv_range=(1, 10))
    q = torch.zeros_like(c.q)
    bias = torch.zeros_like(c.bias)
    O, L, M = oracle.tri_fwd(q, c.k, c.v, bias, kv_lengths=c.kv_lengths, scale=c.scale)
    for n in range(4):
        Lv = int(c.kv_lengths[0, n])
        mean = _f64(c.v[0, n, :, :Lv]).mean(dim=1).numpy()  # (H, D)
        for h in range(2):
            np.testing.assert_allclose(O[0, n, h], np.broadcast_to(mean[h], (3, 8)), atol=1e-14)
        np.testing.assert_allclose(L[0, n], math.log(Lv), atol=1e-14)
        np.testing.assert_allclose(M[0, n], 0.0, atol=0)


def test_single_valid_key():
    c = synth.make_triangle("t", 1, 2, 2, 4, 6, 8, "f32", "f32", seed=13, mask="kvlen", kv_const=1)
    O, L, M = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale)
    s = float(np.float32(c.scale))
    for n in range(2):
        for h in range(2):
            for i in range(4):
                x0 = s * float((_f64(c.q[0, n, h, i]) * _f64(c.k[0, n, h, 0])).sum()) + float(c.bias[0, 0, h, i, 0])
                np.testing.assert_allclose(O[0, n, h, i], _f64(c.v[0, n, h, 0]).numpy(), atol=1e-14)
                assert L[0, n, h, i] == pytest.approx(x0, abs=1e-12)
                assert M[0, n, h, i] == pytest.approx(x0, abs=1e-12)


@pytest.mark.parametrize("how", ["kvlen0", "kvlen_negative", "dense_zero"])
def test_all_masked_row_is_mean_of_all_values(how):
    """Every logit is replaced by -1e9: uniform softmax over all K keys, whatever the bias."""
    K = 12
    c = synth.make_triangle("t", 1, 2, 2, 5, K, 8, "f32", "f32", seed=14, bias_std=50.0)
    bias = c.bias.clone()
    bias[..., ::2] = 1e6  # a masked key's bias must not matter
    kw = {}
    if how == "kvlen0":
        kw["kv_lengths"] = torch.zeros(1, 2, dtype=torch.int32)
    elif how == "kvlen_negative":
        kw["kv_lengths"] = torch.full((1, 2), -5, dtype=torch.int32)
    else:
        kw["mask"] = torch.zeros(1, 2, 1, 1, K, dtype=torch.uint8)
    O, L, M = oracle.tri_fwd(c.q, c.k, c.v, bias, scale=c.scale, **kw)
    mean = _f64(c.v).mean(dim=3, keepdim=True).expand(-1, -1, -1, 5, -1).numpy()
    np.testing.assert_allclose(O, mean, atol=1e-14)
    np.testing.assert_allclose(M, -1e9, atol=0)
    np.testing.assert_allclose(L, -1e9 + math.log(K), atol=1e-6)


def test_kvlen_above_k_is_clamped():
    c = synth.make_triangle("t", 1, 2, 1, 3, 8, 8, "f32", "f32", seed=15)
    full = oracle.tri_fwd(c.q, c.k, c.v, c.bias, scale=c.scale)
    big = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=torch.full((1, 2), 1000, dtype=torch.int32),
                         scale=c.scale)
    for a, b in zip(full, big):
        np.testing.assert_array_equal(a, b)


def test_bias_shift_moves_lse_and_max_only():
    c = synth.make_triangle("t", 1, 3, 2, 6, 9, 8, "f32", "f32", seed=16, mask="kvlen", kv_range=(1, 9))
    bias = torch.round(c.bias * 64) / 64  # on a coarse grid, so that adding 2.5 is exact in fp32
    a = oracle.tri_fwd(c.q, c.k, c.v, bias, kv_lengths=c.kv_lengths, scale=c.scale)
    b = oracle.tri_fwd(c.q, c.k, c.v, bias + 2.5, kv_lengths=c.kv_lengths, scale=c.scale)
    np.testing.assert_allclose(b[0], a[0], atol=1e-13)
    np.testing.assert_allclose(b[1], a[1] + 2.5, atol=1e-12)
    np.testing.assert_allclose(b[2], a[2] + 2.5, atol=1e-12)


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

def test_kv_lengths_equals_right_padded_dense_mask():
    c = synth.make_triangle("t", 2, 5, 2, 7, 13, 8, "bf16", "bf16", seed=17, mask="kvlen", kv_range=(0, 13))
    pos = torch.arange(13)
    dense = (pos.view(1, 1, 13) < c.kv_lengths.view(2, 5, 1)).view(2, 5, 1, 1, 13).to(torch.uint8)
    a = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale)
    b = oracle.tri_fwd(c.q, c.k, c.v, c.bias, mask=dense, scale=c.scale)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_joint_key_permutation_leaves_output_unchanged():
    c = synth.make_triangle("t", 1, 3, 2, 5, 10, 8, "f32", "f32", seed=18, mask="dense")
    perm = torch.randperm(10, generator=torch.Generator().manual_seed(3))
    a = oracle.tri_fwd(c.q, c.k, c.v, c.bias, mask=c.mask, scale=c.scale)
    b = oracle.tri_fwd(c.q, c.k[:, :, :, perm], c.v[:, :, :, perm], c.bias[..., perm],
                       mask=c.mask[..., perm], scale=c.scale)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-13)


def test_n_slice_alone_gives_same_rows():
    """The bias (B,1,H,Q,K) is shared over N: one n computed alone must agree."""
    c = synth.make_triangle("t", 1, 4, 2, 5, 9, 8, "f16", "f32", seed=19, mask="kvlen", kv_range=(0, 9))
    a = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale)
    for n in range(4):
        sl = slice(n, n + 1)
        b = oracle.tri_fwd(c.q[:, sl], c.k[:, sl], c.v[:, sl], c.bias, kv_lengths=c.kv_lengths[:, sl],
                           scale=c.scale)
        np.testing.assert_array_equal(a[0][:, sl], b[0])
        np.testing.assert_array_equal(a[1][:, sl], b[1])


def test_lse_bounds():
    c = synth.make_triangle("t", 1, 6, 2, 8, 16, 8, "f32", "f32", seed=20, bias_std=4.0, mask="dense")
    _, L, M = oracle.tri_fwd(c.q, c.k, c.v, c.bias, mask=c.mask, scale=c.scale)
    assert (M <= L + 1e-12).all()
    assert (L <= M + math.log(16) + 1e-12).all()


def test_row_subset_matches_full():
    c = synth.make_triangle("t", 1, 3, 2, 5, 9, 8, "bf16", "bf16", seed=21, mask="kvlen", kv_range=(0, 9))
    O, L, M = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale)
    rows = np.array([0, 7, 13, 29])
    o, l, m = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale, rows=rows)
    np.testing.assert_array_equal(o, O.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(l, L.reshape(-1)[rows])
    np.testing.assert_array_equal(m, M.reshape(-1)[rows])


# ---------------------------------------------------------------------------
# Library special cases (torch SDPA in fp64 on the CPU)
# ---------------------------------------------------------------------------

def _sdpa(q, k, v, attn_mask, scale):
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=attn_mask, scale=scale)


def test_unmasked_equals_sdpa_with_bias():
    c = synth.make_triangle("t", 2, 3, 2, 7, 11, 16, "f32", "f32", seed=22, bias_std=2.0)
    O, _, _ = oracle.tri_fwd(c.q, c.k, c.v, c.bias, scale=c.scale)
    s = float(np.float32(c.scale))
    ref = _sdpa(_f64(c.q), _f64(c.k), _f64(c.v), _f64(c.bias), s)  # bias broadcasts over N
    np.testing.assert_allclose(O, ref.numpy(), atol=1e-12)


def test_identity_values_give_softmax_weights():
    """With V = I (D = K) the output row is the softmax itself; lse = x_k - log p_k."""
    K = 6
    c = synth.make_triangle("t", 1, 2, 1, 4, K, K, "f32", "f32", seed=23)
    v = torch.eye(K).view(1, 1, 1, K, K).expand(1, 2, 1, K, K).contiguous()
    O, L, _ = oracle.tri_fwd(c.q, c.k, v, c.bias, scale=c.scale)
    s = float(np.float32(c.scale))
    ref = _sdpa(_f64(c.q), _f64(c.k), _f64(v), _f64(c.bias), s)
    np.testing.assert_allclose(O, ref.numpy(), atol=1e-13)
    assert np.allclose(O.sum(-1), 1.0, atol=1e-14)


def test_prefix_lengths_equal_sdpa_on_truncated_keys():
    """A row with L >= 1 valid prefix keys equals plain attention over those L keys
    (the -1e9 logits contribute exactly zero weight)."""
    c = synth.make_triangle("t", 1, 4, 2, 6, 12, 8, "f16", "f32", seed=24, mask="kvlen", kv_range=(1, 12))
    O, _, _ = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale)
    s = float(np.float32(c.scale))
    for n in range(4):
        L = int(c.kv_lengths[0, n])
        ref = _sdpa(_f64(c.q[0, n]), _f64(c.k[0, n, :, :L]), _f64(c.v[0, n, :, :L]),
                    _f64(c.bias[0, 0, :, :, :L]), s)
        np.testing.assert_allclose(O[0, n], ref.numpy(), atol=1e-12)


def test_dense_mask_equals_sdpa_with_boolean_mask():
    c = synth.make_triangle("t", 1, 4, 2, 6, 12, 8, "bf16", "bf16", seed=25, mask="dense", mask_p=0.6)
    c.mask[..., 0] = 1  # every row keeps at least one key, so -1e9 and -inf agree
    O, _, _ = oracle.tri_fwd(c.q, c.k, c.v, c.bias, mask=c.mask, scale=c.scale)
    s = float(np.float32(c.scale))
    for n in range(4):
        keep = c.mask[0, n, 0, 0].bool().view(1, 1, 12)
        add = torch.where(keep, _f64(c.bias[0, 0]), torch.tensor(float("-inf"), dtype=torch.float64))
        ref = _sdpa(_f64(c.q[0, n]), _f64(c.k[0, n]), _f64(c.v[0, n]), add, s)
        np.testing.assert_allclose(O[0, n], ref.numpy(), atol=1e-12)


# ---------------------------------------------------------------------------
# Packed sequences + BlockMask
# ---------------------------------------------------------------------------

def test_to_dense_reconstruction_hand_case():
    """The BlockMask page's loop: entries past the count are never read, repeats set once."""
    num = np.array([2, 0, 3])
    idx = np.array([[1, 3, 0], [2, 2, 2], [0, 0, 2]])
    d = oracle.to_dense(num, idx, 4)
    np.testing.assert_array_equal(d, [[0, 1, 0, 1], [0, 0, 0, 0], [1, 0, 1, 0]])


def _varlen_sdpa(c, keep_fn):
    """Per (sequence, head) SDPA in fp64 with a boolean keep-mask from keep_fn(Lq, Lk)."""
    s = float(np.float32(c.scale))
    outs = []
    for i in range(len(c.lengths)):
        a, b = int(c.cu_seqlens[i]), int(c.cu_seqlens[i + 1])
        q = _f64(c.q[a:b]).transpose(0, 1)
        k = _f64(c.k[a:b]).transpose(0, 1)
        v = _f64(c.v[a:b]).transpose(0, 1)
        keep = keep_fn(b - a, b - a)
        outs.append(_sdpa(q, k, v, keep, s).transpose(0, 1))
    return torch.cat(outs).numpy()


def test_varlen_causal_blockmask_equals_causal_attention():
    c = synth.make_varlen("t", 3, 130, 300, 2, 16, "bf16", seed=26, lengths=[130, 257, 300])
    O, L, M = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, c.kv_num_blocks,
                                c.kv_indices, c.full_kv_num_blocks, c.full_kv_indices, mask_mod="causal")
    ref = _varlen_sdpa(c, lambda lq, lk: torch.ones(lq, lk, dtype=torch.bool).tril())
    np.testing.assert_allclose(O, ref, atol=1e-12)
    assert (M <= L).all()


def test_varlen_no_lists_no_mask_is_full_attention():
    c = synth.make_varlen("t", 2, 20, 40, 2, 8, "f16", seed=27, lengths=[20, 33], block_lists="none",
                          mask_mod="none")
    O, _, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, mask_mod="none")
    ref = _varlen_sdpa(c, lambda lq, lk: None)
    np.testing.assert_allclose(O, ref, atol=1e-12)


def test_varlen_random_lists_equal_reconstructed_dense_mask():
    """block-sparse == its reconstructed dense mask, partial blocks under causal mask_mod."""
    g = np.random.default_rng(5)
    lengths = [300, 200]
    c = synth.make_varlen("t", 2, 0, 0, 2, 8, "f32", seed=28, lengths=lengths, block_lists="none")
    MQ = MK = 3
    kv_num = np.zeros((2, 1, MQ), np.int32)
    kv_idx = np.zeros((2, 1, MQ, MK), np.int32)
    full_num = np.zeros((2, 1, MQ), np.int32)
    full_idx = np.zeros((2, 1, MQ, MK), np.int32)
    for s, L in enumerate(lengths):
        nb = (L + 127) // 128
        for qb in range(nb):
            blocks = list(g.permutation(nb))
            nf = int(g.integers(0, len(blocks) + 1))
            full = blocks[:nf]
            part = blocks[nf:]
            if 0 not in full and 0 not in part:
                full.append(0)
            full_num[s, 0, qb] = len(full)
            full_idx[s, 0, qb, :len(full)] = full
            kv_num[s, 0, qb] = len(part)
            kv_idx[s, 0, qb, :len(part)] = part
            kv_idx[s, 0, qb, len(part):] = 99  # past the count: must never be read
    # Every row keeps key 0 (block 0 is listed; under causal k=0 <= q), so -1e9 == -inf here.
    O, _, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale,
                                torch.from_numpy(kv_num), torch.from_numpy(kv_idx),
                                torch.from_numpy(full_num), torch.from_numpy(full_idx), mask_mod="causal")

    def keep_for(s):
        def fn(lq, lk):
            nbq, nbk = (lq + 127) // 128, (lk + 127) // 128
            part = oracle.to_dense(kv_num[s, 0, :nbq], kv_idx[s, 0, :nbq], nbk)
            full = oracle.to_dense(full_num[s, 0, :nbq], full_idx[s, 0, :nbq], nbk)
            qi = torch.arange(lq).view(-1, 1)
            kj = torch.arange(lk).view(1, -1)
            pb = torch.from_numpy(part)[qi // 128, kj // 128].bool()
            fb = torch.from_numpy(full)[qi // 128, kj // 128].bool()
            return fb | (pb & (kj <= qi))
        return fn

    outs = []
    s32 = float(np.float32(c.scale))
    for i in range(2):
        a, b = int(c.cu_seqlens[i]), int(c.cu_seqlens[i + 1])
        keep = keep_for(i)(b - a, b - a)
        outs.append(_sdpa(_f64(c.q[a:b]).transpose(0, 1), _f64(c.k[a:b]).transpose(0, 1),
                          _f64(c.v[a:b]).transpose(0, 1), keep, s32).transpose(0, 1))
    np.testing.assert_allclose(O, torch.cat(outs).numpy(), atol=1e-12)


def test_varlen_unlisted_row_is_mean_of_sequence_values():
    """A q-block with no listed kv block: every logit is -1e9, so O = mean of V over the sequence."""
    c = synth.make_varlen("t", 1, 0, 0, 2, 8, "f32", seed=29, lengths=[200], block_lists="none")
    kv_num = torch.zeros(1, 1, 2, dtype=torch.int32)
    kv_idx = torch.zeros(1, 1, 2, 2, dtype=torch.int32)
    O, L, M = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, kv_num, kv_idx,
                                mask_mod="causal")
    mean = _f64(c.v).mean(dim=0).numpy()
    np.testing.assert_allclose(O, np.broadcast_to(mean, O.shape), atol=1e-13)
    np.testing.assert_allclose(M, -1e9)
    np.testing.assert_allclose(L, -1e9 + math.log(200), atol=1e-6)


# ---------------------------------------------------------------------------
# The page's worked example
# ---------------------------------------------------------------------------

def test_page_example_golden():
    with open(os.path.join(HERE, "golden", "page_example.json")) as f:
        g = json.load(f)
    S, V = g["seq_len"], g["seq_lengths"][0]
    mask = synth.page_example_kv_lengths(S, V)
    kl, prefix = oracle.mask_to_kv_lengths(mask)
    exp = g["kv_lengths_from_example_mask"]
    assert kl[0, :V].tolist() == [exp["rows_lt_96"]] * V
    assert kl[0, V:].tolist() == [exp["rows_ge_96"]] * (S - V)
    assert bool(prefix.all())
    # Output shape printed by the example, on a reduced copy of its inputs
    c = synth.fp16_page_example()
    O, L, M = oracle.tri_fwd(c.q[:, :2], c.k[:, :2], c.v[:, :2], c.bias, kv_lengths=kl[:, :2], scale=c.scale)
    assert list(O.shape)[2:] == g["printed_shapes"]["output"][2:]
    assert list(c.q.shape) == g["printed_shapes"]["output"]
    assert list(c.bias.shape) == g["printed_shapes"]["bias.grad"]


def test_mask_to_kv_lengths_flags_holey_rows():
    m = torch.tensor([[1, 1, 0, 0], [1, 0, 1, 0], [0, 0, 0, 0], [1, 1, 1, 1]], dtype=torch.uint8)
    kl, pre = oracle.mask_to_kv_lengths(m.view(1, 4, 1, 1, 4))
    assert kl.view(-1).tolist() == [2, 1, 0, 4]
    assert pre.view(-1).tolist() == [True, False, True, True]


def _varlen_sdpa_pairs(c, keep_fn):
    """Per (sequence, head) fp64 SDPA over Lq x Lk with keep_fn(seq, head, Lq, Lk) -> bool (Lq, Lk)."""
    s = float(np.float32(c.scale))
    out = torch.zeros(c.q.shape, dtype=torch.float64)
    for i in range(len(c.lengths)):
        a, b = int(c.cu_seqlens[i]), int(c.cu_seqlens[i + 1])
        ka, kb = int(c.cu_seqlens_k[i]), int(c.cu_seqlens_k[i + 1])
        for h in range(c.H):
            keep = keep_fn(i, h, b - a, kb - ka)
            out[a:b, h] = _sdpa(_f64(c.q[a:b, h]), _f64(c.k[ka:kb, h]), _f64(c.v[ka:kb, h]), keep, s)
    return out.numpy()


def test_varlen_causal_top_left_when_key_and_query_lengths_differ():
    """Lq != Lk: causal keeps key k for query q when k <= q, both counted from the start of their
    own sequence (top-left alignment); checked against SDPA with that element mask."""
    c = synth.make_varlen("t", 3, 0, 0, 2, 8, "f32", seed=30, lengths=[200, 70, 130], lengths_k=[90, 260, 130],
                          block_lists="none", mask_mod="causal")
    O, L, M = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens_k, c.scale, mask_mod="causal")
    ref = _varlen_sdpa_pairs(c, lambda i, h, lq, lk: torch.arange(lk).view(1, -1) <= torch.arange(lq).view(-1, 1))
    np.testing.assert_allclose(O, ref, atol=1e-12)
    # a query row past every key (q >= Lk) sees the whole key sequence
    a = int(c.cu_seqlens[0])
    full = _sdpa(_f64(c.q[a + 150:a + 151, 0]), _f64(c.k[:90, 0]), _f64(c.v[:90, 0]), None,
                 float(np.float32(c.scale)))
    np.testing.assert_allclose(O[a + 150, 0], full[0].numpy(), atol=1e-12)
    # no mask: plain attention over each sequence's own keys
    O2, _, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens_k, c.scale, mask_mod="none")
    np.testing.assert_allclose(O2, _varlen_sdpa_pairs(c, lambda i, h, lq, lk: None), atol=1e-12)


def test_varlen_lists_with_key_and_query_lengths_differ():
    """Random block lists over an Lq x Lk block grid equal their element mask (full | partial & causal)."""
    g = np.random.default_rng(31)
    lq, lk = [300, 140], [180, 390]
    c = synth.make_varlen("t", 2, 0, 0, 2, 8, "bf16", seed=31, lengths=lq, lengths_k=lk, block_lists="none")
    MQ, MK = 3, 4
    kv_num = np.zeros((2, 1, MQ), np.int32)
    kv_idx = np.full((2, 1, MQ, MK), 77, np.int32)
    full_num = np.zeros((2, 1, MQ), np.int32)
    full_idx = np.full((2, 1, MQ, MK), 77, np.int32)
    for s in range(2):
        nbq, nbk = (lq[s] + 127) // 128, (lk[s] + 127) // 128
        for qb in range(nbq):
            blocks = [int(x) for x in g.permutation(nbk)]
            if 0 in blocks:  # block 0 always listed, so every row keeps key 0 under causal
                blocks.remove(0)
            blocks = [0] + blocks[:int(g.integers(0, len(blocks) + 1))]
            nf = int(g.integers(0, len(blocks) + 1))
            full_num[s, 0, qb] = nf
            full_idx[s, 0, qb, :nf] = blocks[:nf]
            kv_num[s, 0, qb] = len(blocks) - nf
            kv_idx[s, 0, qb, :len(blocks) - nf] = blocks[nf:]
    O, _, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens_k, c.scale, torch.from_numpy(kv_num),
                                torch.from_numpy(kv_idx), torch.from_numpy(full_num), torch.from_numpy(full_idx),
                                mask_mod="causal")

    def keep(i, h, nq, nk):
        qi = torch.arange(nq).view(-1, 1)
        kj = torch.arange(nk).view(1, -1)
        fb = torch.zeros(nq, nk, dtype=torch.bool)
        pb = torch.zeros(nq, nk, dtype=torch.bool)
        for qb in range((nq + 127) // 128):
            for t in range(full_num[i, 0, qb]):
                fb[qb * 128:(qb + 1) * 128, full_idx[i, 0, qb, t] * 128:(full_idx[i, 0, qb, t] + 1) * 128] = True
            for t in range(kv_num[i, 0, qb]):
                pb[qb * 128:(qb + 1) * 128, kv_idx[i, 0, qb, t] * 128:(kv_idx[i, 0, qb, t] + 1) * 128] = True
        return fb | (pb & (kj <= qi))

    np.testing.assert_allclose(O, _varlen_sdpa_pairs(c, keep), atol=1e-12)


def test_varlen_per_head_lists_index_by_head():
    """mask_heads = H: head h reads row [seq, h, q block] of the lists; per-head SDPA with the
    element mask of that head's lists."""
    lengths = [260, 200]
    c = synth.make_varlen("t", 2, 0, 0, 3, 8, "f32", seed=32, lengths=lengths, block_lists="none")
    kn, ki, fn, fi = synth.causal_block_lists(lengths, mask_heads=3)
    fn[:, 1] = 0              # head 1: diagonal blocks only
    kn[:, 2] = 0              # head 2: full blocks only (the diagonal block is unlisted)
    O, _, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, kn, ki, fn, fi,
                                mask_mod="causal")

    def keep(i, h, nq, nk):
        qi = torch.arange(nq).view(-1, 1)
        kj = torch.arange(nk).view(1, -1)
        same_block = (qi // 128) == (kj // 128)
        earlier_block = (kj // 128) < (qi // 128)
        if h == 0:
            return kj <= qi
        if h == 1:
            return same_block & (kj <= qi)
        return earlier_block

    ref = _varlen_sdpa_pairs(c, keep)
    # head 2, q block 0 lists nothing: every logit is -1e9 -> mean of V over the sequence (not SDPA's NaN)
    for i, L in enumerate(lengths):
        a = int(c.cu_seqlens[i])
        ref[a:a + min(128, L), 2] = _f64(c.v[a:a + L, 2]).mean(0).numpy()
    np.testing.assert_allclose(O, ref, atol=1e-12)


@pytest.mark.parametrize("window", [1, 5, 130, 1000])
def test_varlen_sliding_window_equals_banded_attention(window):
    """mask_mod sliding_window(W): query q keeps keys q - W < k <= q (itself and the W - 1 before
    it), local indices; W = 1 keeps only the diagonal, W >= L is plain causal."""
    c = synth.make_varlen("t", 3, 0, 0, 2, 8, "f32", seed=33, lengths=[200, 7, 300], block_lists="none",
                          mask_mod="sliding_window")
    O, L, M = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, mask_mod="sliding_window",
                                window=window)

    def keep(i, h, nq, nk):
        qi = torch.arange(nq).view(-1, 1)
        kj = torch.arange(nk).view(1, -1)
        return (kj <= qi) & (qi - kj < window)

    np.testing.assert_allclose(O, _varlen_sdpa_pairs(c, keep), atol=1e-12)
    if window == 1:  # one key per row: O is that key's value, lse = max = its logit
        np.testing.assert_allclose(O, _f64(c.v).numpy(), atol=1e-12)
        np.testing.assert_allclose(L, M, atol=1e-12)


def test_varlen_sliding_window_with_block_lists():
    """The window applies on partial blocks only; full blocks keep every key."""
    lengths = [300, 260]
    c = synth.make_varlen("t", 2, 0, 0, 2, 8, "bf16", seed=34, lengths=lengths, block_lists="none")
    kn, ki, fn, fi = synth.causal_block_lists(lengths)   # diagonal partial, earlier blocks full
    W = 40
    O, _, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, kn, ki, fn, fi,
                                mask_mod="sliding_window", window=W)

    def keep(i, h, nq, nk):
        qi = torch.arange(nq).view(-1, 1)
        kj = torch.arange(nk).view(1, -1)
        diag = (qi // 128) == (kj // 128)
        earlier = (kj // 128) < (qi // 128)
        return earlier | (diag & (kj <= qi) & (qi - kj < W))

    np.testing.assert_allclose(O, _varlen_sdpa_pairs(c, keep), atol=1e-12)


@pytest.mark.parametrize("window", [1, 100, 128, 129, 300])
def test_window_block_lists_give_banded_attention(window):
    """The sliding-window block lists of the input generator (full where the whole block pair is
    inside the band, partial where the band's edge or the diagonal crosses it) with mask_mod
    sliding_window reproduce the banded attention q - W < k <= q exactly (fp64 SDPA with the
    band built here), so skipping unlisted blocks loses nothing."""
    lengths = [400, 129, 1, 260]
    c = synth.make_varlen("t", 4, 0, 0, 2, 8, "f32", seed=38, lengths=lengths, mask_mod="sliding_window",
                          block_lists=f"window{window}")
    O, L, M = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, c.kv_num_blocks, c.kv_indices,
                                c.full_kv_num_blocks, c.full_kv_indices, mask_mod="sliding_window", window=window)

    def keep(i, h, nq, nk):
        qi = torch.arange(nq).view(-1, 1)
        kj = torch.arange(nk).view(1, -1)
        return (kj <= qi) & (qi - kj < window)

    np.testing.assert_allclose(O, _varlen_sdpa_pairs(c, keep), atol=1e-12)
    # the lists are minimal: every listed block pair holds a kept (q, k) pair of the band
    for i, Lq in enumerate(lengths):
        nb = (Lq + 127) // 128
        for qb in range(nb):
            listed = [int(x) for x in c.kv_indices[i, 0, qb, :int(c.kv_num_blocks[i, 0, qb])]]
            listed += [int(x) for x in c.full_kv_indices[i, 0, qb, :int(c.full_kv_num_blocks[i, 0, qb])]]
            assert len(listed) == len(set(listed))
            for kb in listed:
                assert kb * 128 <= qb * 128 + 127 and kb * 128 + 127 > qb * 128 - window


@pytest.mark.parametrize("prefix", [0, 1, 50, 129, [10, 0, 400]])
def test_varlen_prefix_lm_equals_prefix_plus_causal(prefix):
    """mask_mod prefix_lm(P): query q keeps keys k <= q or k < P (the prefix is seen by every
    query of the sequence); P = 0 is plain causal; P may differ per sequence."""
    lengths = [200, 70, 300]
    c = synth.make_varlen("t", 3, 0, 0, 2, 8, "f32", seed=35, lengths=lengths, block_lists="none",
                          mask_mod="prefix_lm")
    O, _, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, mask_mod="prefix_lm",
                                prefix_lengths=prefix)
    per = prefix if isinstance(prefix, list) else [prefix] * 3

    def keep(i, h, nq, nk):
        qi = torch.arange(nq).view(-1, 1)
        kj = torch.arange(nk).view(1, -1)
        return (kj <= qi) | (kj < per[i])

    np.testing.assert_allclose(O, _varlen_sdpa_pairs(c, keep), atol=1e-12)
    if per == [0, 0, 0]:
        Oc, _, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, mask_mod="causal")
        np.testing.assert_array_equal(O, Oc)


@pytest.mark.parametrize("mask_mod", ["none", "causal"])
def test_varlen_bias_equals_sdpa_with_additive_bias(mask_mod):
    """Post-scale bias on the packed form (Transformer Engine fused_attn.h, NVTE_POST_SCALE_BIAS):
    bias (H, max_q, max_k) indexed by each sequence's local positions, added to the scaled
    logits of valid keys; SDPA with the sliced bias (and -inf off the causal triangle)."""
    lengths, lk = [70, 130, 9], [50, 140, 16]
    c = synth.make_varlen("t", 3, 0, 0, 2, 8, "f32", seed=36, lengths=lengths, lengths_k=lk, block_lists="none",
                          mask_mod=mask_mod)
    g = torch.Generator().manual_seed(37)
    bias = (2.0 * torch.randn(2, 136, 144, generator=g)).to(torch.bfloat16)
    O, L, M = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens_k, c.scale, mask_mod=mask_mod, bias=bias)
    s = float(np.float32(c.scale))
    ref = torch.zeros(c.q.shape, dtype=torch.float64)
    for i in range(3):
        a, b = int(c.cu_seqlens[i]), int(c.cu_seqlens[i + 1])
        ka, kb = int(c.cu_seqlens_k[i]), int(c.cu_seqlens_k[i + 1])
        nq, nk = b - a, kb - ka
        for h in range(2):
            add = _f64(bias[h, :nq, :nk]).clone()
            if mask_mod == "causal":
                add[torch.arange(nk).view(1, -1) > torch.arange(nq).view(-1, 1)] = float("-inf")
            ref[a:b, h] = _sdpa(_f64(c.q[a:b, h]), _f64(c.k[ka:kb, h]), _f64(c.v[ka:kb, h]), add, s)
    np.testing.assert_allclose(O, ref.numpy(), atol=1e-12)
    O0, L0, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens_k, c.scale, mask_mod=mask_mod,
                                  bias=torch.zeros(2, 136, 144))
    O1, L1, _ = oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens_k, c.scale, mask_mod=mask_mod,
                                  bias=torch.full((2, 136, 144), 3.0))
    np.testing.assert_allclose(O1, O0, atol=1e-13)        # a constant bias leaves O unchanged ...
    np.testing.assert_allclose(L1, L0 + 3.0, atol=1e-12)  # ... and shifts lse by that constant
