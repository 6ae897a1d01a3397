"""GPU parity: the library against the fp64 oracle on the same seeded inputs.

Tolerances (max-abs): fp32 inputs O 1e-4, lse/max 1e-5; fp16/bf16 inputs
O 2e-2, lse/max 5e-3.  The named workloads run at full size (the largest one
is checked on a sample of rows the oracle computes one by one, in the same
launch configuration the benchmark times); edge cases cover ragged tails,
every supported head dimension, all-masked rows and kv_lengths extremes.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity_helpers import check_triangle, check_varlen, compare, run_triangle, run_varlen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from masked_attention_tri_gb300 import build
    build.build()


# ---------------------------------------------------------------------------
# The named workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny_fp32", "fp16_kvlen", "fp16_dense", "fp16_page_example", "bf16_pairstack"])
def test_workload_full(name):
    check_triangle(synth.TRIANGLE_WORKLOADS[name]())


def test_bf16_long_all_rows():
    """The largest workload, every row, in the launch configuration the benchmark times.  The oracle
    runs on the host's cores in slab chunks (about 15 s of CPU work on 16 cores)."""
    c = synth.bf16_long()
    O, L, M = run_triangle(c)
    O = O.reshape(-1, c.D)
    L, M = L.reshape(-1), M.reshape(-1)
    per_n = c.H * c.Q
    chunk = 96  # (b, n) slabs per oracle call
    worst = 0.0
    for n0 in range(0, c.B * c.N, chunk):
        rows = np.arange(n0 * per_n, min(c.B * c.N, n0 + chunk) * per_n, dtype=np.int64)
        rO, rL, rM = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale, rows=rows)
        sel = torch.as_tensor(rows, device=O.device)
        worst = max(worst, compare(f"{c.name}[n {n0}..]", c.dtype, O[sel], L[sel], M[sel], rO, rL, rM))
    assert worst > 0.0


def test_bf16_varlen_full():
    check_varlen(synth.bf16_varlen())


def test_bf16_varlen_window512_full():
    """The benchmark's sliding-window workload (the bf16_varlen sequences, window 512 with its
    block lists), every row."""
    check_varlen(synth.bf16_varlen_window512(), window=512)


def test_bf16_d256_full():
    """The benchmark's D = 256 workload (CUDA-core kernel), every row."""
    check_triangle(synth.bf16_d256())


# ---------------------------------------------------------------------------
# Edge cases: ragged tiles, head dimensions, kv_lengths extremes
# ---------------------------------------------------------------------------

# D <= 64 runs on the key-split kernel (D in (48, 64] stores each key half's
# 32 O columns at once, smaller D in 8-column pieces); D > 64 on the
# two-tile kernel.
@pytest.mark.parametrize("D", [8, 16, 24, 32, 40, 48, 56, 64, 96, 128])
def test_bf16_head_dims_ragged(D):
    c = synth.make_triangle(f"bf16_D{D}", 1, 3, 2, 200, 136, D, "bf16", "bf16", seed=100 + D, mask="kvlen",
                            kv_range=(0, 136))
    c.kv_lengths.view(-1)[:3] = torch.tensor([0, 136, 1000], dtype=torch.int32)
    check_triangle(c)


@pytest.mark.parametrize("D", [8, 32, 56, 64, 128])
def test_fp16_fp32_bias_no_mask(D):
    c = synth.make_triangle(f"f16_D{D}", 2, 2, 3, 130, 264, D, "f16", "f32", seed=200 + D)
    check_triangle(c)


@pytest.mark.parametrize("L", [0, 1, 7, 127, 128, 129, 255, 256, 300, 1000, -4])
def test_kv_length_values(L):
    c = synth.make_triangle(f"kvlen_{L}", 1, 2, 2, 160, 256, 64, "bf16", "bf16", seed=300, mask="kvlen", kv_const=L)
    check_triangle(c)


def test_dense_mask_special_rows():
    c = synth.make_triangle("dense_rows", 1, 6, 2, 150, 200, 32, "f16", "f16", seed=301, mask="dense", mask_p=0.3)
    c.mask[0, 0] = 0                 # all masked -> mean of V
    c.mask[0, 1] = 0
    c.mask[0, 1, ..., 199] = 1       # one valid key, in the ragged last tile
    c.mask[0, 2] = 1                 # all valid
    c.mask[0, 3, ..., 128:] = 0      # second tile fully masked
    check_triangle(c)


# Dense masks on the two-tile kernel (D > 64): the bias warp's mask-bit words and the
# masking of boundary tiles, with all-masked rows, one valid key in the ragged last
# tile, a fully masked middle tile and an all-valid row.
@pytest.mark.parametrize("D,dtype,bias_dtype", [(96, "bf16", "bf16"), (128, "bf16", "f32"), (96, "f16", "f32"),
                                                (128, "f16", "f16")])
def test_dense_mask_wide_heads(D, dtype, bias_dtype):
    c = synth.make_triangle(f"dense_D{D}", 1, 6, 2, 150, 328, D, dtype, bias_dtype, seed=302 + D, mask="dense",
                            mask_p=0.3)
    c.mask[0, 0] = 0                 # all masked -> mean of V
    c.mask[0, 1] = 0
    c.mask[0, 1, ..., 327] = 1       # one valid key, in the ragged last tile
    c.mask[0, 2] = 1                 # all valid
    c.mask[0, 3, ..., 128:256] = 0   # middle tile fully masked
    check_triangle(c)


# Strided q / k / v (the triangle form read in place): a (B,N,Q,H,D) buffer viewed as
# (B,N,H,Q,D), and rows padded past D; on the key-split kernel (D <= 64), the two-tile
# kernel (D > 64), the fp32 CUDA-core kernel and, for 16-bit D > 128 (whose tensor-core
# kernel takes contiguous tensors only), the CUDA-core kernel.  Same result as the
# contiguous copy.
@pytest.mark.parametrize("D,dtype", [(64, "bf16"), (32, "f16"), (128, "bf16"), (16, "f32"), (192, "bf16")])
def test_triangle_strided_views(D, dtype):
    c = synth.make_triangle(f"strided_D{D}", 2, 3, 2, 150, 136, D, dtype, dtype, seed=720 + D, mask="kvlen",
                            kv_range=(0, 136))
    import masked_attention_tri_gb300 as ta
    q, k, v, bias, kl = (t.cuda() for t in (c.q, c.k, c.v, c.bias, c.kv_lengths))
    # q: transposed from (B,N,Q,H,D); k: rows padded to D + 8; v: transposed and padded
    qt = torch.empty(c.B, c.N, c.Q, c.H, D, dtype=q.dtype, device="cuda")
    qt.copy_(q.transpose(2, 3))
    kp = torch.full((c.B, c.N, c.H, c.K, D + 8), 7.0, dtype=k.dtype, device="cuda")
    kp[..., :D] = k
    vt = torch.full((c.B, c.N, c.K, c.H, D + 8), -3.0, dtype=v.dtype, device="cuda")
    vt[..., :D].copy_(v.transpose(2, 3))
    qv, kv_, vv = qt.transpose(2, 3), kp[..., :D], vt[..., :D].transpose(2, 3)
    assert not qv.is_contiguous() and not kv_.is_contiguous() and not vv.is_contiguous()
    o1, l1, m1 = ta.triangle_attention(qv, kv_, vv, bias, scale=c.scale, return_aux=True, kv_lengths=kl)
    o0, l0, m0 = ta.triangle_attention(q, k, v, bias, scale=c.scale, return_aux=True, kv_lengths=kl)
    torch.cuda.synchronize()
    assert ta.get_status() == 0
    assert o1.is_contiguous()
    rO, rL, rM = oracle.tri_fwd(c.q, c.k, c.v, c.bias, kv_lengths=c.kv_lengths, scale=c.scale)
    compare(c.name, c.dtype, o1, l1, m1, rO, rL, rM)
    if D > 128 and dtype != "f32":  # the views and the contiguous copy take different kernels here
        compare(c.name + "_contiguous", c.dtype, o0, l0, m0, rO, rL, rM)
    else:
        assert torch.equal(o1, o0) and torch.equal(l1, l0) and torch.equal(m1, m0)


# D in (128, 256] (the page's forward bound for half precision): 16-bit inputs on the
# tensor-core kernel with 64-key tiles, fp32 on the CUDA-core kernel; ragged tiles and
# kv_lengths extremes.
@pytest.mark.parametrize("dtype,bias_dtype,D", [("bf16", "bf16", 136), ("bf16", "f32", 192), ("bf16", "bf16", 256),
                                                ("f16", "f32", 256), ("f16", "f16", 200), ("f32", "f32", 256)])
def test_wide_head_dims(dtype, bias_dtype, D):
    c = synth.make_triangle(f"wide_{dtype}_D{D}", 1, 3, 2, 70, 136, D, dtype, bias_dtype, seed=470 + D, mask="kvlen",
                            kv_range=(0, 136))
    c.kv_lengths.view(-1)[:3] = torch.tensor([0, 136, 1], dtype=torch.int32)
    check_triangle(c)


def test_wide_head_dim_dense_mask():
    c = synth.make_triangle("wide_dense", 2, 2, 2, 33, 80, 256, "bf16", "f32", seed=480, mask="dense")
    c.mask[1, 1] = 0
    check_triangle(c)


# The tensor-core kernel for D in (128, 256] (64-key tiles): more work items than CTAs, several
# query and key tiles per slab with ragged tails, kv_lengths extremes, and large logits (the
# lazy O correction over all D columns).
@pytest.mark.parametrize("dtype,bias_dtype,D", [("bf16", "bf16", 256), ("f16", "f32", 144), ("bf16", "f32", 200)])
def test_wide_head_dims_many_tiles(dtype, bias_dtype, D):
    c = synth.make_triangle(f"wide_tiles_{dtype}_{D}", 1, 40, 4, 300, 264, D, dtype, bias_dtype, seed=485 + D,
                            mask="kvlen", kv_range=(0, 264))
    c.kv_lengths.view(-1)[:5] = torch.tensor([0, 1, 64, 65, 264], dtype=torch.int32)
    check_triangle(c)


def test_wide_head_dims_large_logits():
    c = synth.make_triangle("wide_large", 1, 3, 2, 200, 200, 256, "bf16", "bf16", seed=489, bias_std=8.0, scale=0.5,
                            mask="kvlen", kv_range=(10, 200))
    check_triangle(c)


@pytest.mark.parametrize("dtype,D", [("bf16", 256), ("f16", 192)])
@pytest.mark.parametrize("lists", ["causal", "none"])
def test_varlen_wide_head_dims(dtype, D, lists):
    c = synth.make_varlen(f"vl_wide_{dtype}_{D}_{lists}", 3, 0, 0, 2, D, dtype, seed=490 + D, lengths=[150, 1, 70],
                          block_lists=lists, mask_mod="causal")
    check_varlen(c)


@pytest.mark.parametrize("D", [4, 12, 32, 100, 128])
def test_fp32_head_dims(D):
    c = synth.make_triangle(f"f32_D{D}", 1, 2, 2, 45, 70, D, "f32", "f32", seed=400 + D, mask="kvlen",
                            kv_range=(0, 70))
    c.kv_lengths.view(-1)[0] = 0
    check_triangle(c)


def test_fp32_dense_mask():
    c = synth.make_triangle("f32_dense", 2, 3, 2, 33, 65, 16, "f32", "f32", seed=450, mask="dense")
    c.mask[1, 2] = 0
    check_triangle(c)


def test_single_query_single_key():
    c = synth.make_triangle("1x8", 1, 1, 1, 1, 8, 8, "bf16", "f32", seed=451)
    check_triangle(c)


def test_large_logits_bias_and_scale():
    c = synth.make_triangle("large", 1, 2, 2, 128, 128, 64, "bf16", "bf16", seed=452, bias_std=30.0, scale=0.5,
                            mask="kvlen", kv_range=(1, 128))
    check_triangle(c)


# ---------------------------------------------------------------------------
# Packed sequences
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("D", [32, 64, 128])
def test_varlen_causal_ragged(D):
    c = synth.make_varlen(f"vl_causal_D{D}", 4, 0, 0, 2, D, "bf16", seed=500 + D, lengths=[1, 129, 300, 128])
    check_varlen(c)


def test_varlen_no_lists_full_and_causal():
    c = synth.make_varlen("vl_none", 3, 0, 0, 2, 64, "f16", seed=510, lengths=[77, 256, 5], block_lists="none",
                          mask_mod="none")
    check_varlen(c)
    c.mask_mod = "causal"
    check_varlen(c)


@pytest.mark.parametrize("mask_mod", ["none", "causal"])
@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("f32", 32)])
def test_varlen_key_lengths_differ(mask_mod, dtype, D):
    """cu_seqlens_q != cu_seqlens_k, no lists: causal is top-left (k <= q, local indices)."""
    c = synth.make_varlen(f"vl_lqlk_{mask_mod}_{D}", 4, 0, 0, 2, D, dtype, seed=560 + D,
                          lengths=[200, 70, 129, 1], lengths_k=[90, 300, 129, 5], block_lists="none",
                          mask_mod=mask_mod)
    check_varlen(c)


def test_varlen_key_lengths_differ_with_lists():
    """Lq != Lk with full / partial lists over the Lq x Lk block grid (causal on partial blocks)."""
    g = np.random.default_rng(7)
    lq, lk = [300, 140, 260], [180, 390, 260]
    c = synth.make_varlen("vl_lqlk_lists", 3, 0, 0, 2, 64, "bf16", seed=570, lengths=lq, lengths_k=lk,
                          block_lists="none")
    MQ, MK = 3, 4
    kn = torch.zeros(3, 1, MQ, dtype=torch.int32)
    ki = torch.full((3, 1, MQ, MK), 77, dtype=torch.int32)
    fn = torch.zeros(3, 1, MQ, dtype=torch.int32)
    fi = torch.full((3, 1, MQ, MK), 77, dtype=torch.int32)
    for s in range(3):
        nbq, nbk = (lq[s] + 127) // 128, (lk[s] + 127) // 128
        for qb in range(nbq):
            blocks = [int(x) for x in g.permutation(nbk)][:int(g.integers(1, nbk + 1))]
            nf = int(g.integers(0, len(blocks) + 1))
            fn[s, 0, qb] = nf
            fi[s, 0, qb, :nf] = torch.tensor(blocks[:nf], dtype=torch.int32)
            kn[s, 0, qb] = len(blocks) - nf
            ki[s, 0, qb, :len(blocks) - nf] = torch.tensor(blocks[nf:], dtype=torch.int32)
    c.kv_num_blocks, c.kv_indices, c.full_kv_num_blocks, c.full_kv_indices = kn, ki, fn, fi
    c.mask_mod = "causal"
    check_varlen(c)


@pytest.mark.parametrize("D", [64, 128])
def test_varlen_uneven_q_block_levels(D):
    """Key-split kernel's deal over (q block level, sequence, head): 60 sequences of 0..900
    tokens (levels that some sequences do not reach, empty sequences), an odd head count, and
    more items than two rounds of the grid, so the cursor skips whole levels and ends in the
    middle of (sequence, head) groups."""
    g = torch.Generator().manual_seed(12)
    lengths = torch.randint(0, 901, (60,), generator=g).tolist()
    lengths[3] = 0
    lengths[7] = 900
    c = synth.make_varlen(f"vl_levels_{D}", len(lengths), 0, 0, 3, D, "bf16", seed=585 + D, lengths=lengths)
    check_varlen(c)


def test_varlen_many_short_sequences():
    """More sequences than the key-split kernel's schedule keeps in shared memory (1024): the
    two-tile kernel runs them; lengths 0..40, causal lists."""
    g = torch.Generator().manual_seed(11)
    lengths = torch.randint(0, 41, (1100,), generator=g).tolist()
    c = synth.make_varlen("vl_many", len(lengths), 0, 0, 2, 32, "bf16", seed=580, lengths=lengths)
    check_varlen(c)


# The parameterised mask_mods (BlockMask page, mask_mod on partial blocks): on the
# key-split kernel (16-bit), the two-tile kernel (more than 1024 sequences) and the
# fp32 CUDA-core kernel.
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 64), ("f32", 32)])
@pytest.mark.parametrize("window", [1, 37, 200])
def test_varlen_sliding_window(dtype, D, window):
    c = synth.make_varlen(f"vl_sw{window}_{D}", 3, 0, 0, 2, D, dtype, seed=590 + window, lengths=[300, 1, 260],
                          block_lists="none", mask_mod="sliding_window")
    check_varlen(c, window=window)


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("f32", 16)])
@pytest.mark.parametrize("prefix", [0, 100, 300, [5, 0, 140, 1000]])
def test_varlen_prefix_lm(dtype, D, prefix):
    c = synth.make_varlen(f"vl_plm_{D}", 4, 0, 0, 2, D, dtype, seed=600 + D, lengths=[300, 129, 200, 64],
                          block_lists="none", mask_mod="prefix_lm")
    check_varlen(c, prefix=prefix)


def test_varlen_sliding_window_with_lists_and_many_sequences():
    """Causal block lists (earlier blocks full, the diagonal partial) with the window on the diagonal;
    and more than 1024 short sequences (the two-tile kernel)."""
    c = synth.make_varlen("vl_sw_lists", 3, 0, 0, 2, 64, "bf16", seed=610, lengths=[400, 260, 129],
                          mask_mod="sliding_window")
    check_varlen(c, window=50)
    g = torch.Generator().manual_seed(12)
    lengths = torch.randint(1, 41, (1030,), generator=g).tolist()
    c2 = synth.make_varlen("vl_sw_many", len(lengths), 0, 0, 1, 32, "bf16", seed=611, lengths=lengths,
                           block_lists="none", mask_mod="sliding_window")
    check_varlen(c2, window=7)
    c2.mask_mod = "prefix_lm"
    check_varlen(c2, prefix=[int(x) % 9 for x in range(1030)])


# Post-scale bias on the packed form (H, max_seqlen_q, max_seqlen_k), indexed by local
# positions: key-split kernel (16-bit, with bf16 / fp16 / fp32 bias) and the fp32 kernel.
@pytest.mark.parametrize("dtype,bias_dtype,D", [("bf16", "bf16", 64), ("bf16", "f32", 128), ("f16", "f16", 32),
                                                ("f16", "f32", 64), ("f32", "f32", 32)])
@pytest.mark.parametrize("lists", ["causal", "none"])
def test_varlen_bias(dtype, bias_dtype, D, lists):
    lengths = [300, 129, 64, 1]
    c = synth.make_varlen(f"vl_bias_{D}_{lists}", 4, 0, 0, 2, D, dtype, seed=620 + D, lengths=lengths,
                          block_lists=lists, mask_mod="causal")
    g = torch.Generator().manual_seed(621)
    bias = (2.0 * torch.randn(2, 304, 304, generator=g)).to(synth.TORCH_DTYPES[bias_dtype])
    c.max_seqlen = c.max_seqlen_k = 304  # the bias's (and the call's) max_seqlen
    check_varlen(c, bias=bias)


def test_varlen_bias_key_lengths_differ_and_window():
    """Lq != Lk with a bias (max_seqlen_q != max_seqlen_k) and the sliding window."""
    c = synth.make_varlen("vl_bias_lqlk", 3, 0, 0, 2, 64, "bf16", seed=630, lengths=[200, 70, 129],
                          lengths_k=[90, 300, 129], block_lists="none", mask_mod="sliding_window")
    g = torch.Generator().manual_seed(631)
    c.max_seqlen, c.max_seqlen_k = 208, 304
    bias = torch.randn(2, 208, 304, generator=g).to(torch.bfloat16)
    check_varlen(c, window=40, bias=bias)


def test_varlen_fp32():
    c = synth.make_varlen("vl_f32", 3, 0, 0, 2, 32, "f32", seed=520, lengths=[40, 200, 131])
    check_varlen(c)


def test_varlen_random_lists_and_unlisted_blocks():
    c = synth.make_varlen("vl_rand", 2, 0, 0, 2, 64, "bf16", seed=530, lengths=[400, 260])
    g = np.random.default_rng(1)
    S, MQ = 2, 4
    kn = torch.zeros(S, 1, MQ, dtype=torch.int32)
    ki = torch.full((S, 1, MQ, MQ), 77, dtype=torch.int32)
    fn = torch.zeros(S, 1, MQ, dtype=torch.int32)
    fi = torch.full((S, 1, MQ, MQ), 77, dtype=torch.int32)
    for s, L in enumerate([400, 260]):
        nb = (L + 127) // 128
        for qb in range(nb):
            if qb == 1:
                continue  # q block with no listed kv block: every logit -1e9 -> mean of V
            perm = g.permutation(nb).tolist()
            nf = int(g.integers(0, nb + 1))
            fn[s, 0, qb] = nf
            fi[s, 0, qb, :nf] = torch.tensor(perm[:nf], dtype=torch.int32)
            kn[s, 0, qb] = nb - nf
            ki[s, 0, qb, :nb - nf] = torch.tensor(perm[nf:], dtype=torch.int32)
    c.kv_num_blocks, c.kv_indices, c.full_kv_num_blocks, c.full_kv_indices = kn, ki, fn, fi
    check_varlen(c)


def test_varlen_per_head_masks():
    c = synth.make_varlen("vl_heads", 2, 0, 0, 2, 64, "bf16", seed=540, lengths=[256, 200])
    kn, ki, fn, fi = synth.causal_block_lists([256, 200], mask_heads=2)
    # head 1: only the diagonal blocks, no full blocks
    fn[:, 1] = 0
    c.kv_num_blocks, c.kv_indices, c.full_kv_num_blocks, c.full_kv_indices = kn, ki, fn, fi
    check_varlen(c)


def test_varlen_length_over_max_is_reported():
    import masked_attention_tri_gb300 as ta
    c = synth.make_varlen("vl_bad", 2, 0, 0, 1, 32, "bf16", seed=550, lengths=[64, 100], block_lists="none")
    cu = c.cu_seqlens.cuda()
    out = ta.varlen_attention(c.q.cuda(), c.k.cuda(), c.v.cuda(), cu, cu, 80, 80, mask_mod="causal")
    assert ta.get_status() == 5  # TA_ERR_DEVICE: a sequence longer than max_seqlen
    assert ta.get_status() == 0  # read-and-clear
    assert torch.isfinite(out[:64].float()).all()


# ---------------------------------------------------------------------------
# mask_to_kv_lengths, the page example flow, robustness
# ---------------------------------------------------------------------------

def test_mask_to_kv_lengths_matches_oracle():
    import masked_attention_tri_gb300 as ta
    g = torch.Generator().manual_seed(9)
    B, N, K = 2, 50, 200
    lens = torch.randint(0, K + 1, (B, N), generator=g)
    m = (torch.arange(K).view(1, 1, K) < lens.view(B, N, 1)).view(B, N, 1, 1, K)
    m[0, 3, 0, 0, 150] = True   # holey rows
    m[1, 7, 0, 0, K - 1] = True
    m[1, 8] = False
    m[1, 8, 0, 0, 40] = True
    kl, cnt = ta.mask_to_kv_lengths(m.cuda(), return_nonprefix=True)
    ref, prefix = oracle.mask_to_kv_lengths(m)
    assert torch.equal(kl.view(B, N).cpu(), ref)
    assert int(cnt.item()) == int((~prefix).sum())


def test_page_example_flow():
    """The triangle_attention page's Example: mask -> kv_lengths -> forward, and the dense-mask call."""
    import masked_attention_tri_gb300 as ta
    c = synth.fp16_page_example()
    mask = synth.page_example_kv_lengths(128, 96).cuda()
    kl = ta.mask_to_kv_lengths(mask)
    assert kl.shape == (1, 128, 1, 1, 1)
    assert kl.view(-1).tolist() == [96] * 96 + [0] * 32
    q, k, v, bias = (x.cuda() for x in (c.q, c.k, c.v, c.bias))
    out, lse, mx = ta.triangle_attention(q=q, k=k, v=v, bias=bias, scale=c.scale, return_aux=True, kv_lengths=kl)
    assert out.shape == (1, 128, 2, 128, 32) and out.dtype == torch.float16
    assert lse.dtype == torch.float32 and mx.dtype == torch.float32
    dense = (torch.rand(1, 128, 1, 1, 128, generator=torch.Generator().manual_seed(0)) < 0.5).cuda()
    o2 = ta.triangle_attention(q=q, k=k, v=v, bias=bias, mask=dense, scale=c.scale)
    rO, _, _ = oracle.tri_fwd(c.q, c.k, c.v, c.bias, mask=dense.cpu(), scale=c.scale)
    assert np.abs(o2.double().cpu().numpy() - rO).max() <= 2e-2
    # B=1 four-dimensional forms
    o4 = ta.triangle_attention(q[0], k[0], v[0], bias[0], scale=c.scale, kv_lengths=kl)
    assert torch.equal(o4, out[0])


def test_deterministic_and_guard_bands():
    import masked_attention_tri_gb300 as ta
    c = synth.make_triangle("guard", 1, 4, 2, 200, 264, 64, "bf16", "bf16", seed=600, mask="kvlen", kv_range=(0, 264))
    q, k, v, bias, kl = (x.cuda() for x in (c.q, c.k, c.v, c.bias, c.kv_lengths))
    n = q.numel()
    pad = 4096
    buf = torch.full((n + 2 * pad,), 12345.0, device="cuda", dtype=torch.bfloat16)
    out = buf[pad:pad + n].view(q.shape)
    ta.triangle_attention(q, k, v, bias, scale=c.scale, kv_lengths=kl, out=out)
    o1 = out.clone()
    ta.triangle_attention(q, k, v, bias, scale=c.scale, kv_lengths=kl, out=out)
    torch.cuda.synchronize()
    assert torch.equal(o1, out)
    assert (buf[:pad] == 12345.0).all() and (buf[pad + n:] == 12345.0).all()


def test_lse_only_outputs_optional():
    c = synth.make_triangle("noaux", 1, 2, 2, 64, 64, 32, "bf16", "bf16", seed=601)
    o = run_triangle(c, return_aux=False)
    O, L, M = run_triangle(c, return_aux=True)
    assert torch.equal(o, O)
