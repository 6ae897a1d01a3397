"""CPU-only checks of the C ABI: the library builds, loads, exports every
declared symbol, and its host-side argument checks return the documented
status codes without touching a GPU (none of these calls reaches CUDA)."""
import os
import re

import pytest

from masked_attention_tri_gb300 import abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*(tri_attn_[a-z0-9_]+)\s*\(", src,
                                flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert len(declared) >= 6
    for name in declared:
        assert hasattr(lib, name), name
    assert set(declared) == set(abi.EXPORTS)


def test_version_and_error_strings(lib):
    assert abi.tri_attn_version() >> 16 == 1
    for code, text in [(0, "ok"), (1, "invalid argument"), (2, "unsupported configuration"), (4, "timed out")]:
        assert text in abi.tri_attn_error_string(code)
    assert abi.tri_attn_error_string(99) == "unknown status"


# Fake, 16-byte aligned addresses: host checks never dereference them.
A = 0x10000
MIS = 0x10008


def _fwd(**kw):
    args = dict(q=A, k=A, v=A, qkv_dtype=abi.TA_BF16, bias=A, bias_dtype=abi.TA_BF16, mask=0, kv_lengths=0, B=1, N=2,
                H=2, Q=64, K=64, D=64, scale=0.125, out=A, lse=0, max_=0, stream=0)
    args.update(kw)
    return lambda: abi.tri_attn_fwd(**args)


@pytest.mark.parametrize("kw,exc", [
    (dict(q=0), ValueError),
    (dict(bias=0), ValueError),
    (dict(B=0), ValueError),
    (dict(K=-1), ValueError),
    (dict(mask=A, kv_lengths=A), ValueError),  # "pass either mask or kv_lengths, not both"
    (dict(q=MIS), ValueError),
    (dict(qkv_dtype=7), ValueError),
    (dict(bias_dtype=abi.TA_F16), NotImplementedError),  # bias must be fp32 or the q dtype
    (dict(D=264), NotImplementedError),  # D <= 256
    (dict(qkv_dtype=abi.TA_F32, bias_dtype=abi.TA_F32, D=260), NotImplementedError),
    (dict(D=12), NotImplementedError),  # 16-bit needs D % 8
    (dict(K=60), NotImplementedError),  # 16-bit needs K % 8
    (dict(qkv_dtype=abi.TA_F32, bias_dtype=abi.TA_F32, D=6), NotImplementedError),
    (dict(Q=1 << 19, K=1 << 19), NotImplementedError),  # a 2^40-byte bias plane: beyond a tensor-map stride
])
def test_triangle_host_checks(lib, kw, exc):
    with pytest.raises(exc):
        _fwd(**kw)()


def _bwd(**kw):
    ws = abi.tri_attn_bwd_workspace_size(1, 2, 2, 64, 64, 64)
    args = dict(q=A, k=A, v=A, qkv_dtype=abi.TA_BF16, bias=A, bias_dtype=abi.TA_BF16, mask=0, kv_lengths=0, B=1, N=2,
                H=2, Q=64, K=64, D=64, scale=0.125, lse=A, out=0, d_out=A, dq=A, dk=A, dv=A, dbias=A, workspace=A,
                workspace_bytes=ws, stream=0)
    args.update(kw)
    return lambda: abi.tri_attn_bwd(**args)


def test_bwd_workspace_size(lib):
    # fp32 dQ (B*N*H*Q*D), dBias (B*H*Q*K) and the per-row sums (B*N*H*Q), each rounded up to 64 floats
    up = lambda n: (n + 63) // 64 * 64
    assert abi.tri_attn_bwd_workspace_size(1, 2, 3, 70, 90, 40) == 4 * (up(6 * 70 * 40) + up(3 * 70 * 90) + up(6 * 70))
    assert abi.tri_attn_bwd_workspace_size(0, 2, 3, 70, 90, 40) == 0


@pytest.mark.parametrize("kw,exc", [
    (dict(q=0), ValueError),
    (dict(lse=0), ValueError),          # the forward's lse is required
    (dict(d_out=0), ValueError),
    (dict(dk=0), ValueError),
    (dict(workspace=0), ValueError),
    (dict(workspace=A + 16), ValueError),  # 256-byte aligned workspace
    (dict(workspace_bytes=1024), ValueError),  # below the required size
    (dict(dq=MIS), ValueError),
    (dict(out=MIS), ValueError),        # the forward's O, when given, 16-byte aligned
    (dict(mask=A, kv_lengths=A), ValueError),
    (dict(Q=0), ValueError),
    (dict(bias_dtype=abi.TA_F16), NotImplementedError),
    (dict(D=264), NotImplementedError),
    (dict(D=12), NotImplementedError),
])
def test_bwd_host_checks(lib, kw, exc):
    with pytest.raises(exc):
        _bwd(**kw)()


def _vbwd(**kw):
    ws = abi.tri_attn_varlen_bwd_workspace_size(100, 2, 64, 64, 64, False)
    args = dict(q=A, k=A, v=A, dtype=abi.TA_BF16, cu_seqlens_q=A, cu_seqlens_k=A, num_seqs=2, total_q=100,
                total_k=100, max_seqlen_q=64, max_seqlen_k=64, H=2, D=64, scale=0.125, kv_num_blocks=0,
                kv_indices=0, full_kv_num_blocks=0, full_kv_indices=0, mask_heads=1, max_q_blocks=1,
                max_kv_blocks=1, block_q=128, block_k=128, mask_mod=abi.TA_MASK_CAUSAL, window=0,
                prefix_lengths=0, prefix_length=0, bias=0, bias_dtype=abi.TA_F32, lse=A, out=A, d_out=A, dq=A,
                dk=A, dv=A, dbias=0, workspace=A, workspace_bytes=ws, stream=0)
    args.update(kw)
    return lambda: abi.tri_attn_varlen_bwd(**args)


def test_varlen_bwd_workspace_size(lib):
    up = lambda n: (n + 63) // 64 * 64
    assert abi.tri_attn_varlen_bwd_workspace_size(100, 2, 64, 64, 80, False) == 4 * (up(200 * 64) + up(200))
    assert abi.tri_attn_varlen_bwd_workspace_size(100, 2, 64, 64, 80, True) == 4 * (up(200 * 64) + up(2 * 64 * 80) +
                                                                                  up(200))


@pytest.mark.parametrize("kw,exc", [
    (dict(out=0), ValueError),           # the forward's O is required for the packed form
    (dict(lse=0), ValueError),
    (dict(dbias=A), ValueError),         # dBias without a bias
    (dict(workspace_bytes=64), ValueError),
    (dict(workspace=A + 64), ValueError),
    (dict(dq=MIS), ValueError),
    (dict(mask_mod=9), ValueError),
    (dict(mask_mod=abi.TA_MASK_SLIDING_WINDOW, window=0), ValueError),
    (dict(kv_num_blocks=A), ValueError),  # lists come in pairs
    (dict(block_q=64), NotImplementedError),
    (dict(D=264), NotImplementedError),
    (dict(bias=A, bias_dtype=abi.TA_F16), NotImplementedError),
])
def test_varlen_bwd_host_checks(lib, kw, exc):
    with pytest.raises(exc):
        _vbwd(**kw)()


def _fwd_strided(**kw):
    args = dict(q=A, k=A, v=A, qkv_dtype=abi.TA_BF16, bias=A, bias_dtype=abi.TA_BF16, mask=0, kv_lengths=0, B=1, N=2,
                H=2, Q=64, K=64, D=64, scale=0.125, q_strides=None, k_strides=None, v_strides=None, out=A, lse=0,
                max_=0, stream=0)
    args.update(kw)
    return lambda: abi.tri_attn_fwd_strided(**args)


@pytest.mark.parametrize("kw,exc", [
    (dict(q_strides=(8192, 4096, 64, 0)), ValueError),           # a stride below 1
    (dict(k_strides=(8192, 4096, 2048, 32)), ValueError),        # rows of 64 elements 32 apart overlap
    (dict(v_strides=(8192, 4096, 2048, 68)), NotImplementedError),  # 136-byte rows: not a 16-byte multiple
    (dict(q_strides=(1 << 40, 4096, 2048, 64)), NotImplementedError),
    (dict(q=MIS, q_strides=(8192, 4096, 2048, 64)), ValueError),
])
def test_triangle_strided_host_checks(lib, kw, exc):
    with pytest.raises(exc):
        _fwd_strided(**kw)()


def _varlen(**kw):
    args = dict(q=A, k=A, v=A, dtype=abi.TA_BF16, cu_seqlens_q=A, cu_seqlens_k=A, num_seqs=2, total_q=400, total_k=400, max_seqlen_q=256,
                max_seqlen_k=256, H=2, D=64, scale=0.125, kv_num_blocks=A, kv_indices=A, full_kv_num_blocks=A,
                full_kv_indices=A, mask_heads=1, max_q_blocks=2, max_kv_blocks=2, block_q=128, block_k=128,
                mask_mod=abi.TA_MASK_CAUSAL, out=A, lse=0, max_=0, stream=0)
    args.update(kw)
    return lambda: abi.tri_attn_varlen_fwd(**args)


@pytest.mark.parametrize("kw,exc", [
    (dict(cu_seqlens_q=0), ValueError),
    (dict(num_seqs=0), ValueError),
    (dict(total_k=-1), ValueError),
    (dict(full_kv_indices=0), ValueError),  # only one of the full_kv_* pair
    (dict(kv_indices=0), ValueError),
    (dict(kv_num_blocks=0, kv_indices=0), ValueError),  # full lists without partial lists
    (dict(mask_heads=3), ValueError),
    (dict(mask_mod=5), ValueError),
    (dict(block_q=64), NotImplementedError),
    (dict(D=264), NotImplementedError),  # D <= 256
])
def test_varlen_host_checks(lib, kw, exc):
    with pytest.raises(exc):
        _varlen(**kw)()


def test_varlen_empty_is_noop(lib):
    _varlen(max_seqlen_q=0)()


def _strided(**kw):
    args = dict(q=A, k=A, v=A, dtype=abi.TA_BF16, cu_seqlens_q=A, cu_seqlens_k=A, num_seqs=2, total_q=400,
                total_k=400, max_seqlen_q=256, max_seqlen_k=256, H=2, D=64, scale=0.125, kv_num_blocks=A,
                kv_indices=A, full_kv_num_blocks=A, full_kv_indices=A, mask_heads=1, max_q_blocks=2,
                max_kv_blocks=2, block_q=128, block_k=128, mask_mod=abi.TA_MASK_CAUSAL, q_row_stride=0,
                k_row_stride=0, v_row_stride=0, out=A, lse=0, max_=0, stream=0)
    args.update(kw)
    return lambda: abi.tri_attn_varlen_fwd_strided(**args)


@pytest.mark.parametrize("kw,exc", [
    (dict(q_row_stride=64), ValueError),                       # shorter than H*D = 128
    (dict(v_row_stride=-128), ValueError),
    (dict(k_row_stride=132), NotImplementedError),             # bf16 rows must be 16-byte multiples
    (dict(dtype=abi.TA_F32, q_row_stride=130), NotImplementedError),
    (dict(q_row_stride=1 << 41), NotImplementedError),
    (dict(k_row_stride=1 << 39), NotImplementedError),         # 2^40 bytes: beyond a tensor-map stride
    (dict(dtype=abi.TA_F32, v_row_stride=1 << 38), NotImplementedError),
])
def test_varlen_strided_host_checks(lib, kw, exc):
    with pytest.raises(exc):
        _strided(**kw)()


@pytest.mark.parametrize("strides", [(0, 0, 0), (384, 384, 384), (128, 256, 256), (136, 144, 128)])
def test_varlen_strided_accepts_packed_strides(lib, strides):
    # QKV_INTERLEAVED (3*H*D), KV_INTERLEAVED (q H*D, k/v 2*H*D) and padded rows pass
    # the host checks; with no query rows the call is a no-op before any device work.
    q, k, v = strides
    _strided(max_seqlen_q=0, q_row_stride=q, k_row_stride=k, v_row_stride=v)()


def _masked(**kw):
    args = dict(q=A, k=A, v=A, dtype=abi.TA_BF16, cu_seqlens_q=A, cu_seqlens_k=A, num_seqs=2, total_q=400,
                total_k=400, max_seqlen_q=256, max_seqlen_k=256, H=2, D=64, scale=0.125, kv_num_blocks=0,
                kv_indices=0, full_kv_num_blocks=0, full_kv_indices=0, mask_heads=1, max_q_blocks=2,
                max_kv_blocks=2, block_q=128, block_k=128, mask_mod=abi.TA_MASK_SLIDING_WINDOW, window=16,
                prefix_lengths=0, prefix_length=0, bias=0, bias_dtype=abi.TA_F32, q_row_stride=0, k_row_stride=0,
                v_row_stride=0, out=A, lse=0, max_=0, stream=0)
    args.update(kw)
    return lambda: abi.tri_attn_varlen_fwd_masked(**args)


@pytest.mark.parametrize("kw,exc", [
    (dict(window=0), ValueError),                                   # a window keeps at least the query itself
    (dict(window=-3), ValueError),
    (dict(mask_mod=4), ValueError),
    (dict(mask_mod=abi.TA_MASK_PREFIX_LM, prefix_length=-1), ValueError),
    (dict(mask_mod=abi.TA_MASK_PREFIX_LM, prefix_lengths=MIS + 2), ValueError),  # 4-byte alignment
    (dict(block_q=64), NotImplementedError),
    (dict(bias=MIS), ValueError),                                   # bias 16-byte alignment
    (dict(bias=A, bias_dtype=abi.TA_F16), NotImplementedError),     # bf16 q: bias f32 or bf16
    (dict(bias=A, bias_dtype=abi.TA_BF16, max_seqlen_k=250), NotImplementedError),  # 500-byte bias rows
    (dict(bias=A, bias_dtype=7), ValueError),
])
def test_varlen_masked_host_checks(lib, kw, exc):
    with pytest.raises(exc):
        _masked(**kw)()


def test_varlen_masked_accepts_parameters_and_older_entries_refuse_them(lib):
    _masked(max_seqlen_q=0)()                                              # window 16: accepted (no rows: no-op)
    _masked(max_seqlen_q=0, mask_mod=abi.TA_MASK_PREFIX_LM, prefix_lengths=A)()
    with pytest.raises(ValueError):  # the strided entry has no parameter for them
        _strided(max_seqlen_q=0, mask_mod=abi.TA_MASK_SLIDING_WINDOW)()
    with pytest.raises(ValueError):
        _varlen(max_seqlen_q=0, mask_mod=abi.TA_MASK_PREFIX_LM)()


def test_row_stride_of_packed_views():
    import torch
    from masked_attention_tri_gb300 import api
    cpu = torch.device("cpu")
    qkv = torch.zeros(10, 3, 2, 64)
    q, k, v = qkv.unbind(1)
    assert [api._row_stride(t, "x", cpu) for t in (q, k, v)] == [384, 384, 384]
    assert api._row_stride(torch.zeros(10, 2, 64), "x", cpu) == 128
    assert api._row_stride(torch.zeros(1, 2, 64)[:, :, :], "x", cpu) == 128
    with pytest.raises(ValueError):  # heads not contiguous
        api._row_stride(torch.zeros(10, 64, 2).transpose(1, 2), "x", cpu)
    with pytest.raises(ValueError):  # elements not contiguous
        api._row_stride(torch.zeros(10, 2, 128)[:, :, ::2], "x", cpu)
    with pytest.raises(ValueError, match="overlap"):  # an expanded view: row stride 0
        api._row_stride(torch.zeros(1, 2, 64).expand(10, 2, 64), "x", cpu)
    with pytest.raises(ValueError, match="overlap"):  # rows that overlap by half a row
        api._row_stride(torch.zeros(1000).as_strided((10, 2, 64), (64, 64, 1)), "x", cpu)


def test_preallocated_out_must_match_q():
    """A preallocated out of the wrong shape or dtype is rejected before any device work."""
    import torch
    from masked_attention_tri_gb300 import api
    q = torch.zeros(1, 2, 2, 16, 8, dtype=torch.bfloat16)
    bias = torch.zeros(1, 1, 2, 16, 16, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 2, 16, 8, dtype=torch.bfloat16)
    for bad in (torch.empty(1, 2, 2, 15, 8, dtype=torch.bfloat16), torch.empty(1, 2, 2, 16, 8, dtype=torch.float16),
                torch.empty(2 * 2 * 16 * 8, dtype=torch.bfloat16)):
        with pytest.raises(ValueError, match="out must be"):
            api.triangle_attention(q, k, k, bias, out=bad)
    qv = torch.zeros(40, 2, 8, dtype=torch.float32)
    cu = torch.tensor([0, 40], dtype=torch.int32)
    for bad in (torch.empty(39, 2, 8), torch.empty(40, 2, 8, dtype=torch.bfloat16)):
        with pytest.raises(ValueError, match="out must be"):
            api.varlen_attention(qv, qv, qv, cu, cu, 40, 40, out=bad)


def test_block_mask_dense_columns_follow_kv_blocks():
    """to_dense has one column per kv block, also when the lists are narrower than the block count."""
    import torch
    from masked_attention_tri_gb300 import api
    kn = torch.tensor([[[1, 2, 1]]], dtype=torch.int32)                    # (S=1, Hm=1, MQ=3)
    ki = torch.tensor([[[[0, 9], [1, 4], [3, 0]]]], dtype=torch.int32)    # MK = 2 < 5 kv blocks
    bm = api.BlockMask.from_kv_blocks(kn, ki, seq_lengths=(384, 640))
    d = bm.to_dense()
    assert d.shape == (1, 1, 3, 5)
    assert d[0, 0].tolist() == [[1, 0, 0, 0, 0], [0, 1, 0, 0, 1], [0, 0, 0, 1, 0]]
    assert bm.numel() == 15 and abs(bm.sparsity() - 100.0 * (1 - 4 / 15)) < 1e-9
    # without seq_lengths the columns reach the highest listed index
    assert api.BlockMask.from_kv_blocks(kn, ki).to_dense().shape == (1, 1, 3, 5)


def test_mask_to_kv_lengths_host_checks(lib):
    with pytest.raises(ValueError):
        abi.tri_attn_mask_to_kv_lengths(0, 1, 1, 8, A, 0, 0)
    with pytest.raises(ValueError):
        abi.tri_attn_mask_to_kv_lengths(A, 1, 0, 8, A, 0, 0)
