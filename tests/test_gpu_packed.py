"""GPU parity of the packed QKV / KV layouts of the varlen form.

Transformer Engine fused_attn.h, NVTE_QKV_Layout: NVTE_QKV_INTERLEAVED stores
q, k, v of a token side by side in one (total, 3, H, D) buffer and
NVTE_KV_INTERLEAVED k and v in one (total_k, 2, H, D) buffer.  The kernels read
them in place through row strides; the results must match the oracle on the
same values and equal, bit for bit, the run on separate contiguous tensors.
"""
import pytest
import torch

import oracle
import synth
from parity_helpers import compare, to_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from masked_attention_tri_gb300 import build
    build.build()


def _block_mask(ta, c):
    if c.kv_num_blocks is None:
        return None
    return ta.BlockMask.from_kv_blocks(to_gpu(c.kv_num_blocks), to_gpu(c.kv_indices), to_gpu(c.full_kv_num_blocks),
                                       to_gpu(c.full_kv_indices), BLOCK_SIZE=c.block, mask_mod=c.mask_mod)


def _reference(c):
    return oracle.varlen_fwd(c.q, c.k, c.v, c.cu_seqlens, c.cu_seqlens, c.scale, c.kv_num_blocks, c.kv_indices,
                             c.full_kv_num_blocks, c.full_kv_indices, block=c.block, mask_mod=c.mask_mod)


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("f16", 128), ("bf16", 32), ("f32", 32)])
@pytest.mark.parametrize("layout", ["qkv", "kv", "padded"])
def test_packed_layouts(dtype, D, layout):
    import masked_attention_tri_gb300 as ta
    c = synth.make_varlen(f"vl_{layout}_{dtype}_D{D}", 4, 0, 0, 3, D, dtype, seed=600 + D,
                          lengths=[1, 129, 300, 128])
    q, k, v = c.q.cuda(), c.k.cuda(), c.v.cuda()
    cu = c.cu_seqlens.cuda()
    bm = _block_mask(ta, c)
    base = ta.varlen_attention(q, k, v, cu, cu, c.max_seqlen, c.max_seqlen, block_mask=bm, scale=c.scale,
                               return_aux=True)
    if layout == "qkv":
        qkv = torch.stack([q, k, v], dim=1).contiguous()  # (total, 3, H, D)
        got = ta.varlen_attention_qkvpacked(qkv, cu, c.max_seqlen, block_mask=bm, scale=c.scale, return_aux=True)
    elif layout == "kv":
        kv = torch.stack([k, v], dim=1).contiguous()  # (total, 2, H, D)
        got = ta.varlen_attention_kvpacked(q, kv, cu, cu, c.max_seqlen, c.max_seqlen, block_mask=bm, scale=c.scale,
                                           return_aux=True)
    else:
        # rows padded to H*D + 16 elements (a 16-byte multiple for every dtype)
        total, H, _ = q.shape
        views = []
        for t in (q, k, v):
            buf = torch.full((total, H * D + 16), float("nan"), device=t.device, dtype=t.dtype)
            buf[:, :H * D] = t.reshape(total, H * D)
            views.append(buf[:, :H * D].view(total, H, D))
        assert views[0].stride(0) == H * D + 16
        got = ta.varlen_attention(*views, cu, cu, c.max_seqlen, c.max_seqlen, block_mask=bm, scale=c.scale,
                                  return_aux=True)
    torch.cuda.synchronize()
    assert ta.get_status() == 0
    for a, b in zip(got, base):
        assert torch.equal(a, b), "packed layout differs from the contiguous run"
    rO, rL, rM = _reference(c)
    compare(c.name, c.dtype, got[0], got[1], got[2], rO, rL, rM)


def test_bad_row_stride_is_rejected():
    import masked_attention_tri_gb300 as ta
    from masked_attention_tri_gb300 import abi
    c = synth.make_varlen("vl_bad_stride", 2, 0, 0, 2, 32, "bf16", seed=610, lengths=[64, 64])
    q, k, v = c.q.cuda(), c.k.cuda(), c.v.cuda()
    cu = c.cu_seqlens.cuda()
    out = torch.empty_like(q)
    H, D = q.shape[1], q.shape[2]
    common = (abi.TA_BF16, cu.data_ptr(), cu.data_ptr(), 2, q.shape[0], k.shape[0], 64, 64, H, D, c.scale,
              0, 0, 0, 0, 1, 0, 0, 128, 128, abi.TA_MASK_CAUSAL)
    with pytest.raises(ValueError):  # shorter than one row of heads
        abi.tri_attn_varlen_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), *common, H * D - 8, 0, 0,
                                        out.data_ptr(), 0, 0, torch.cuda.current_stream().cuda_stream)
    with pytest.raises(NotImplementedError):  # not a 16-byte multiple
        abi.tri_attn_varlen_fwd_strided(q.data_ptr(), k.data_ptr(), v.data_ptr(), *common, H * D + 4, 0, 0,
                                        out.data_ptr(), 0, 0, torch.cuda.current_stream().cuda_stream)
