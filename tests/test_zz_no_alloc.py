"""tri_attn_bwd_noalloc: the backward in the library's static scratch, no allocation.

Collected last (file name).  The GPU tests compare two calls in a row with the
workspace entry point tri_attn_bwd on the same inputs; they run the same
kernels, so results differ only by the order of the fp32 atomic sums (tolerance
below).  Torch's allocator counter must not move across the two calls (the
outputs are allocated before).  Sizes beyond the scratch are refused before any
launch, which the CPU test checks.
"""
from __future__ import annotations

import pytest
import torch

import synth
from masked_attention_tri_gb300 import abi, build

# |a - b| <= atol * max|b| + rtol * |b|: fp32 outputs differ only by the atomic order;
# 16-bit outputs may also land on the other side of one rounding (one ulp, 2^-8 for bf16).
TOL = {"f32": (1e-5, 1e-5), "bf16": (1e-3, 2 ** -7), "f16": (1e-3, 2 ** -9)}


def _close(a, b, dtype, name):
    atol, rtol = TOL[dtype]
    a, b = a.float(), b.float()
    bound = atol * b.abs().max() + rtol * b.abs()
    err = (a - b).abs()
    assert bool((err <= bound).all()), f"{name}: max excess {float((err - bound).max()):.3e}"


def test_noalloc_refuses_problems_beyond_its_scratch():
    build.build()
    A = 0x10000
    # 32 slabs x 512 rows x D 256: the fp32 dQ accumulator alone is 16.8 MB, beyond the 16 MiB scratch
    need = abi.tri_attn_bwd_workspace_size(1, 8, 4, 512, 512, 256)
    assert need > abi.BWD_NOALLOC_SCRATCH_BYTES
    with pytest.raises(NotImplementedError):
        abi.tri_attn_bwd_noalloc(A, A, A, abi.TA_BF16, A, abi.TA_BF16, 0, 0, 1, 8, 4, 512, 512, 256, 0.0625, A, 0, A,
                                 A, A, A, A, 0)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,bias_dtype,mask", [("f32", "f32", "kvlen"), ("bf16", "bf16", "dense"),
                                                   ("f16", "f32", "none")])
def test_noalloc_matches_workspace_entry_twice(dtype, bias_dtype, mask):
    import masked_attention_tri_gb300 as ta
    from masked_attention_tri_gb300.api import _DT, _ptr
    c = synth.make_triangle(f"noalloc_{dtype}", 2, 3, 2, 50, 72, 64, dtype, bias_dtype, seed=800, mask=mask,
                            kv_range=(0, 72))
    dev = torch.device("cuda", 0)
    q, k, v, bias = (x.to(dev) for x in (c.q, c.k, c.v, c.bias))
    mask = None if c.mask is None else c.mask.to(dev)
    m8 = None if mask is None else mask.view(torch.uint8)
    kl = None if c.kv_lengths is None else c.kv_lengths.to(dev)
    d_out = synth.grad_out(c, 801).to(dev)
    o, lse, _ = ta.triangle_attention(q, k, v, bias, mask, c.scale, True, kv_lengths=kl)
    ref = ta.triangle_attention_backward(q, k, v, bias, lse, d_out, mask, c.scale, kv_lengths=kl, out=o)
    B, N, H, Q, D = q.shape
    K = k.shape[3]
    outs = [tuple(torch.empty_like(t) for t in (q, k, v, bias)) for _ in range(2)]
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    before = torch.cuda.memory_stats(dev).get("allocation.all.allocated", 0)
    for dq, dk, dv, db in outs:
        abi.tri_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(bias), _DT[bias.dtype], _ptr(m8),
                                 _ptr(kl), B, N, H, Q, K, D, c.scale, _ptr(lse), _ptr(o), _ptr(d_out), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(db), stream.cuda_stream)
    torch.cuda.synchronize(dev)
    assert torch.cuda.memory_stats(dev).get("allocation.all.allocated", 0) == before
    assert ta.get_status() == 0
    for i, got in enumerate(outs):
        for nm, g, r in zip(("dq", "dk", "dv", "dbias"), got, ref):
            _close(g, r, bias_dtype if nm == "dbias" else dtype, f"call {i + 1} {nm}")
