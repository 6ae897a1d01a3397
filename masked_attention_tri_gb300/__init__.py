"""GB300-native (sm_103a) forward of masked, biased triangle attention.

O[b,n,h,q,:] = sum_k softmax_k(s * Q.K + bias[b,h,q,k], or -1e9 where the key
is masked) V[b,n,h,k,:], with the per-row logsumexp and max, as defined on the
cuEquivariance triangle_attention API page; plus a packed-sequence form with a
block-sparse (BlockMask) mask, and the backward of the triangle form.  The work runs in libtriattn.so (hand-written
CUDA, tcgen05 / TMA); this package only marshals tensors into its C ABI.
"""
from . import abi
from .api import (BlockMask, get_status, mask_to_kv_lengths, triangle_attention, triangle_attention_autograd,
                  triangle_attention_backward, varlen_attention, varlen_attention_backward,
                  varlen_attention_kvpacked, varlen_attention_qkvpacked)

__all__ = ["abi", "BlockMask", "get_status", "mask_to_kv_lengths", "triangle_attention", "triangle_attention_autograd",
           "triangle_attention_backward", "varlen_attention", "varlen_attention_backward", "varlen_attention_kvpacked",
           "varlen_attention_qkvpacked"]
