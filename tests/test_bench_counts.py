"""The effective-FLOP counts behind bench.py's metric, recounted pair by pair on tiny cases.

`bench.triangle_work` and `bench.varlen_work` use closed forms (a clamp of kv_lengths, a mask
popcount, the causal / window triangle sums); here every (query, key) pair is visited and
kept or not by the definition of the mask, and each kept pair counts 4 D flops (QK^T and PV).
"""
import torch

import bench
import synth


def test_triangle_flops_count_valid_pairs():
    c = synth.make_triangle("cnt_kvlen", 2, 3, 2, 5, 7, 8, "bf16", "bf16", seed=1, mask="kvlen", kv_range=(0, 7))
    c.kv_lengths.view(-1)[:3] = torch.tensor([-2, 9, 0], dtype=torch.int32)  # clamps to 0 and K
    pairs = 0
    for b in range(c.B):
        for n in range(c.N):
            L = int(c.kv_lengths[b, n])
            for _h in range(c.H):
                for _q in range(c.Q):
                    pairs += sum(1 for k in range(c.K) if 0 <= k < L)
    assert bench.triangle_work(c)[0] == 4.0 * c.D * pairs

    d = synth.make_triangle("cnt_dense", 1, 4, 3, 6, 9, 16, "f16", "f32", seed=2, mask="dense")
    pairs = 0
    for n in range(d.N):
        for _h in range(d.H):
            for _q in range(d.Q):
                pairs += sum(1 for k in range(d.K) if d.mask[0, n, 0, 0, k] != 0)
    assert bench.triangle_work(d)[0] == 4.0 * d.D * pairs


def test_varlen_flops_count_kept_pairs():
    lengths = [1, 5, 13]
    for mod, window in (("causal", 0), ("sliding_window", 4), ("none", 0)):
        c = synth.make_varlen(f"cnt_{mod}", 3, 0, 0, 2, 32, "bf16", seed=3, lengths=lengths, block_lists="none",
                              mask_mod=mod)
        pairs = 0
        for L in lengths:
            for q in range(L):
                for k in range(L):
                    keep = {"causal": k <= q, "sliding_window": q - window < k <= q, "none": True}[mod]
                    pairs += keep
        assert bench.varlen_work(c, window=window)[0] == 4.0 * c.H * c.D * pairs, mod
