"""The failure path of the bounded pipeline waits, on the GPU, without a fault or a hang.

A test build of the library (its own .so, built with -DTRIATTN_WAIT_LIMIT_CYCLES=2000000,
about 1 ms, and -DTRIATTN_TEST_MISSING_ARRIVAL) has one softmax warp of CTA 0 withhold
its first arrival on the P barrier.  The MMA warp's bounded wait for that barrier runs
out; the CTA raises its abort flag, every role leaves its loop through its own bounded
waits, the MMAs in flight drain and the tensor memory is released, and the kernel
records TA_ERR_TIMEOUT in the status word.  The test checks that status comes back
within a second, that it is cleared on read, and that the production library then
runs correctly on the same device.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from parity_helpers import check_triangle

pytestmark = pytest.mark.gpu

TA_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def timeout_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from masked_attention_tri_gb300 import build
    build.build()
    path = build.build_variant("timeout_test", ["TRIATTN_WAIT_LIMIT_CYCLES=2000000LL", "TRIATTN_TEST_MISSING_ARRIVAL"])
    lib = ctypes.CDLL(path)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.tri_attn_fwd.argtypes = [P, P, P, I, P, I, P, P, I, I, I, I, I, I, F, P, P, P, P]
    lib.tri_attn_fwd.restype = I
    lib.tri_attn_get_status.argtypes = [P]
    lib.tri_attn_get_status.restype = I
    return lib


def test_missing_arrival_reports_timeout_and_device_stays_usable(timeout_lib):
    c = synth.make_triangle("timeout", 1, 8, 2, 256, 256, 64, "bf16", "bf16", seed=700, mask="kvlen",
                            kv_range=(1, 256))
    q, k, v, bias, kl = (t.cuda() for t in (c.q, c.k, c.v, c.bias, c.kv_lengths))
    out = torch.empty_like(q)
    lse = torch.empty(c.B, c.N, c.H, c.Q, device="cuda", dtype=torch.float32)
    mx = torch.empty_like(lse)
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = timeout_lib.tri_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), 2, bias.data_ptr(), 2, None,
                                  kl.data_ptr(), c.B, c.N, c.H, c.Q, c.K, c.D, c.scale, out.data_ptr(),
                                  lse.data_ptr(), mx.data_ptr(), stream)
    assert st == 0  # the launch itself succeeds; the fault is found inside the kernel
    status = timeout_lib.tri_attn_get_status(stream)
    elapsed = time.perf_counter() - t0
    assert status == TA_ERR_TIMEOUT, status
    assert elapsed < 1.0, elapsed
    assert timeout_lib.tri_attn_get_status(stream) == 0  # read and cleared
    # The production library, same device and context, same inputs: correct and clean.
    check_triangle(c)
