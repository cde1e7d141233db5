"""The allocation-free W2A8 product entry point (vla_w2a8_ternary_gemm_noalloc).

It serves callers that cannot allocate device memory while they run (a
control loop with a hard period, or a process whose device memory is
reserved up front by another runtime).  Called through the C ABI, it must
give the same int32 accumulators and bf16 outputs, bit for bit, as the
allocating entry point vla_w2a8_ternary_gemm, on two calls in a row (the
second reuses the shared scratch that the first one filled), and it must
refuse a product larger than its fixed scratch.  This file is collected
last so that a run that stops at the first failure has run everything else.
"""

import ctypes

import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import prefix_cached_flow_gb300 as V
    fn = V.lib().vla_w2a8_ternary_gemm_noalloc
    vp, ci = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, ctypes.c_float, ci, ci, ci, vp, vp, vp]
    fn.restype = ci
    return fn


def _inputs(seed, M, N, K):
    rng = np.random.default_rng(seed)
    a = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    packed = O.pack_ternary(rng.integers(-1, 2, size=(N, K)).astype(np.int8))
    alpha = rng.uniform(1e-4, 1.0, M).astype(np.float32)
    return a, alpha, packed


def test_noalloc_matches_allocating_entry_point_twice():
    import torch
    import prefix_cached_flow_gb300 as V
    fn = _noalloc_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed, (M, N, K), beta in ((1, (16, 5632, 2048), 0.0171), (2, (8, 2048, 5632), 0.0093)):
        a, alpha, packed = _inputs(seed, M, N, K)
        ta, tal, tq = (torch.from_numpy(x).cuda() for x in (a, alpha, packed))
        y_ref, acc_ref = V.ternary_gemm(ta, tal, tq, beta)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        acc = torch.full((M, N), -1, dtype=torch.int32, device="cuda")
        st = fn(ctypes.c_void_p(ta.data_ptr()), ctypes.c_void_p(tal.data_ptr()), ctypes.c_void_p(tq.data_ptr()),
                beta, M, N, K, ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(acc.data_ptr()), stream)
        assert st == 0
        torch.cuda.synchronize()
        assert torch.equal(acc, acc_ref)
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_noalloc_rejects_products_beyond_its_scratch():
    import torch
    fn = _noalloc_fn()
    M, N, K = 1025, 1024, 64  # M * N = 1,049,600 > 1,048,576
    a = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    alpha = torch.ones(M, dtype=torch.float32, device="cuda")
    q = torch.full((N, K // 4), 0x55, dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = fn(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(alpha.data_ptr()), ctypes.c_void_p(q.data_ptr()),
            1.0, M, N, K, ctypes.c_void_p(y.data_ptr()), None,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3  # VLA_ERR_UNSUPPORTED
