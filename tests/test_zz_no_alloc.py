"""The allocation-free W2A8 product entry point (vla_w2a8_ternary_gemm_noalloc).

It serves callers that cannot allocate device memory while they run (a
control loop with a hard period, or a process whose device memory is
reserved up front by another runtime).  Called through the C ABI, it must
give the same int32 accumulators and bf16 outputs, bit for bit, as the
allocating entry point vla_w2a8_ternary_gemm and as the oracle's Eq. (4)
product, on two calls in a row (the second reuses the shared scratch that the
first one filled); it must accept a product that fills its fixed scratch
exactly and refuse one larger than it, and refuse a misaligned code pointer
before launching anything; and a call must not take memory from the stream's
pool.  This file is collected last so that a run that stops at the first
failure has run everything else.
"""

import ctypes

import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.gpu

MAX_ELEMS = 1048576  # VLA_NOALLOC_MAX_ELEMS


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


def _call(fn, ta, tal, tq, beta, M, N, K, y, acc):
    import torch
    return fn(ctypes.c_void_p(ta.data_ptr()), ctypes.c_void_p(tal.data_ptr()), ctypes.c_void_p(tq.data_ptr()),
              beta, M, N, K, ctypes.c_void_p(y.data_ptr()), None if acc is None else ctypes.c_void_p(acc.data_ptr()),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_allocating_entry_point_and_oracle_twice():
    import torch
    import prefix_cached_flow_gb300 as V
    fn = _noalloc_fn()
    for seed, (M, N, K), beta in ((1, (16, 5632, 2048), 0.0171), (2, (8, 2048, 5632), 0.0093)):
        a, alpha, packed = _inputs(seed, M, N, K)
        ta, tal, tq = (torch.from_numpy(x).cuda() for x in (a, alpha, packed))
        y_ref, acc_ref = V.ternary_gemm(ta, tal, tq, beta)
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        acc = torch.full((M, N), -1, dtype=torch.int32, device="cuda")
        assert _call(fn, ta, tal, tq, beta, M, N, K, y, acc) == 0
        torch.cuda.synchronize()
        assert torch.equal(acc, acc_ref)
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
        yo, acco = O.ternary_linear(a, alpha, packed, np.float32(beta))
        assert np.array_equal(acc.cpu().numpy().astype(np.int64), acco)
        assert np.array_equal(y.view(torch.int16).cpu().numpy().astype(np.uint16),
                              (yo.view(np.uint32) >> 16).astype(np.uint16))


def test_noalloc_fills_its_scratch_exactly():
    """M * N equal to the scratch size is accepted and exact."""
    import torch
    fn = _noalloc_fn()
    M, N, K = 256, 4096, 64
    assert M * N == MAX_ELEMS
    a, alpha, packed = _inputs(3, M, N, K)
    ta, tal, tq = (torch.from_numpy(x).cuda() for x in (a, alpha, packed))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    assert _call(fn, ta, tal, tq, 0.5, M, N, K, y, acc) == 0
    torch.cuda.synchronize()
    yo, acco = O.ternary_linear(a, alpha, packed, np.float32(0.5))
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acco)
    assert np.array_equal(y.view(torch.int16).cpu().numpy().astype(np.uint16),
                          (yo.view(np.uint32) >> 16).astype(np.uint16))


def test_noalloc_takes_nothing_from_the_stream_pool():
    import torch
    fn = _noalloc_fn()
    M, N, K = 8, 2048, 2048
    a, alpha, packed = _inputs(4, M, N, K)
    ta, tal, tq = (torch.from_numpy(x).cuda() for x in (a, alpha, packed))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert _call(fn, ta, tal, tq, 1.0, M, N, K, y, None) == 0  # first call: looks up the scratch address
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _call(fn, ta, tal, tq, 1.0, M, N, K, y, None) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_refuses_before_launching():
    import torch
    fn = _noalloc_fn()
    # a product larger than the scratch: M * N = 1,049,600 > 1,048,576
    M, N, K = 1025, 1024, 64
    a = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    alpha = torch.ones(M, dtype=torch.float32, device="cuda")
    q = torch.full((N, K // 4), 0x55, dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert _call(fn, a, alpha, q, 1.0, M, N, K, y, None) == 3  # VLA_ERR_UNSUPPORTED
    # codes that start one byte into an allocation (the kernel reads 32-bit words)
    buf = torch.zeros(8 * K + 16, dtype=torch.int8, device="cuda")
    a_off = buf[1:1 + 8 * K].view(8, K)
    assert a_off.data_ptr() % 4 == 1
    y8 = torch.empty((8, N), dtype=torch.bfloat16, device="cuda")
    assert _call(fn, a_off, alpha, q, 1.0, 8, N, K, y8, None) == 1  # VLA_ERR_INVALID_ARG
    # N not a multiple of 4, as the allocating entry point
    assert _call(fn, a, alpha, q, 1.0, 8, 1022, K, y8, None) == 1
