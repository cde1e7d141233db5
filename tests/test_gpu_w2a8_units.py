"""Bit-exact unit parity of the W2A8 kernels ("vla.cpp: A Unified Inference
Runtime for Vision-Language-Action Models", §III-D Eq. (4)): the int8 codes,
the fp32 row scales, the int32 accumulators and the bf16 outputs must equal
the oracle's bit for bit on identical fp32 / int8 inputs."""

import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.gpu


def _rows(rng, M, K):
    x = rng.standard_normal((M, K)).astype(np.float32) * rng.uniform(1e-3, 1e3, (M, 1)).astype(np.float32)
    x[0] = 0.0                                # all-zero row: alpha is the 1e-5 floor
    x[1, :] = rng.integers(-254, 255, K) / np.float32(2)   # halves with absmax 127 -> alpha = 1, ties
    x[1, 0] = 127.0
    x[2, :] = 1e-7                           # below the floor
    return x


@pytest.mark.parametrize("K", [64, 2048, 5632])
def test_quantize_rows_bit_exact(K):
    import torch
    import prefix_cached_flow_gb300 as V
    rng = np.random.default_rng(K)
    x = _rows(rng, 37, K)
    a, alpha = V.quantize_rows(torch.from_numpy(x).cuda())
    a_ref, alpha_ref = O.quantize_rows(x)
    assert np.array_equal(alpha.cpu().numpy().view(np.uint32), alpha_ref.view(np.uint32))
    assert np.array_equal(a.cpu().numpy(), a_ref)


@pytest.mark.parametrize("M,N,K", [(8, 2048, 2048), (16, 512, 5632), (3, 200, 64)])
def test_ternary_gemm_bit_exact(M, N, K):
    import torch
    import prefix_cached_flow_gb300 as V
    rng = np.random.default_rng(M * N + K)
    a = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    packed = O.pack_ternary(q)
    alpha = rng.uniform(1e-4, 1.0, M).astype(np.float32)
    beta = np.float32(0.0123)
    y, acc = V.ternary_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(alpha).cuda(),
                            torch.from_numpy(packed).cuda(), float(beta))
    y_ref, acc_ref = O.ternary_linear(a, alpha, packed, beta)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_ref)
    y_bits = y.view(torch.int16).cpu().numpy().astype(np.uint16)
    ref_bits = (y_ref.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(y_bits, ref_bits)


def test_ternary_gemm_extreme_accumulator():
    """|acc| = 127 * 5632, the largest the full-size W2A8 shapes reach."""
    import torch
    import prefix_cached_flow_gb300 as V
    K = 5632
    a = np.full((2, K), 127, np.int8)
    a[1] = -127
    packed = O.pack_ternary(np.ones((128, K), np.int8))
    alpha = np.ones(2, np.float32)
    y, acc = V.ternary_gemm(torch.from_numpy(a).cuda(), torch.from_numpy(alpha).cuda(),
                            torch.from_numpy(packed).cuda(), 1.0)
    acc = acc.cpu().numpy()
    assert np.all(acc[0] == 127 * K) and np.all(acc[1] == -127 * K)


def test_gelu_forms_within_bound():
    """The many-token epilogue's GeLU (erf by Abramowitz & Stegun 7.1.26,
    |erf error| <= 1.5e-7, approximate reciprocal and exponential) against
    the erff form and the fp64 definition: |error| <= 4e-7 (1 + |x|)."""
    import torch
    import prefix_cached_flow_gb300 as V
    x = np.concatenate([np.linspace(-12, 12, 200001), np.random.default_rng(5).standard_normal(100000) * 3])
    x = x.astype(np.float32)
    exact, fast = V.gelu_forms(torch.from_numpy(x).cuda())
    exact, fast = exact.cpu().numpy().astype(np.float64), fast.cpu().numpy().astype(np.float64)
    ref = O.gelu(x.astype(np.float64))
    bound = 4e-7 * (1 + np.abs(x))
    assert np.all(np.abs(fast - ref) <= bound)
    assert np.all(np.abs(exact - ref) <= 2e-7 * (1 + np.abs(x)))
