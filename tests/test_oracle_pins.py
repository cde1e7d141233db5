"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test names what fixes the expected value: a closed form, an invariant of
the method, brute force on tiny inputs, or a library routine (torch fp64).
Sources: "vla.cpp: A Unified Inference Runtime for Vision-Language-Action
Models", §III-A Eq. (1), §III-B Eq. (2)-(3), §III-D Eq. (4), §III-E Eq. (5).
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as tF

import oracle as O
from workloads import ExpertConfig, make_observations, make_weights

PIN = ExpertConfig("pin", L=2, D=32, F=48, n_q=4, n_kv=2, d_h=8, d_vlm=24, P=10, H=5,
                   d_a=3, S=3, B=2, d_t=16, seed=11, dtype="f32")


def _setup(cfg=PIN, zero=()):
    w = make_weights(cfg, zero=zero)
    Z, noise = make_observations(cfg)
    return w, Z.astype(np.float64), noise.astype(np.float64)


# ---------------------------------------------------------------- attention

def _rand_attn(rng, B=2, H=3, n_q=4, n_kv=2, d_h=5, P=6):
    q = rng.standard_normal((B, H, n_q, d_h))
    ks = rng.standard_normal((B, H, n_kv, d_h))
    vs = rng.standard_normal((B, H, n_kv, d_h))
    Kc = rng.standard_normal((B, n_kv, P, d_h))
    Vc = rng.standard_normal((B, n_kv, P, d_h))
    return q, ks, vs, Kc, Vc


def test_attention_vs_bruteforce_softmax():
    """Two-pass max-shifted softmax == direct exp / sum(exp) with exact sums (Eq. 2)."""
    rng = np.random.default_rng(0)
    q, ks, vs, Kc, Vc = _rand_attn(rng)
    o = O.joint_attention(q, ks, vs, Kc, Vc)
    B, H, n_q, d_h = q.shape
    n_kv = ks.shape[2]
    P = Kc.shape[2]
    for b in range(B):
        for t in range(H):
            for j in range(n_q):
                g = j * n_kv // n_q
                keys = [Kc[b, g, p] for p in range(P)] + [ks[b, s, g] for s in range(H)]
                vals = [Vc[b, g, p] for p in range(P)] + [vs[b, s, g] for s in range(H)]
                wts = [math.exp(math.fsum(q[b, t, j, d] * k[d] for d in range(d_h)) / math.sqrt(d_h))
                       for k in keys]
                den = math.fsum(wts)
                for d in range(d_h):
                    num = math.fsum(wi * v[d] for wi, v in zip(wts, vals))
                    assert abs(o[b, t, j, d] - num / den) <= 1e-12 * max(1.0, abs(num / den))


def test_attention_vs_library_sdpa_gqa_and_mask():
    """Grouped joint attention == torch scaled_dot_product_attention(enable_gqa) in fp64."""
    rng = np.random.default_rng(1)
    q, ks, vs, Kc, Vc = _rand_attn(rng, B=2, H=4, n_q=6, n_kv=3, d_h=7, P=9)
    vis = rng.random((2, 9)) > 0.3
    o = O.joint_attention(q, ks, vs, Kc, Vc, prefix_visible=vis)
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)
    tk = torch.cat([torch.from_numpy(Kc), torch.from_numpy(ks).permute(0, 2, 1, 3)], dim=2)
    tv = torch.cat([torch.from_numpy(Vc), torch.from_numpy(vs).permute(0, 2, 1, 3)], dim=2)
    mask = torch.cat([torch.from_numpy(vis), torch.ones(2, 4, dtype=torch.bool)], dim=1)[:, None, None, :]
    ref = tF.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, enable_gqa=True)
    np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-13)


def test_attention_single_visible_key_returns_its_value():
    """All prefix keys masked (M = -inf) and one action token: output = that token's V."""
    rng = np.random.default_rng(2)
    q, ks, vs, Kc, Vc = _rand_attn(rng, B=1, H=1, n_q=4, n_kv=2, d_h=5, P=6)
    o = O.joint_attention(q, ks, vs, Kc, Vc, prefix_visible=np.zeros((1, 6), bool))
    for j in range(4):
        np.testing.assert_array_equal(o[0, 0, j], vs[0, 0, j // 2])


def test_attention_zero_query_is_mean_of_all_values():
    """q = 0 gives uniform weights over P prefix + H suffix keys (catches a dropped suffix)."""
    rng = np.random.default_rng(3)
    q, ks, vs, Kc, Vc = _rand_attn(rng, B=1, H=3, n_q=2, n_kv=1, d_h=4, P=5)
    o = O.joint_attention(np.zeros_like(q), ks, vs, Kc, Vc)
    mean = (Vc[0, 0].sum(0) + vs[0, :, 0].sum(0)) / 8.0
    np.testing.assert_allclose(o[0, 1, 1], mean, rtol=0, atol=1e-15)


# ---------------------------------------------------------- building blocks

def test_elementwise_vs_library():
    x = np.linspace(-6, 6, 1001)
    t = torch.from_numpy(x)
    np.testing.assert_allclose(O.gelu(x), tF.gelu(t, approximate="none").numpy(), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(O.silu(x), tF.silu(t).numpy(), rtol=1e-14, atol=1e-15)
    rng = np.random.default_rng(4)
    h = rng.standard_normal((3, 5, 16))
    g = rng.standard_normal(16) * 0.1
    b = rng.standard_normal(16) * 0.1
    ref = tF.rms_norm(torch.from_numpy(h), (16,), eps=1e-6).numpy() * (1 + g) + b
    np.testing.assert_allclose(O.rmsnorm_modulate(h, g, b, 1e-6), ref, rtol=1e-13, atol=1e-14)


def test_time_embedding_special_values():
    d_t = 16
    e0 = O.sinusoidal_time_embedding(0.0, d_t)
    np.testing.assert_array_equal(e0, np.r_[np.zeros(8), np.ones(8)])
    for tau in (0.1, 0.37, 1.0):
        e = O.sinusoidal_time_embedding(tau, d_t)
        np.testing.assert_allclose(e[:8] ** 2 + e[8:] ** 2, 1.0, atol=1e-14)
    # lowest index has unit angular rate: sin(1000 tau) = 1 at tau = pi / 2000
    assert abs(O.sinusoidal_time_embedding(math.pi / 2000, d_t)[0] - 1.0) < 1e-15
    # the rate of index i is 10000^(-i/8): zero of the cos half at 1000 tau w_i = pi/2
    i = 5
    tau = (math.pi / 2) / (1000 * 10000 ** (-i / 8))
    assert abs(O.sinusoidal_time_embedding(tau, d_t)[8 + i]) < 1e-12


def test_prefix_kv_layout_vs_library_linear():
    """K_C = Z W_K per layer and head, laid out [L, B, n_kv, P, d_h] (Eq. 2)."""
    w, Z, _ = _setup()
    K, V = O.prefix_kv(Z, w, PIN)
    for l in range(PIN.L):
        for name, C in (("wk_pre", K), ("wv_pre", V)):
            ref = tF.linear(torch.from_numpy(Z), torch.from_numpy(w[name][l].astype(np.float64)))
            ref = ref.view(PIN.B, PIN.P, PIN.n_kv, PIN.d_h).permute(0, 2, 1, 3).numpy()
            np.testing.assert_allclose(C[l], ref, rtol=0, atol=1e-13)


def _torch_velocity(x, tau, Kc, Vc, w, cfg):
    """The velocity network expressed with torch library routines (fp64)."""
    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    e = T(O.sinusoidal_time_embedding(tau, cfg.d_t))
    sc = tF.silu(tF.linear(tF.silu(tF.linear(e, T(w["wt1"]))), T(w["wt2"])))
    h = tF.linear(T(x), T(w["win"]))
    B, H, _ = x.shape
    for l in range(cfg.L):
        ga, ba, gm, bm = tF.linear(sc, T(w["wmod"][l])).view(4, cfg.D)
        u = tF.rms_norm(h, (cfg.D,), eps=cfg.eps) * (1 + ga) + ba
        q = tF.linear(u, T(w["wq"][l])).view(B, H, cfg.n_q, cfg.d_h).transpose(1, 2)
        k = tF.linear(u, T(w["wk"][l])).view(B, H, cfg.n_kv, cfg.d_h).transpose(1, 2)
        v = tF.linear(u, T(w["wv"][l])).view(B, H, cfg.n_kv, cfg.d_h).transpose(1, 2)
        k = torch.cat([T(Kc[l]), k], dim=2)
        v = torch.cat([T(Vc[l]), v], dim=2)
        o = tF.scaled_dot_product_attention(q, k, v, enable_gqa=True).transpose(1, 2).reshape(B, H, -1)
        h = h + tF.linear(o, T(w["wo"][l]))
        u = tF.rms_norm(h, (cfg.D,), eps=cfg.eps) * (1 + gm) + bm
        h = h + tF.linear(tF.gelu(tF.linear(u, T(w["wup"][l]))), T(w["wdown"][l]))
    gf, bf = tF.linear(sc, T(w["wmod_f"])).view(2, cfg.D)
    return tF.linear(tF.rms_norm(h, (cfg.D,), eps=cfg.eps) * (1 + gf) + bf, T(w["wout"])).numpy()


def test_velocity_vs_library_routines():
    w, Z, noise = _setup()
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    for tau in (0.0, 1.0 / 3.0):
        v = O.velocity(noise, tau, Kc, Vc, w, PIN)
        np.testing.assert_allclose(v, _torch_velocity(noise, tau, Kc, Vc, w, PIN), rtol=0, atol=1e-12)


# ---------------------------------------------------------- solver / cache

def test_cache_reuse_equals_recompute_bitwise():
    """Reusing K_C, V_C across solver steps == recomputing them every step (§III-B)."""
    w, Z, noise = _setup()
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    x1, v1 = O.denoise(noise, Kc, Vc, w, PIN)
    x2, v2 = O.denoise_recompute(noise, Z, w, PIN)
    assert np.array_equal(x1, x2) and np.array_equal(v1, v2)


def test_prefix_permutation_invariance():
    """Bidirectional, position-free prefix: permuting Z's tokens changes nothing."""
    w, Z, noise = _setup()
    perm = np.random.default_rng(5).permutation(PIN.P)
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    Kp, Vp = O.prefix_kv(Z[:, perm], w, PIN)
    x1, v1 = O.denoise(noise, Kc, Vc, w, PIN)
    x2, v2 = O.denoise(noise, Kp, Vp, w, PIN)
    np.testing.assert_allclose(v2, v1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(x2, x1, rtol=0, atol=1e-12)


def test_suffix_permutation_equivariance():
    w, Z, noise = _setup()
    perm = np.random.default_rng(6).permutation(PIN.H)
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    x1, _ = O.denoise(noise, Kc, Vc, w, PIN)
    x2, _ = O.denoise(noise[:, perm], Kc, Vc, w, PIN)
    np.testing.assert_allclose(x2, x1[:, perm], rtol=0, atol=1e-12)


def test_batch_independence():
    w, Z, noise = _setup()
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    xb, _ = O.denoise(noise, Kc, Vc, w, PIN)
    for b in range(PIN.B):
        x1, _ = O.denoise(noise[b:b + 1], Kc[:, b:b + 1], Vc[:, b:b + 1], w, PIN)
        np.testing.assert_allclose(x1[0], xb[b], rtol=0, atol=1e-12)


def test_zero_velocity_head_returns_noise_bitwise():
    w, Z, noise = _setup(zero=("wout",))
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    x, vs = O.denoise(noise, Kc, Vc, w, PIN)
    assert np.array_equal(x, noise) and not np.any(vs)


def test_constant_velocity_field_closed_form():
    """W_in = 0 and a zero time MLP make v independent of x and tau, so Euler
    gives X^S = X^0 + (tau_S - tau_0) v_0 exactly up to rounding (Eq. 1).
    With h = 0 the first layer's attention has q = k_s = v_s = 0, so its
    output is the mean of the prefix values over P + H keys."""
    w, Z, noise = _setup(zero=("win", "wt1", "wt2"))
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    x, vs = O.denoise(noise, Kc, Vc, w, PIN)
    for k in range(1, PIN.S):
        assert np.array_equal(vs[k], vs[0])
    np.testing.assert_allclose(x, noise + 1.0 * vs[0], rtol=0, atol=1e-12)
    taps = {}
    O.velocity(noise, 0.0, Kc, Vc, w, PIN, taps=taps)
    o = taps["attn"][0].reshape(PIN.B, PIN.H, PIN.n_q, PIN.d_h)
    for j in range(PIN.n_q):
        g = j * PIN.n_kv // PIN.n_q
        mean = Vc[0][:, g].sum(axis=1) / (PIN.P + PIN.H)
        np.testing.assert_allclose(o[:, 2, j], mean, rtol=0, atol=1e-14)


def test_single_step():
    w, Z, noise = _setup()
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    x, vs = O.denoise(noise, Kc, Vc, w, PIN, S=1)
    v = O.velocity(noise, 0.0, Kc, Vc, w, PIN)
    assert np.array_equal(vs[0], v)
    np.testing.assert_allclose(x, noise + v, rtol=0, atol=1e-15)


def test_schedule_spans_unit_interval():
    for S in (1, 4, 8, 10):
        tau = O.schedule(S)
        assert tau[0] == 0.0 and tau[-1] == 1.0 and np.all(np.diff(tau) > 0)


def test_gqa_equals_replicated_mha():
    """n_kv < n_q with contiguous groups == n_kv = n_q with each K/V head copied."""
    w, Z, noise = _setup()
    mha = PIN.replace(n_kv=PIN.n_q)
    rep = PIN.n_q // PIN.n_kv
    w2 = dict(w)
    for name in ("wk_pre", "wv_pre", "wk", "wv"):
        a = w[name].reshape(PIN.L, PIN.n_kv, PIN.d_h, -1)
        w2[name] = np.repeat(a, rep, axis=1).reshape(PIN.L, mha.n_kv * PIN.d_h, -1)
    K1, V1 = O.prefix_kv(Z, w, PIN)
    K2, V2 = O.prefix_kv(Z, w2, mha)
    x1, v1 = O.denoise(noise, K1, V1, w, PIN)
    x2, v2 = O.denoise(noise, K2, V2, w2, mha)
    np.testing.assert_allclose(v2, v1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(x2, x1, rtol=0, atol=1e-12)


# ---------------------------------------------------------- Eq. (4) W2A8

def test_quantizer_worked_ties():
    """Row with absmax exactly 127 -> alpha = 1 exactly, so codes are
    round-half-even of the values themselves (Eq. 4, nearest-even ties)."""
    x = np.array([[2.5, 3.5, -2.5, -0.5, 126.5, 127.0, -1.5, 0.49999997]], np.float32)
    a, alpha = O.quantize_rows(x)
    assert alpha.dtype == np.float32 and alpha[0] == np.float32(1.0)
    assert a.tolist() == [[2, 4, -2, 0, 126, 127, -2, 0]]


def test_quantizer_zero_row_and_floor():
    x = np.zeros((2, 8), np.float32)
    x[1, 3] = 1e-7  # absmax below the 1e-5 floor: alpha is the floor
    x[1, 4] = -3e-8
    a, alpha = O.quantize_rows(x)
    assert np.all(alpha == np.float32(np.float32(1e-5) / np.float32(127)))
    assert not np.any(a[0])
    # 1e-7 / (1e-5/127) = 1.27 -> 1 ; -3e-8 / (1e-5/127) = -0.381 -> 0
    assert a[1].tolist() == [0, 0, 0, 1, 0, 0, 0, 0]


def test_quantizer_error_bound_and_range():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 333)) * rng.uniform(1e-3, 1e3, (64, 1))).astype(np.float32)
    a, alpha = O.quantize_rows(x)
    assert a.min() >= -127 and a.max() <= 127
    assert np.all(np.abs(a).max(axis=1) == 127)  # the absmax element maps to +-127
    err = np.abs(x.astype(np.float64) - alpha[:, None].astype(np.float64) * a)
    assert np.all(err <= alpha[:, None] * (0.5 + 1e-6))


def test_bf16_rounding_vs_library_conversion():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0, -0.0], np.float32)
    x = np.concatenate([x, ties])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(O.bf16_rne(x).view(np.uint32), ref.view(np.uint32))


def test_pack_unpack_roundtrip_and_invalid_code():
    rng = np.random.default_rng(9)
    q = rng.integers(-1, 2, size=(5, 16)).astype(np.int8)
    assert np.array_equal(O.unpack_ternary(O.pack_ternary(q)), q)
    # code layout: q = +1 at j = 1 only -> code 2 at bits 2..3, the rest code 1
    q1 = np.zeros((1, 4), np.int8)
    q1[0, 1] = 1
    assert O.pack_ternary(q1)[0, 0] == 0b01011001
    with pytest.raises(ValueError):
        O.unpack_ternary(np.array([[0xFF]], np.uint8))


def test_ternary_linear_vs_int_bruteforce():
    rng = np.random.default_rng(10)
    M, N, K = 3, 5, 12
    a = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    alpha = rng.uniform(0.01, 1, M).astype(np.float32)
    beta = np.float32(0.37)
    y, acc = O.ternary_linear(a, alpha, O.pack_ternary(q), beta)
    for m in range(M):
        for n in range(N):
            s = sum(int(a[m, j]) * int(q[n, j]) for j in range(K))
            assert acc[m, n] == s
            y32 = np.float32(np.float32(np.float32(s) * alpha[m]) * beta)
            ref = torch.tensor(float(y32), dtype=torch.float32).to(torch.bfloat16).float().item()
            assert y[m, n] == np.float32(ref)


def test_ternary_linear_special_weights():
    rng = np.random.default_rng(11)
    a = rng.integers(-127, 128, size=(4, 64)).astype(np.int8)
    alpha = np.ones(4, np.float32)
    ones = O.pack_ternary(np.ones((3, 64), np.int8))
    _, acc = O.ternary_linear(a, alpha, ones, np.float32(1))
    assert np.array_equal(acc, np.repeat(a.astype(np.int64).sum(1, keepdims=True), 3, axis=1))
    y, acc = O.ternary_linear(a, alpha, O.pack_ternary(np.zeros((3, 64), np.int8)), np.float32(1))
    assert not np.any(acc) and not np.any(y)


def test_ternary_linear_extreme_accumulator_exact():
    """Largest |acc| for K = 5632: 127 * 5632 < 2^24, still exact through fp32."""
    K = 5632
    a = np.full((2, K), 127, np.int8)
    a[1] = -127
    q = np.ones((1, K), np.int8)
    y, acc = O.ternary_linear(a, np.ones(2, np.float32), O.pack_ternary(q), np.float32(1))
    assert acc[0, 0] == 127 * K and acc[1, 0] == -127 * K


def test_w2a8_zero_ternary_weights_leave_residual_stream():
    """All six ternary maps zero: every layer adds 0, so v = head(x W_in)."""
    cfg = PIN.replace(w2a8=True, dtype="bf16", D=32, F=48)
    w = make_weights(cfg, zero=("wq", "wk", "wv", "wo", "wup", "wdown"))
    Z, noise = make_observations(cfg)
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    v = O.velocity_w2a8(noise, 0.25, Kc, Vc, w, cfg)
    _, final = O.time_conditioning(w, cfg, 0.25)
    h = O.linear(noise, w["win"])
    ref = O.linear(O.rmsnorm_modulate(h, final[0], final[1], cfg.eps), w["wout"])
    np.testing.assert_allclose(v, ref, rtol=0, atol=1e-13)


def _torch_unpack_ternary(packed):
    """2-bit fields (code q+1, little-endian in the byte) -> int64 q, in torch."""
    p = torch.from_numpy(np.asarray(packed)).to(torch.int64)
    f = torch.stack([(p >> (2 * i)) & 3 for i in range(4)], dim=-1)
    return f.reshape(*p.shape[:-1], p.shape[-1] * 4) - 1


def _torch_w2a8_map(u, packed, beta):
    """Eq. (4) written with torch routines: per-row absmax scale (fp32 IEEE
    division), round-half-to-even codes, an exact integer product (fp64 sums
    of small integers), (acc * alpha) * beta in fp32, then bf16 round-to-
    nearest-even by torch's conversion; returned as fp64."""
    u32 = u.to(torch.float32)
    alpha = torch.clamp(u32.abs().amax(dim=-1, keepdim=True), min=1e-5) / torch.tensor(127.0, dtype=torch.float32)
    a = torch.clamp(torch.round(u32 / alpha), -128, 127)
    q = _torch_unpack_ternary(packed).to(torch.float64)
    acc = a.to(torch.float64) @ q.transpose(0, 1)
    b = torch.from_numpy(np.atleast_1d(np.asarray(beta, dtype=np.float32)))
    b = torch.repeat_interleave(b, acc.shape[1] // b.numel())  # one scale per group of output rows
    y = (acc.to(torch.float32) * alpha) * b
    return y.to(torch.bfloat16).to(torch.float64)


def _torch_velocity_w2a8(x, tau, Kc, Vc, w, cfg):
    """The W2A8 velocity network with torch library routines (fp64 outside
    Eq. 4): every per-layer map replaced by its own quantised product, Q, K
    and V quantising the same normalised rows, the O-projection quantising the
    attention output and W_down the GeLU output."""
    T = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))
    e = T(O.sinusoidal_time_embedding(tau, cfg.d_t))
    sc = tF.silu(tF.linear(tF.silu(tF.linear(e, T(w["wt1"]))), T(w["wt2"])))
    h = tF.linear(T(x), T(w["win"]))
    B, H, _ = x.shape
    lin = lambda u, name, l: _torch_w2a8_map(u.reshape(B * H, -1), w[name][l], w["beta_" + name][l]).view(B, H, -1)
    for l in range(cfg.L):
        ga, ba, gm, bm = tF.linear(sc, T(w["wmod"][l])).view(4, cfg.D)
        u = tF.rms_norm(h, (cfg.D,), eps=cfg.eps) * (1 + ga) + ba
        q = lin(u, "wq", l).view(B, H, cfg.n_q, cfg.d_h).transpose(1, 2)
        k = lin(u, "wk", l).view(B, H, cfg.n_kv, cfg.d_h).transpose(1, 2)
        v = lin(u, "wv", l).view(B, H, cfg.n_kv, cfg.d_h).transpose(1, 2)
        k = torch.cat([T(Kc[l]), k], dim=2)
        v = torch.cat([T(Vc[l]), v], dim=2)
        o = tF.scaled_dot_product_attention(q, k, v, enable_gqa=True).transpose(1, 2).reshape(B, H, -1)
        h = h + lin(o, "wo", l)
        u = tF.rms_norm(h, (cfg.D,), eps=cfg.eps) * (1 + gm) + bm
        h = h + lin(tF.gelu(lin(u, "wup", l)), "wdown", l)
    gf, bf = tF.linear(sc, T(w["wmod_f"])).view(2, cfg.D)
    return tF.linear(tF.rms_norm(h, (cfg.D,), eps=cfg.eps) * (1 + gf) + bf, T(w["wout"])).numpy()


def test_w2a8_velocity_vs_library_routines():
    """velocity_w2a8 with non-zero ternary maps and six distinct scales per
    layer against an independent torch restatement: a swapped scale, the
    GeLU input quantised instead of its output, or Q's codes reused for the
    O-projection would each change the result."""
    cfg = PIN.replace(w2a8=True, dtype="bf16", L=2)
    w = make_weights(cfg)
    for l in range(cfg.L):
        betas = [float(w["beta_" + n][l]) for n in ("wq", "wk", "wv", "wo", "wup", "wdown")]
        assert len(set(betas)) == 6
    Z, noise = make_observations(cfg)
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    for tau in (0.0, 1.0 / 3.0, 0.75):
        v = O.velocity_w2a8(noise, tau, Kc, Vc, w, cfg)
        ref = _torch_velocity_w2a8(noise.astype(np.float64), tau, Kc, Vc, w, cfg)
        assert np.max(np.abs(v)) > 0.1
        np.testing.assert_allclose(v, ref, rtol=0, atol=1e-9)


def test_w2a8_velocity_detects_swapped_scales():
    """The restatement above is sensitive to the scale wiring: exchanging the
    W_k and W_v scales of one layer moves the velocity by far more than the
    tolerance used there."""
    cfg = PIN.replace(w2a8=True, dtype="bf16", L=2)
    w = make_weights(cfg)
    Z, noise = make_observations(cfg)
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    v = O.velocity_w2a8(noise, 0.5, Kc, Vc, w, cfg)
    w2 = dict(w)
    w2["beta_wk"], w2["beta_wv"] = w["beta_wv"].copy(), w["beta_wk"].copy()
    v2 = O.velocity_w2a8(noise, 0.5, Kc, Vc, w2, cfg)
    assert np.max(np.abs(v - v2)) > 1e-6


def test_w2a8_linear_is_eq4_of_rows():
    """One W2A8 map on a batch of rows == Eq. 4 applied row by row."""
    cfg = PIN.replace(w2a8=True, dtype="bf16")
    w = make_weights(cfg)
    rng = np.random.default_rng(12)
    u = rng.standard_normal((7, cfg.D)).astype(np.float32)
    a, alpha = O.quantize_rows(u)
    y, _ = O.ternary_linear(a, alpha, w["wup"][1], w["beta_wup"][1])
    for m in range(7):
        a1, al1 = O.quantize_rows(u[m:m + 1])
        y1, _ = O.ternary_linear(a1, al1, w["wup"][1], w["beta_wup"][1])
        assert np.array_equal(y1[0], y[m])


# ---------------------------------------------------------- Eq. (5)

def test_parity_metrics():
    Ahat = np.arange(12.0).reshape(3, 4)
    A = Ahat.copy()
    A[1, 2] += 0.25
    m = O.parity_metrics(A, Ahat)
    assert m["e_inf"] == 0.25
    assert abs(m["e_rel"] - 0.25 / np.linalg.norm(Ahat)) < 1e-15
    z = O.parity_metrics(np.full(4, 0.5), np.zeros(4))
    assert z["e_rel"] is None and z["e_abs"] == 1.0 and z["e_inf"] == 0.5


def test_w2a8_unpacked_cache_is_same_function():
    cfg = PIN.replace(w2a8=True, dtype="bf16")
    w = make_weights(cfg)
    Z, noise = make_observations(cfg)
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    v1 = O.velocity_w2a8(noise, 0.5, Kc, Vc, w, cfg)
    v2 = O.velocity_w2a8(noise, 0.5, Kc, Vc, O.with_unpacked(w), cfg)
    assert np.array_equal(v1, v2)


# ---------------------------------------------------------- request options (§III-A, §III-C)

def test_philox_matches_library_philox():
    """The oracle's Philox4x64-10 against numpy's Philox bit generator (an
    independent implementation of the same published generator; numpy's
    n-th block of four words uses counter n + 1)."""
    for seed in (0, 1, 12345, 2 ** 63 + 5):
        raw = np.random.Philox(key=seed).random_raw(16)
        for n in range(4):
            got = O.philox4x64([n + 1, 0, 0, 0], [seed, 0])
            assert [int(x) for x in raw[4 * n:4 * n + 4]] == got


def test_gaussian_noise_inverts_to_the_generator_words():
    """Box-Muller run backwards: for each pair (z0, z1) of the stream,
    exp(-(z0^2 + z1^2) / 2) is the first uniform and atan2(z1, z0) / 2 pi
    (mod 1) the second, both formed from numpy's Philox words."""
    seed = 99
    z = O.gaussian_noise(seed, (4000,)).astype(np.float64)
    # numpy's generator increments its counter before each block: start it one
    # below zero so that its first block is counter 0
    top = np.iinfo(np.uint64).max
    words = np.random.Philox(key=seed, counter=[top, top, top, top]).random_raw(4000).astype(np.uint64)
    z = z.reshape(-1, 2)
    w = words.reshape(-1, 2)
    u1 = ((w[:, 0] >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0 ** -53
    u2 = (w[:, 1] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r2 = z[:, 0] ** 2 + z[:, 1] ** 2
    np.testing.assert_allclose(np.exp(-r2 / 2), u1, rtol=2e-6 * (1 + r2.max()), atol=1e-7)
    ang = np.mod(np.arctan2(z[:, 1], z[:, 0]) / (2 * np.pi), 1.0)
    d = np.abs(ang - u2)
    assert np.all(np.minimum(d, 1 - d) <= 1e-6)


def test_gaussian_noise_is_standard_normal_and_prefix_stable():
    from scipy import stats
    z = O.gaussian_noise(7, (20000,)).astype(np.float64)
    assert stats.kstest(z, "norm").pvalue > 1e-3
    assert abs(z.mean()) < 0.03 and abs(z.std() - 1) < 0.03
    a = O.gaussian_noise(3, (4, 5, 7))
    b = O.gaussian_noise(3, (1, 5, 7))
    assert np.array_equal(a[:1], b)


def test_prefix_mask_bits_vs_packbits():
    rng = np.random.default_rng(3)
    v = rng.random((3, 77)) < 0.5
    words = O.prefix_mask_bits(v)
    ref = np.packbits(np.pad(v, ((0, 0), (0, 96 - 77))), axis=1, bitorder="little").view("<u4")
    assert np.array_equal(words, ref)


def test_reverse_schedule_constant_field_endpoint():
    """tau runs 1 -> 0: with a tau-independent, token-independent velocity
    field the solve ends at X^0 + (tau_S - tau_0) v = X^0 - v (the sign
    change of the reverse convention)."""
    cfg = PIN.replace(reverse=True)
    w, Z, noise = _setup(cfg, zero=("win", "wt1", "wt2", "wmod", "wmod_f"))
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    xS, vs = O.denoise(noise, Kc, Vc, w, cfg)
    assert np.allclose(vs, vs[0:1], atol=1e-13, rtol=0)
    np.testing.assert_allclose(xS, noise - vs[0], rtol=0, atol=1e-12)
    assert np.array_equal(O.schedule(4, True), np.array([1.0, 0.75, 0.5, 0.25, 0.0]))


def test_reverse_schedule_evaluates_the_reversed_time():
    cfg = PIN.replace(reverse=True)
    w, Z, noise = _setup(cfg)
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    _, vs = O.denoise(noise, Kc, Vc, w, cfg)
    np.testing.assert_allclose(vs[0], O.velocity(noise, 1.0, Kc, Vc, w, cfg), rtol=0, atol=1e-13)
    x1 = noise - vs[0] / cfg.S
    np.testing.assert_allclose(vs[1], O.velocity(x1, 1.0 - 1.0 / cfg.S, Kc, Vc, w, cfg), rtol=0, atol=1e-12)


def test_hidden_prefix_keys_equal_deleted_keys():
    """M = -inf on a prefix key (Eq. 2) is the same as removing the key from
    the cache, for every observation independently; hiding every prefix key
    leaves attention over the action tokens alone."""
    cfg = PIN.replace(B=2, P=10)
    w, Z, noise = _setup(cfg)
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    vis = np.array([[1, 0, 1, 1, 0, 0, 1, 0, 1, 1], [0] * 10], dtype=bool)
    xS, _ = O.denoise(noise, Kc, Vc, w, cfg, prefix_visible=vis)
    for b in range(2):
        keep = np.flatnonzero(vis[b])
        xb, _ = O.denoise(noise[b:b + 1], Kc[:, b:b + 1][:, :, :, keep], Vc[:, b:b + 1][:, :, :, keep], w,
                          cfg.replace(B=1))
        np.testing.assert_allclose(xS[b:b + 1], xb, rtol=0, atol=1e-12)



# ---------------------------------------------------------- W2A8 scale groups and ternary prefix maps (§III-D)

def test_ternary_linear_group_scales_are_blockwise_tensor_scales():
    """beta_{g(n)} per group of rows == the (pinned) per-tensor product on
    each block of rows with that block's scale."""
    rng = np.random.default_rng(21)
    a = rng.integers(-127, 128, size=(5, 64)).astype(np.int8)
    q = rng.integers(-1, 2, size=(32, 64)).astype(np.int8)
    packed = O.pack_ternary(q)
    alpha = rng.uniform(1e-3, 1.0, 5).astype(np.float32)
    beta = rng.uniform(0.01, 0.1, 4).astype(np.float32)
    y, acc = O.ternary_linear(a, alpha, packed, beta)
    for g in range(4):
        yg, ag = O.ternary_linear(a, alpha, packed[8 * g:8 * g + 8], beta[g])
        assert np.array_equal(y[:, 8 * g:8 * g + 8], yg) and np.array_equal(acc[:, 8 * g:8 * g + 8], ag)


def test_prefix_kv_w2a8_vs_library_routines():
    """Ternary prefix maps: K_C, V_C equal, bit for bit, an independent torch
    restatement of Eq. (4) on the prefix rows with per-group scales."""
    cfg = PIN.replace(w2a8=True, dtype="bf16", w2a8_prefix=True, beta_group=4)
    w = make_weights(cfg)
    assert w["wk_pre"].dtype == np.uint8 and w["beta_wk_pre"].shape == (cfg.L, cfg.kvdim // 4)
    Z, _ = make_observations(cfg)
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    Zt = torch.from_numpy(Z.astype(np.float64)).reshape(-1, cfg.d_vlm)
    for l in range(cfg.L):
        for name, ref in (("wk_pre", Kc), ("wv_pre", Vc)):
            y = _torch_w2a8_map(Zt, w[name][l], w["beta_" + name][l]).numpy()
            y = y.reshape(cfg.B, cfg.P, cfg.n_kv, cfg.d_h).transpose(0, 2, 1, 3)
            assert np.array_equal(y, ref[l])


def test_w2a8_velocity_group_scales_vs_library_routines():
    cfg = PIN.replace(w2a8=True, dtype="bf16", L=2, beta_group=8)
    w = make_weights(cfg)
    assert w["beta_wq"].shape == (cfg.L, cfg.qdim // 8)
    Z, noise = make_observations(cfg)
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    v = O.velocity_w2a8(noise, 0.4, Kc, Vc, w, cfg)
    ref = _torch_velocity_w2a8(noise.astype(np.float64), 0.4, Kc, Vc, w, cfg)
    np.testing.assert_allclose(v, ref, rtol=0, atol=1e-9)



# ---------------------------------------------------------- neuron-selected FFN (rMuscle Action Cache)

def test_selecting_every_neuron_in_any_order_is_the_dense_expert():
    """MLP hidden units are exchangeable: all F neurons, permuted, give the
    dense velocity."""
    w, Z, noise = _setup()
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    perm = np.stack([np.random.default_rng(l).permutation(PIN.F) for l in range(PIN.L)])
    v = O.velocity(noise, 0.3, Kc, Vc, O.select_ffn_neurons(w, perm), PIN)
    np.testing.assert_allclose(v, O.velocity(noise, 0.3, Kc, Vc, w, PIN), rtol=0, atol=1e-12)


def test_selected_neurons_equal_zeroing_the_others():
    """Evaluating a subset of neurons equals the dense expert whose other
    neurons' W_down columns are zero (their GeLU outputs then contribute 0)."""
    w, Z, noise = _setup()
    Kc, Vc = O.prefix_kv(Z, w, PIN)
    rng = np.random.default_rng(5)
    idx = np.stack([np.sort(rng.choice(PIN.F, PIN.F // 3, replace=False)) for _ in range(PIN.L)])
    wz = dict(w)
    wz["wdown"] = np.zeros_like(w["wdown"])
    for l in range(PIN.L):
        wz["wdown"][l][:, idx[l]] = w["wdown"][l][:, idx[l]]
    v = O.velocity(noise, 0.6, Kc, Vc, O.select_ffn_neurons(w, idx), PIN)
    np.testing.assert_allclose(v, O.velocity(noise, 0.6, Kc, Vc, wz, PIN), rtol=0, atol=1e-12)



# ---------------------------------------------------------- alternating joint / cross attention layers (§III-B)

def test_cross_attention_vs_library_sdpa():
    """suffix=False: the queries attend to the cached prefix keys only,
    torch's scaled_dot_product_attention over those keys (GQA)."""
    rng = np.random.default_rng(31)
    q, ks, vs, Kc, Vc = _rand_attn(rng)
    o = O.joint_attention(q, ks, vs, Kc, Vc, suffix=False)
    T = lambda a: torch.from_numpy(a)
    ref = tF.scaled_dot_product_attention(T(q).transpose(1, 2), T(Kc), T(Vc), enable_gqa=True).transpose(1, 2)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def test_cross_layers_ignore_the_action_keys():
    """In a cross-attention layer the action tokens' W_k, W_v do not enter:
    zeroing them there leaves the velocity unchanged, while in joint layers
    it changes it."""
    cfg = PIN.replace(cross_every=2)
    w, Z, noise = _setup(cfg)
    Kc, Vc = O.prefix_kv(Z, w, cfg)
    v = O.velocity(noise, 0.5, Kc, Vc, w, cfg)
    w1 = dict(w)
    w1["wk"] = w["wk"].copy(); w1["wv"] = w["wv"].copy()
    w1["wk"][1] = 0.0; w1["wv"][1] = 0.0            # layer 1 is a cross layer
    np.testing.assert_allclose(O.velocity(noise, 0.5, Kc, Vc, w1, cfg), v, rtol=0, atol=1e-14)
    w0 = dict(w)
    w0["wk"] = w["wk"].copy(); w0["wk"][0] = 0.0     # layer 0 is a joint layer
    assert np.max(np.abs(O.velocity(noise, 0.5, Kc, Vc, w0, cfg) - v)) > 1e-6
