"""Per-request options on the GPU against the oracle ("vla.cpp: A Unified
Inference Runtime for Vision-Language-Action Models", §III-C: requests carry
inputs plus optional noise and masks; §III-A: the 1 -> 0 time convention;
§III-B Eq. (2): M = -inf on hidden keys).

* In-library noise: the library's Philox4x64-10 / Box-Muller stream equals
  the oracle's within one fp32 rounding, and a request without noise solves
  from exactly that X^0.
* Prefix masks: random visibility per observation (one observation with
  every cached key hidden, one with a prefix length) on every attention
  kernel (clustered, streaming, CUDA-core, persistent) and on the W2A8 path,
  against the oracle's masked Eq. (2), within the bf16 gates.
* Reverse schedule: tau 1 -> 0 with dt = -1/S, against the oracle.
"""

import numpy as np
import pytest

import oracle as O
from _harness import GATES, weights
from workloads import CONFIGS, make_observations

pytestmark = pytest.mark.gpu


def _expert(cfg, B, P, flags=0):
    import prefix_cached_flow_gb300 as V
    w = weights(cfg)
    ex = V.Expert(cfg, V.upload_weights(w, cfg.dtype, cfg.w2a8), max_batch=B, max_prefix=P, flags=flags)
    return ex, w


def _cache(ex, cfg, Z):
    import torch
    dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    B, P = Z.shape[0], Z.shape[1]
    Kc, Vc = ex.alloc_cache(B, P)
    ex.prefix_kv_build(torch.from_numpy(Z).to(dt).cuda(), Kc, Vc)
    return Kc, Vc


def test_noise_stream_matches_oracle():
    import prefix_cached_flow_gb300 as V
    for seed, n in ((0, 1), (5, 1000), (2 ** 40 + 3, 4003)):
        got = V.noise_fill(seed, n).cpu().numpy()
        ref = O.gaussian_noise(seed, (n,))
        ulp = np.spacing(np.abs(ref).astype(np.float32))
        assert np.all(np.abs(got - ref) <= ulp), seed


def _masks(rng, B, P):
    vis = rng.random((B, P)) < 0.6
    vis[0, :] = False                 # observation 0: every cached key hidden
    if B > 2:
        vis[2, :] = np.arange(P) < P // 3   # observation 2: a prefix length
    return vis


def _gate(cfg):
    return GATES["w2a8" if cfg.w2a8 else ("f32" if cfg.dtype == "f32" else "bf16")][1]


@pytest.mark.parametrize("form", ["default", "split", "stream", "simt", "persist"])
def test_prefix_mask_and_seeded_noise(form):
    import torch
    import prefix_cached_flow_gb300 as V
    flags = {"default": 0, "split": V.FLAG_ATTN_SPLIT, "stream": V.FLAG_ATTN_STREAM, "simt": V.FLAG_SIMT_GEMM,
             "persist": V.FLAG_PERSIST}[form]
    cfg = CONFIGS["small_bf16"]
    B, P = 3, 77
    c = cfg.replace(B=B, P=P)
    Z, _ = make_observations(c, B)
    ex, w = _expert(cfg, B, P, flags)
    Kc, Vc = _cache(ex, c, Z)
    vis = _masks(np.random.default_rng(11), B, P)
    mask = torch.from_numpy(O.prefix_mask_bits(vis).view(np.int32)).cuda()
    seed = 1234
    nout = torch.empty((B, c.H, c.d_a), dtype=torch.float32, device="cuda")
    act = ex.denoise_ex(Kc, Vc, B, prefix_mask=mask, seed=seed, noise_out=nout)
    torch.cuda.synchronize()
    assert ex.poll_status() == 0
    x0 = O.gaussian_noise(seed, (B, c.H, c.d_a))
    assert np.max(np.abs(nout.cpu().numpy() - x0)) <= 1e-6
    Kr, Vr = O.prefix_kv(Z.astype(np.float64), w, c)
    xr, _ = O.denoise(x0.astype(np.float64), Kr, Vr, w, c, prefix_visible=vis)
    err = np.max(np.abs(act.cpu().numpy() - xr))
    print(form, "masked chunk max-abs", err)
    assert err <= _gate(cfg)
    # the mask matters: the unmasked solve from the same noise is far from it
    xu, _ = O.denoise(x0.astype(np.float64), Kr, Vr, w, c)
    assert np.max(np.abs(xu - xr)) > 10 * _gate(cfg)


def test_prefix_mask_w2a8():
    import torch
    cfg = CONFIGS["w2a8_b1"].replace(L=4)
    B, P = 2, 200
    c = cfg.replace(B=B, P=P)
    Z, noise = make_observations(c, B)
    ex, w = _expert(cfg, B, P)
    Kc, Vc = _cache(ex, c, Z)
    vis = _masks(np.random.default_rng(12), B, P)
    mask = torch.from_numpy(O.prefix_mask_bits(vis).view(np.int32)).cuda()
    act = ex.denoise_ex(Kc, Vc, B, prefix_mask=mask, noise=torch.from_numpy(noise).cuda())
    torch.cuda.synchronize()
    assert ex.poll_status() == 0
    Kr, Vr = O.prefix_kv(Z.astype(np.float64), w, c)
    xr, _ = O.denoise_w2a8(noise.astype(np.float64), Kr, Vr, w, c, prefix_visible=vis)
    assert np.max(np.abs(act.cpu().numpy() - xr)) <= _gate(cfg)


@pytest.mark.parametrize("name,flags", [("small_bf16", 0), ("full_bf16_b1", 0), ("small_bf16", "persist"),
                                        ("small_bf16", "wide"), ("tiny_f32", 0)])
def test_reverse_schedule(name, flags):
    """flags "wide": the many-token linears with the factored norm, whose
    W beta tables follow the reversed time."""
    import torch
    import prefix_cached_flow_gb300 as V
    cfg = CONFIGS[name].replace(reverse=True)
    fl = {0: 0, "persist": V.FLAG_PERSIST, "wide": V.FLAG_LINEAR_WIDE}[flags]
    Z, noise = make_observations(cfg, cfg.B)
    ex, w = _expert(cfg, cfg.B, cfg.P, fl)
    Kc, Vc = _cache(ex, cfg, Z)
    tap = torch.empty((cfg.S, cfg.B, cfg.H, cfg.d_a), dtype=torch.float32, device="cuda")
    act = ex.denoise(Kc, Vc, torch.from_numpy(noise).cuda(), vel_tap=tap)
    torch.cuda.synchronize()
    assert ex.poll_status() == 0
    Kr, Vr = O.prefix_kv(Z.astype(np.float64), w, cfg)
    xr, _ = O.denoise(noise.astype(np.float64), Kr, Vr, w, cfg)
    assert np.max(np.abs(act.cpu().numpy() - xr)) <= _gate(cfg)
    # teacher-forced first velocity at tau = 1
    v0 = O.velocity(noise.astype(np.float64), 1.0, Kr, Vr, w, cfg)
    assert np.max(np.abs(tap[0].cpu().numpy() - v0)) <= GATES["bf16" if cfg.dtype == "bf16" else "f32"][0]
