"""Seeded synthetic workloads for the prefix-cached flow-matching action expert.

This module is shared by both sides of the parity harness (the CPU oracle and
the CUDA library).  It holds shapes and random inputs only: none of the
method's arithmetic lives here.  Values that the method consumes in bf16 are
rounded to bf16 (round-to-nearest-even) *here*, before either side sees them,
so that the two sides differ only in how they compute.

Workload shapes follow the action-expert description in "vla.cpp: A Unified
Inference Runtime for Vision-Language-Action Models" (§III-A/B: H x d_a action
chunk, T solver steps, a fixed multimodal prefix of a few hundred tokens) and
the five configurations this library is measured on.

Random streams: numpy SFC64, one independent stream per (seed, purpose), so
that observation b of a batch-B draw equals observation b of any larger draw
with the same seed (used by batch-independence checks).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "ExpertConfig",
    "CONFIGS",
    "bf16_round",
    "make_weights",
    "make_observations",
    "TERNARY_NAMES",
    "WEIGHT_NAMES",
]

# Per-layer linear maps of the action expert that become ternary in the W2A8
# variant (vla.cpp §III-D); the rest (prefix K/V, in/out, time MLP,
# modulation) stay bf16.
TERNARY_NAMES = ("wq", "wk", "wv", "wo", "wup", "wdown")
WEIGHT_NAMES = ("wk_pre", "wv_pre", "wq", "wk", "wv", "wo", "wup", "wdown",
                "wmod", "win", "wout", "wt1", "wt2", "wmod_f")


@dataclasses.dataclass(frozen=True)
class ExpertConfig:
    """Shape of one action-expert workload.

    Notation: P prefix tokens of width d_vlm; L expert layers of width D, MLP
    width F, n_q query heads sharing n_kv key/value heads of size d_h; an action
    chunk of H actions with d_a dims; S Euler solver steps; d_t sinusoidal time
    embedding width; B independent observations.
    """

    name: str
    L: int
    D: int
    F: int
    n_q: int
    n_kv: int
    d_h: int
    d_vlm: int
    P: int
    H: int
    d_a: int
    S: int
    B: int = 1
    d_t: int = 256
    seed: int = 0
    dtype: str = "bf16"  # "f32" or "bf16": storage type of weights, Z, K/V cache
    w2a8: bool = False
    eps: float = 1e-6
    reverse: bool = False  # integration direction of the schedule: 0 -> 1, or 1 -> 0
    beta_group: int = 0    # W2A8: output rows per weight-scale group (0: one scale per tensor)
    w2a8_prefix: bool = False  # W2A8: the prefix K/V maps are ternary too
    cross_every: int = 0   # layers l with l % cross_every == cross_every - 1 attend to the prefix only

    def replace(self, **kw) -> "ExpertConfig":
        return dataclasses.replace(self, **kw)

    @property
    def tokens(self) -> int:
        return self.B * self.H

    @property
    def qdim(self) -> int:
        return self.n_q * self.d_h

    @property
    def kvdim(self) -> int:
        return self.n_kv * self.d_h

    def token_dependent_params(self) -> int:
        """Weights whose GEMM input depends on the action tokens (read every step)."""
        per_layer = (self.qdim + 2 * self.kvdim) * self.D + self.D * self.qdim + 2 * self.D * self.F
        return self.L * per_layer + self.D * self.d_a + self.d_a * self.D


CONFIGS = {
    # Tiny fp32 parity case.
    "tiny_f32": ExpertConfig("tiny_f32", L=2, D=128, F=512, n_q=4, n_kv=1, d_h=32,
                             d_vlm=128, P=64, H=8, d_a=7, S=4, B=1, seed=0, dtype="f32"),
    # Small bf16 (dual-arm action chunk).
    "small_bf16": ExpertConfig("small_bf16", L=6, D=512, F=2048, n_q=8, n_kv=2, d_h=64,
                               d_vlm=1024, P=256, H=16, d_a=14, S=4, B=1, seed=1),
    # Full-size bf16, batch 1 (latency): 3 images x 256 patches + 48 text tokens.
    "full_bf16_b1": ExpertConfig("full_bf16_b1", L=18, D=1024, F=4096, n_q=8, n_kv=1, d_h=256,
                                 d_vlm=2048, P=816, H=50, d_a=32, S=10, B=1, seed=2),
    # Same expert, 64 independent observations (throughput).
    "full_bf16_b64": ExpertConfig("full_bf16_b64", L=18, D=1024, F=4096, n_q=8, n_kv=1, d_h=256,
                                  d_vlm=2048, P=816, H=50, d_a=32, S=10, B=64, seed=3),
    # W2A8 (ternary weights, int8 activations); d_vlm is unstated -> width.
    "w2a8_b1": ExpertConfig("w2a8_b1", L=24, D=2048, F=5632, n_q=16, n_kv=4, d_h=128,
                            d_vlm=2048, P=512, H=8, d_a=7, S=8, B=1, seed=4, w2a8=True),
    "w2a8_b16": ExpertConfig("w2a8_b16", L=24, D=2048, F=5632, n_q=16, n_kv=4, d_h=128,
                             d_vlm=2048, P=512, H=8, d_a=7, S=8, B=16, seed=4, w2a8=True),
}


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 container."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def _rng(seed: int, purpose: int) -> np.random.Generator:
    return np.random.Generator(np.random.SFC64(np.random.SeedSequence([seed, purpose])))


def _shapes(cfg: ExpertConfig) -> dict:
    L, D, F = cfg.L, cfg.D, cfg.F
    return {
        "wk_pre": (L, cfg.kvdim, cfg.d_vlm),
        "wv_pre": (L, cfg.kvdim, cfg.d_vlm),
        "wq": (L, cfg.qdim, D),
        "wk": (L, cfg.kvdim, D),
        "wv": (L, cfg.kvdim, D),
        "wo": (L, D, cfg.qdim),
        "wup": (L, F, D),
        "wdown": (L, D, F),
        "wmod": (L, 4 * D, D),
        "win": (D, cfg.d_a),
        "wout": (cfg.d_a, D),
        "wt1": (D, cfg.d_t),
        "wt2": (D, D),
        "wmod_f": (2 * D, D),
    }


def weight_shapes(cfg: ExpertConfig) -> dict:
    """Logical [.., out, in] shape of every weight (ternary ones before packing)."""
    return _shapes(cfg)


def make_weights(cfg: ExpertConfig, zero: tuple = ()) -> dict:
    """Seeded synthetic weights, stored out-major ([.., out, in], in contiguous).

    Dense weights are i.i.d. N(0, 1/fan_in), rounded to bf16 for bf16 configs.
    For W2A8 configs the six per-layer token-dependent maps are ternary:
    codes c = q + 1 drawn i.i.d. uniform over {0, 1, 2} (so P(q = 0) = 1/3),
    packed four per byte, code of input index j at bits 2*(j mod 4) of byte
    j // 4 (little-endian within the byte); key ``<name>`` holds the packed
    uint8 [L, out, in/4] array and ``beta_<name>`` the fp32 per-tensor scale
    [L] (or, with ``beta_group`` > 0, one scale per group of that many output
    rows, [L, out / beta_group]; with ``w2a8_prefix`` the prefix maps W_K, W_V
    are ternary as well).  The scale is the expected absmean of an N(0, 1/fan_in) latent,
    sqrt(2/pi)/sqrt(fan_in), with a seeded +-5% jitter per (layer, tensor) so
    that a mixed-up scale index is visible.

    ``zero`` lists weight names to set to zero (used by closed-form checks).
    """
    shapes = _shapes(cfg)
    rng = _rng(cfg.seed, 0)
    rng_t = _rng(cfg.seed, 3)
    out = {}
    for name in WEIGHT_NAMES:
        shp = shapes[name]
        fan_in = shp[-1]
        if cfg.w2a8 and (name in TERNARY_NAMES or (cfg.w2a8_prefix and name in ("wk_pre", "wv_pre"))):
            if fan_in % 4:
                raise ValueError(f"{name}: fan_in {fan_in} not a multiple of 4")
            codes = rng_t.integers(0, 3, size=shp, dtype=np.uint8)
            c = codes.reshape(shp[:-1] + (fan_in // 4, 4))
            packed = (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)
            groups = (cfg.L,) if cfg.beta_group == 0 else (cfg.L, shp[-2] // cfg.beta_group)
            beta = (math.sqrt(2.0 / math.pi) / math.sqrt(fan_in)) * (
                1.0 + 0.05 * rng_t.uniform(-1.0, 1.0, size=groups))
            if name in zero:
                packed = np.full_like(packed, 0x55)  # every code 1 -> q = 0
            out[name] = np.ascontiguousarray(packed)
            out["beta_" + name] = beta.astype(np.float32)
            continue
        w = rng.standard_normal(size=shp, dtype=np.float32)
        w *= np.float32(1.0 / math.sqrt(fan_in))
        if name in zero:
            w[...] = 0.0
        if cfg.dtype == "bf16":
            w = bf16_round(w)
        out[name] = np.ascontiguousarray(w)
    return out


def make_observations(cfg: ExpertConfig, B: int | None = None):
    """Seeded prefix hidden states Z [B, P, d_vlm] and noise X^0 [B, H, d_a].

    Z ~ N(0, 1) i.i.d. (rounded to bf16 for bf16 configs; the prefix is
    position-free so its token structure does not enter the values).  The
    noise is fp32 N(0, 1).  Observation b is the same for every B > b.
    """
    B = cfg.B if B is None else B
    rz = _rng(cfg.seed, 1)
    rn = _rng(cfg.seed, 2)
    Z = rz.standard_normal(size=(B, cfg.P, cfg.d_vlm), dtype=np.float32)
    if cfg.dtype == "bf16":
        Z = bf16_round(Z)
    noise = rn.standard_normal(size=(B, cfg.H, cfg.d_a), dtype=np.float32)
    return np.ascontiguousarray(Z), np.ascontiguousarray(noise)
