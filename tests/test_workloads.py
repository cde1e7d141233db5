"""The seeded synthetic inputs both sides receive, against the recipe they
are documented to follow (no GPU needed).

Every parity test and the benchmark draw their inputs here, so a generator
that silently changed (a different stream, values no longer representable
in bf16, a skewed ternary code distribution) would change what is measured
and compared without any test noticing.  The recipe: dense weights
N(0, 1/fan_in), prefix states and noise N(0, 1), bf16 configurations rounded
to bf16 (nearest, ties to even) before either side sees them, ternary codes
uniform over {-1, 0, 1} packed four per byte (code q + 1 of input index j at
bits 2 (j mod 4)), per-tensor scales sqrt(2/pi)/sqrt(fan_in) within +-5%.
"""

import math

import numpy as np
import pytest
import torch

from workloads import CONFIGS, bf16_round, make_observations, make_weights, weight_shapes


def _small_w2a8():
    return CONFIGS["w2a8_b1"].replace(L=2, D=256, F=512, n_q=4, n_kv=2, d_h=64, d_vlm=256, P=40)


def test_generators_are_deterministic_per_seed():
    cfg = CONFIGS["small_bf16"]
    w1, w2 = make_weights(cfg), make_weights(cfg)
    assert all(np.array_equal(w1[k], w2[k]) for k in w1)
    (z1, n1), (z2, n2) = make_observations(cfg), make_observations(cfg)
    assert np.array_equal(z1, z2) and np.array_equal(n1, n2)
    w3 = make_weights(cfg.replace(seed=cfg.seed + 1))
    assert not np.array_equal(w1["wq"], w3["wq"])


def test_observation_b_does_not_depend_on_the_batch_size():
    cfg = CONFIGS["small_bf16"]
    z4, n4 = make_observations(cfg, 4)
    z2, n2 = make_observations(cfg, 2)
    assert np.array_equal(z4[:2], z2) and np.array_equal(n4[:2], n2)


def test_shapes_match_the_configuration():
    cfg = CONFIGS["small_bf16"]
    w = make_weights(cfg)
    for name, shp in weight_shapes(cfg).items():
        assert w[name].shape == shp, name
    Z, noise = make_observations(cfg, 3)
    assert Z.shape == (3, cfg.P, cfg.d_vlm) and noise.shape == (3, cfg.H, cfg.d_a)
    assert noise.dtype == np.float32


def test_bf16_configs_hand_bf16_representable_values():
    cfg = CONFIGS["small_bf16"]
    w = make_weights(cfg)
    Z, noise = make_observations(cfg)
    for x in [Z] + [w[k] for k in ("wq", "wup", "win", "wmod")]:
        assert np.array_equal(x, bf16_round(x))
        assert np.array_equal(torch.from_numpy(x).to(torch.bfloat16).float().numpy(), x)
    # the noise stays fp32 (it is the solver state, not a bf16 operand)
    assert not np.array_equal(noise, bf16_round(noise))


def test_bf16_round_is_nearest_even():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 1.0 + 2.0 ** -8 + 2.0 ** -20],
                 dtype=np.float32)
    # halfway cases go to the even neighbour; just above halfway goes up
    assert bf16_round(x).tolist() == [1.0, 1.0, 1.0 + 2.0 ** -6, -1.0, 1.0 + 2.0 ** -7]
    r = np.random.default_rng(0).standard_normal(4096).astype(np.float32)
    assert np.array_equal(bf16_round(r), torch.from_numpy(r).to(torch.bfloat16).float().numpy())


def test_dense_weight_and_input_distributions():
    cfg = CONFIGS["small_bf16"]
    w = make_weights(cfg)
    for name in ("wq", "wo", "wup", "wdown"):
        x = w[name].astype(np.float64)
        fan_in = x.shape[-1]
        # variance 1/fan_in within a few standard errors of the sample variance
        assert abs(x.var() * fan_in - 1.0) < 0.02, name
        assert abs(x.mean()) * math.sqrt(fan_in) < 0.01, name
    Z, noise = make_observations(cfg, 2)
    assert abs(Z.astype(np.float64).var() - 1.0) < 0.01 and abs(Z.mean()) < 0.01


def test_ternary_codes_layout_distribution_and_scales():
    cfg = _small_w2a8()
    w = make_weights(cfg)
    shapes = weight_shapes(cfg)
    for name in ("wq", "wk", "wv", "wo", "wup", "wdown"):
        L, n_out, k_in = shapes[name]
        packed = w[name]
        assert packed.dtype == np.uint8 and packed.shape == (L, n_out, k_in // 4)
        codes = np.stack([(packed >> (2 * j)) & 3 for j in range(4)], axis=-1).reshape(L, n_out, k_in)
        assert codes.max() <= 2  # code 3 is never drawn
        frac = np.bincount(codes.ravel(), minlength=3) / codes.size
        assert np.all(np.abs(frac - 1.0 / 3.0) < 0.01), (name, frac)
        beta = w["beta_" + name]
        nominal = math.sqrt(2.0 / math.pi) / math.sqrt(k_in)
        assert beta.shape == (L,) and np.all(np.abs(beta / nominal - 1.0) <= 0.05 + 1e-6)
    # a zeroed ternary map holds code 1 (q = 0) everywhere
    wz = make_weights(cfg, zero=("wo",))
    assert np.all(wz["wo"] == 0x55)


def test_group_scales_have_one_entry_per_group():
    cfg = _small_w2a8().replace(beta_group=64)
    w = make_weights(cfg)
    shapes = weight_shapes(cfg)
    for name in ("wq", "wup", "wdown"):
        L, n_out, _ = shapes[name]
        assert w["beta_" + name].shape == (L, n_out // 64)


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_every_configuration_is_consistent(name):
    cfg = CONFIGS[name]
    assert cfg.n_q % cfg.n_kv == 0
    assert cfg.D % 64 == 0 and cfg.F % 64 == 0 and cfg.d_vlm % 64 == 0
    if cfg.w2a8:
        assert cfg.D % 4 == 0 and cfg.F % 4 == 0 and cfg.qdim % 4 == 0
