"""W2A8 prefix cache build and per-group weight scales ("vla.cpp: A Unified
Inference Runtime for Vision-Language-Action Models", §III-D Eq. (4): ternary
maps with a checkpoint scale beta_{g(n)} per output group; §III-B Eq. (2):
the prefix K/V projection).

* The ternary prefix build (every prefix row of Z quantised per Eq. (4), one
  packed-ternary product over all layers' W_K and W_V with the cache scatter
  in its epilogue) equals the oracle bit for bit: K_C and V_C^T in bf16.
* A whole W2A8 solve with ternary prefix maps and per-group scales meets the
  W2A8 gates against the oracle.
"""

import numpy as np
import pytest

import oracle as O
from _harness import GATES, REL_GATES, gpu_run, oracle_compare
from workloads import CONFIGS

pytestmark = pytest.mark.gpu


def _bits(x):
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("B,P,group", [(1, 512, 128), (3, 77, 0), (2, 200, 64)])
def test_w2a8_prefix_build_bit_exact(B, P, group):
    cfg = CONFIGS["w2a8_b1"].replace(L=3, w2a8_prefix=True, beta_group=group, S=1)
    run = gpu_run(cfg, B=B, P=P)
    assert run["status"] == 0
    c = run["cfg"]
    Kr, Vr = O.prefix_kv(run["Z"], run["w"], c)
    assert np.array_equal(_bits(run["Kc"]), _bits(Kr))
    assert np.array_equal(_bits(run["Vc"]), _bits(Vr))


@pytest.mark.parametrize("name", ["w2a8_b1", "w2a8_b16"])
def test_w2a8_group_scales_and_ternary_prefix_end_to_end(name):
    cfg = CONFIGS[name].replace(w2a8_prefix=True, beta_group=128)
    run = gpu_run(cfg)
    assert run["status"] == 0
    res = oracle_compare(run, obs=[0] if cfg.B == 1 else [0, cfg.B - 1])
    g_v, g_x = GATES["w2a8"]
    print(name, "kv", res["kv"], "v_tf", res["v_tf"], "x", [m["e_inf"] for m in res["x"]])
    assert max(res["kv"]) == 0.0  # the cache is bit-exact
    assert max(res["v_tf"]) <= g_v and max(res["v_tf_rel"]) <= REL_GATES["w2a8"]
    assert all(m["e_inf"] <= g_x for m in res["x"])
