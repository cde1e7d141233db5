"""Architecture variants of the same solver loop on the GPU against the
oracle ("vla.cpp: A Unified Inference Runtime for Vision-Language-Action
Models", §III-B: SmolVLA alternates joint- and cross-attention layers;
"rMuscle" page: during the memory-bound denoising loop the expert evaluates
only selected FFN neurons).

* Neuron-selected FFN: the library's compact W_up rows / W_down columns of a
  random selection against the oracle's expert restricted to the same
  neurons; restoring the full MLP gives the dense result again; invalid
  selections are refused and leave the handle unchanged.
* Alternating joint / cross attention (every second layer attends to the
  cached prefix only) on every attention kernel.
"""

import numpy as np
import pytest

import oracle as O
from _harness import GATES, gpu_run, oracle_compare
from workloads import CONFIGS, make_observations

pytestmark = pytest.mark.gpu


def _solve(ex, cfg, Z, noise):
    import torch
    Kc, Vc = ex.alloc_cache(cfg.B, cfg.P)
    ex.prefix_kv_build(torch.from_numpy(Z).to(torch.bfloat16).cuda(), Kc, Vc)
    act = ex.denoise(Kc, Vc, torch.from_numpy(noise).cuda())
    torch.cuda.synchronize()
    assert ex.poll_status() == 0
    return act.cpu().numpy()


@pytest.mark.parametrize("name,frac", [("small_bf16", 2), ("full_bf16_b1", 4)])
def test_selected_ffn_neurons(name, frac):
    import torch
    import prefix_cached_flow_gb300 as V
    cfg = CONFIGS[name]
    run = gpu_run(cfg)
    ex, w = run["expert"], run["w"]
    rng = np.random.default_rng(17)
    Fs = cfg.F // frac
    idx = np.stack([np.sort(rng.choice(cfg.F, Fs, replace=False)) for _ in range(cfg.L)]).astype(np.int32)
    ex.select_ffn(torch.from_numpy(idx).cuda())
    act = _solve(ex, cfg, run["Z"], run["noise"])
    ws = O.select_ffn_neurons(w, idx)
    Kr, Vr = O.prefix_kv(run["Z"].astype(np.float64), w, cfg)
    xr, _ = O.denoise(run["noise"].astype(np.float64), Kr, Vr, ws, cfg)
    err = np.max(np.abs(act - xr))
    print(name, "selected", Fs, "of", cfg.F, "chunk max-abs", err)
    assert err <= GATES["bf16"][1]
    # refused selections keep the selection in force
    bad = idx.copy()
    bad[0, 1] = bad[0, 0]  # not strictly increasing
    with pytest.raises(V.VlaError):
        ex.select_ffn(torch.from_numpy(bad).cuda())
    assert np.array_equal(_solve(ex, cfg, run["Z"], run["noise"]), act)
    # the full MLP again
    ex.select_ffn(None)
    assert np.array_equal(_solve(ex, cfg, run["Z"], run["noise"]), run["act"])


@pytest.mark.parametrize("form", ["default", "split", "stream", "simt"])
def test_alternating_cross_attention_layers(form):
    import prefix_cached_flow_gb300 as V
    flags = {"default": 0, "split": V.FLAG_ATTN_SPLIT, "stream": V.FLAG_ATTN_STREAM, "simt": V.FLAG_SIMT_GEMM}[form]
    cfg = CONFIGS["small_bf16"].replace(cross_every=2)
    run = gpu_run(cfg, B=2, P=77, flags=flags)
    assert run["status"] == 0
    res = oracle_compare(run, obs=[0, 1])
    g_v, g_x = GATES["bf16"]
    print(form, "v_tf", res["v_tf"], "x", [m["e_inf"] for m in res["x"]])
    assert max(res["v_tf"]) <= g_v
    assert all(m["e_inf"] <= g_x for m in res["x"])


def test_alternating_cross_attention_full_size():
    cfg = CONFIGS["full_bf16_b1"].replace(cross_every=2)
    run = gpu_run(cfg)
    assert run["status"] == 0
    res = oracle_compare(run, obs=[0])
    g_v, g_x = GATES["bf16"]
    assert max(res["v_tf"]) <= g_v
    assert res["x"][0]["e_inf"] <= g_x
