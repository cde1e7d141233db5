"""Shared helpers for the GPU parity tests: run the CUDA library and the CPU
oracle on the same seeded inputs and compare with the Eq. (5) metrics of
"vla.cpp: A Unified Inference Runtime for Vision-Language-Action Models"
(§III-E)."""

from __future__ import annotations

import numpy as np

import oracle as O
from workloads import make_observations, make_weights

# Gates: bf16 paths, max-abs error on every per-step velocity (teacher-forced:
# the oracle evaluates v at the GPU's own x_k) and on the final chunk
# (free-running); the fp32 instance is held to a much tighter bound.
GATES = {"bf16": (2e-2, 1e-2), "f32": (1e-4, 1e-4),
         # W2A8 end to end: the quantiser turns rounding-level differences of
         # its fp32 input into whole-code flips.  Perturbing the oracle's own
         # quantiser inputs by 2^-22 (relative) flips 3-11 codes per velocity
         # evaluation of the 24-layer expert and moves v by max-abs 0.04-0.08
         # (relative RMS 2-3%); the gate is twice that self-sensitivity.  The
         # integer codes, scales and accumulators themselves are checked bit
         # for bit in test_gpu_w2a8_units.py.
         "w2a8": (0.16, 0.08)}
REL_GATES = {"bf16": 0.01, "f32": 1e-5, "w2a8": 0.06}

_WEIGHTS = {}


def weights(cfg):
    key = cfg.replace(name="", B=1, P=1, S=1)
    if key not in _WEIGHTS:
        _WEIGHTS.clear()  # keep host memory bounded: one weight set at a time
        w = make_weights(cfg)
        _WEIGHTS[key] = O.with_unpacked(w) if cfg.w2a8 else w
    return _WEIGHTS[key]


def gpu_run(cfg, B=None, P=None, flags=0, noise=None, Z=None, max_batch=None, max_prefix=None, w=None):
    import torch

    import prefix_cached_flow_gb300 as V

    B = cfg.B if B is None else B
    P = cfg.P if P is None else P
    c = cfg.replace(B=B, P=P)
    w = weights(cfg) if w is None else w
    Zn, nz = make_observations(c, B)
    Z = Zn if Z is None else Z
    noise = nz if noise is None else noise
    dw = V.upload_weights(w, c.dtype, c.w2a8)
    ex = V.Expert(c, dw, max_batch=max_batch or B, max_prefix=max_prefix or P, flags=flags)
    del dw
    dt = torch.float32 if c.dtype == "f32" else torch.bfloat16
    Zt = torch.from_numpy(np.ascontiguousarray(Z)).to(dt).cuda()
    nt = torch.from_numpy(np.ascontiguousarray(noise)).cuda()
    Kc, Vc = ex.alloc_cache(B, P)
    ex.prefix_kv_build(Zt, Kc, Vc)
    tap = torch.empty((c.S, B, c.H, c.d_a), dtype=torch.float32, device="cuda")
    act = ex.denoise(Kc, Vc, nt, vel_tap=tap)
    torch.cuda.synchronize()
    status = ex.poll_status()
    out = {
        "cfg": c, "w": w, "Z": Z, "noise": noise, "status": status, "expert": ex,
        # V_C is stored transposed [L, B, n_kv, d_h, P8]; compare as [.., P, d_h]
        "Kc": Kc.float().cpu().numpy(), "Vc": Vc[..., :P].transpose(-1, -2).float().cpu().numpy(),
        "act": act.cpu().numpy(), "tap": tap.cpu().numpy(),
    }
    return out


def oracle_compare(run, obs=None, teacher_forced=True, free_running=True):
    """Per-observation Eq. (5) metrics of the GPU run against the oracle."""
    c, w = run["cfg"], run["w"]
    obs = range(c.B) if obs is None else obs
    vel = O.velocity_w2a8 if c.w2a8 else O.velocity
    tau = O.schedule(c.S)
    res = {"v_tf": [], "x": [], "kv": []}
    for b in obs:
        Z = run["Z"][b:b + 1].astype(np.float64)
        Kc, Vc = O.prefix_kv(Z, w, c)
        kv_err = max(float(np.max(np.abs(run["Kc"][:, b:b + 1] - Kc) / (np.abs(Kc) + 0.25))),
                     float(np.max(np.abs(run["Vc"][:, b:b + 1] - Vc) / (np.abs(Vc) + 0.25))))
        res["kv"].append(kv_err)
        x0 = run["noise"][b:b + 1].astype(np.float64)
        if teacher_forced:
            xk = run["noise"][b:b + 1].astype(np.float32)
            worst = worst_rel = 0.0
            for k in range(c.S):
                v_ref = vel(xk.astype(np.float64), tau[k], Kc, Vc, w, c)
                v_gpu = run["tap"][k, b:b + 1]
                m = O.parity_metrics(v_gpu, v_ref)
                worst = max(worst, m["e_inf"])
                worst_rel = max(worst_rel, m["e_rel"])
                xk = (xk + np.float32(tau[k + 1] - tau[k]) * v_gpu).astype(np.float32)
            res["v_tf"].append(worst)
            res.setdefault("v_tf_rel", []).append(worst_rel)
        if free_running:
            xs, _ = O.denoise(x0, Kc, Vc, w, c, vel=vel)
            res["x"].append(O.parity_metrics(run["act"][b:b + 1], xs))
    return res
