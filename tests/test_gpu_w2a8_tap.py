"""Operation-by-operation parity of the W2A8 solver on its own intermediate
tensors ("vla.cpp: A Unified Inference Runtime for Vision-Language-Action
Models", §III-D Eq. (4); §III-E: intermediate tensors localise discrepancies).

The library records every layer of one solver step (vla_expert_set_w2a8_tap):
the fp32 rows each Eq. (4) quantiser received, the codes and row scales it
produced, the exact accumulators of every ternary map, the bf16 outputs, the
attention and GeLU outputs and the residual stream.  Each operation is then
checked against the oracle fed with the GPU's own inputs of that operation:

* quantiser (the solver's own kernels, the norm-fused one and the row one):
  codes and alpha bits equal to oracle.quantize_rows of the tapped fp32 rows;
* ternary maps (every solver epilogue: the QKV scatter, the residual add and
  the GeLU): int32 accumulators equal to the int64 brute force of the tapped
  codes against the packed weights, bf16 outputs equal bit for bit, residual
  updates equal to the fp32 sum h + y bit for bit;
* the floating-point steps between them (modulated RMSNorm, attention,
  GeLU) within fp32 / bf16 rounding of the oracle's definition.
"""

import numpy as np
import pytest

import oracle as O
from _harness import weights
from workloads import CONFIGS, make_observations

pytestmark = pytest.mark.gpu


def _bf16_bits(x):
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _run_tapped(cfg, step):
    import torch

    import prefix_cached_flow_gb300 as V
    w = weights(cfg)
    Z, noise = make_observations(cfg, cfg.B)
    ex = V.Expert(cfg, V.upload_weights(w, cfg.dtype, True), max_batch=cfg.B, max_prefix=cfg.P)
    Kc, Vc = ex.alloc_cache(cfg.B, cfg.P)
    ex.prefix_kv_build(torch.from_numpy(Z).to(torch.bfloat16).cuda(), Kc, Vc)
    ex.set_w2a8_tap(step)
    tap = torch.empty((cfg.S, cfg.B, cfg.H, cfg.d_a), dtype=torch.float32, device="cuda")
    ex.denoise(Kc, Vc, torch.from_numpy(noise).cuda(), vel_tap=tap)
    torch.cuda.synchronize()
    assert ex.poll_status() == 0
    recs = ex.w2a8_tap_views(cfg.B)
    ex.set_w2a8_tap(None)
    kc = Kc.float().cpu().numpy().astype(np.float64)
    vc = Vc[..., :cfg.P].transpose(-1, -2).float().cpu().numpy().astype(np.float64)
    x = noise.astype(np.float32)
    velo = tap.cpu().numpy()
    tau = O.schedule(cfg.S)
    for k in range(step):  # the solver state entering the tapped step, as the GPU had it
        x = (x + np.float32(tau[k + 1] - tau[k]) * velo[k]).astype(np.float32)
    return w, recs, kc, vc, x, tau[step]


def _check_quant(u, codes, alpha):
    a_ref, al_ref = O.quantize_rows(u)
    assert np.array_equal(alpha.view(np.uint32), al_ref.view(np.uint32)), "alpha bits"
    assert np.array_equal(codes.astype(np.int64), a_ref.astype(np.int64)), "codes"
    return a_ref, al_ref


def _ternary(w, name, l, a, alpha, beta):
    y, acc = O.ternary_linear(a, alpha, None, beta, q=w["q_" + name][l])
    return y, acc


@pytest.mark.parametrize("name,step,group", [("w2a8_b1", 1, 0), ("w2a8_b16", 3, 0), ("w2a8_b1", 2, 128)])
def test_w2a8_solver_ops_bit_exact(name, step, group):
    """group > 0: one weight scale per group of that many output rows."""
    cfg = CONFIGS[name].replace(beta_group=group)
    w, recs, kc, vc, x, tau = _run_tapped(cfg, step)
    B, H, D = cfg.B, cfg.H, cfg.D
    T = B * H
    per_layer, _ = O.time_conditioning(w, cfg, tau)
    # layer 0 input: x W_in^T (fp32 on the GPU)
    h0 = O.linear(x.reshape(T, -1), w["win"])
    assert np.max(np.abs(recs[0]["h_in"] - h0)) <= 1e-5 * (1 + np.max(np.abs(h0)))
    worst_u = worst_o = worst_g = 0.0
    for l, r in enumerate(recs):
        if l > 0:
            assert np.array_equal(r["h_in"], recs[l - 1]["h_out"])
        ga, ba, gm, bm = per_layer[l]
        # attention branch: modulated norm -> Eq. (4) -> [W_q; W_k; W_v]
        u_ref = O.rmsnorm_modulate(r["h_in"].astype(np.float64), ga, ba, cfg.eps)
        worst_u = max(worst_u, float(np.max(np.abs(r["u_a"] - u_ref) / (1 + np.abs(u_ref)))))
        a, al = _check_quant(r["u_a"], r["c_a"], r["al_a"])
        acc = {}
        yq = {}
        for nm in ("wq", "wk", "wv"):
            yq[nm], acc[nm] = _ternary(w, nm, l, a, al, w["beta_" + nm][l])
        assert np.array_equal(r["acc_qkv"].astype(np.int64), np.concatenate([acc["wq"], acc["wk"], acc["wv"]], 1))
        q = yq["wq"].reshape(B, H, cfg.n_q, cfg.d_h).transpose(0, 2, 1, 3)
        ks = yq["wk"].reshape(B, H, cfg.n_kv, cfg.d_h).transpose(0, 2, 1, 3)
        vsT = yq["wv"].reshape(B, H, cfg.n_kv, cfg.d_h).transpose(0, 2, 3, 1)
        assert np.array_equal(_bf16_bits(r["q"]), _bf16_bits(q))
        assert np.array_equal(_bf16_bits(r["k_s"]), _bf16_bits(ks))
        assert np.array_equal(_bf16_bits(r["v_sT"][..., :H]), _bf16_bits(vsT))
        # attention on the GPU's own bf16 q, k_s, v_s and cache
        o_ref = O.joint_attention(q.transpose(0, 2, 1, 3).astype(np.float64),
                                  ks.transpose(0, 2, 1, 3).astype(np.float64),
                                  vsT.transpose(0, 3, 1, 2).astype(np.float64), kc[l], vc[l])
        o_ref = o_ref.reshape(T, cfg.qdim)
        worst_o = max(worst_o, float(np.max(np.abs(r["o"] - o_ref))))
        # O-projection: Eq. (4) of the attention output, residual add in fp32
        a, al = _check_quant(r["o"], r["c_o"], r["al_o"])
        y, acc_o = _ternary(w, "wo", l, a, al, w["beta_wo"][l])
        assert np.array_equal(r["acc_o"].astype(np.int64), acc_o)
        assert np.array_equal(r["h_mid"], (r["h_in"] + y).astype(np.float32))
        # MLP: modulated norm -> Eq. (4) -> W_up -> GeLU -> Eq. (4) -> W_down
        u_ref = O.rmsnorm_modulate(r["h_mid"].astype(np.float64), gm, bm, cfg.eps)
        worst_u = max(worst_u, float(np.max(np.abs(r["u_m"] - u_ref) / (1 + np.abs(u_ref)))))
        a, al = _check_quant(r["u_m"], r["c_m"], r["al_m"])
        y, acc_up = _ternary(w, "wup", l, a, al, w["beta_wup"][l])
        assert np.array_equal(r["acc_up"].astype(np.int64), acc_up)
        g_ref = O.gelu(y.astype(np.float64))
        worst_g = max(worst_g, float(np.max(np.abs(r["g"] - g_ref) / (1 + np.abs(y)))))
        a, al = _check_quant(r["g"], r["c_d"], r["al_d"])
        y, acc_d = _ternary(w, "wdown", l, a, al, w["beta_wdown"][l])
        assert np.array_equal(r["acc_d"].astype(np.int64), acc_d)
        assert np.array_equal(r["h_out"], (r["h_mid"] + y).astype(np.float32))
    print(name, "modnorm", worst_u, "attention abs", worst_o, "gelu", worst_g)
    # fp32 modulated norm (with the fp32 time-conditioning table) and fp32
    # GeLU (erff: a few ulp), both relative to 1 + |value|; attention from
    # bf16 operands with an fp32 softmax and bf16 probabilities
    assert worst_u <= 1e-5
    assert worst_g <= 2e-6
    assert worst_o <= 1e-2
