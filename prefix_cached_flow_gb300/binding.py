"""ctypes binding of libvla (include/vla.h): argument marshalling only.

Every operation runs in the CUDA library; this module turns torch tensors
into device pointers and the current torch stream into the `stream` argument,
and raises VlaError for a non-OK status.  If libvla.so has not been built it
raises at import of the library -- there is no other implementation to fall
back to.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libvla.so")

VLA_OK = 0
STATUS_NAMES = {0: "VLA_OK", 1: "VLA_ERR_INVALID_ARG", 2: "VLA_ERR_SHAPE", 3: "VLA_ERR_UNSUPPORTED",
                4: "VLA_ERR_OOM", 5: "VLA_ERR_CUDA", 6: "VLA_ERR_TIMEOUT", 7: "VLA_ERR_ABORTED",
                8: "VLA_ERR_NO_DEVICE"}
DTYPE_F32, DTYPE_BF16 = 0, 1
FLAG_SIMT_GEMM, FLAG_NO_GRAPH, FLAG_ATTN_SPLIT, FLAG_ATTN_STREAM = 1, 2, 4, 8
FLAG_LINEAR_SPLIT, FLAG_LINEAR_WIDE, FLAG_PERSIST = 16, 32, 64

EXPORTED = ("vla_expert_create", "vla_expert_create_w2a8", "vla_expert_destroy", "vla_prefix_cache_bytes",
            "vla_prefix_kv_build", "vla_action_denoise", "vla_action_denoise_w2a8", "vla_policy_step_host",
            "vla_expert_poll_status", "vla_expert_set_abort", "vla_w2a8_quantize_rows",
            "vla_w2a8_ternary_gemm", "vla_expert_launch_count", "vla_status_string", "vla_version", "vla_last_error",
            "vla_expert_set_wait_limit", "vla_expert_check_wait_timeout", "vla_expert_w2a8_tap_bytes",
            "vla_expert_set_w2a8_tap", "vla_debug_gelu_forms", "vla_action_denoise_ex", "vla_noise_fill",
            "vla_expert_select_ffn")


class VlaError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class VlaConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layers", "width", "mlp_width", "n_q_heads", "n_kv_heads", "head_dim", "vlm_hidden", "action_dim",
        "horizon", "time_dim", "max_batch", "max_prefix", "dtype")] + [("rms_eps", ctypes.c_float),
                                                                         ("flags", ctypes.c_uint),
                                                                         ("schedule", ctypes.c_int),
                                                                         ("cross_every", ctypes.c_int)]


DENSE_FIELDS = ("wk_pre", "wv_pre", "wq", "wk", "wv", "wo", "wup", "wdown", "wmod", "win", "wout", "wt1", "wt2",
                "wmod_f")
W2A8_FIELDS = ("wk_pre", "wv_pre", "wq", "wk", "wv", "wo", "wup", "wdown", "beta_wq", "beta_wk", "beta_wv",
               "beta_wo", "beta_wup", "beta_wdown", "wmod", "win", "wout", "wt1", "wt2", "wmod_f")


class VlaRequest(ctypes.Structure):
    _fields_ = [("prefix_mask_dev", ctypes.c_void_p), ("noise_dev", ctypes.c_void_p), ("seed", ctypes.c_ulonglong),
                ("noise_out_dev", ctypes.c_void_p)]


class VlaWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in DENSE_FIELDS]


W2A8_PREFIX_FIELDS = ("wk_pre_t", "wv_pre_t", "beta_wk_pre", "beta_wv_pre")


class VlaWeightsW2A8(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in W2A8_FIELDS] + [("beta_group", ctypes.c_int)] + [
        (n, ctypes.c_void_p) for n in W2A8_PREFIX_FIELDS]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libvla.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libvla is not built ({LIB_PATH} missing); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sig = {
        "vla_expert_create": [ctypes.POINTER(VlaConfig), ctypes.POINTER(VlaWeights), ci, vp, ctypes.POINTER(vp)],
        "vla_expert_create_w2a8": [ctypes.POINTER(VlaConfig), ctypes.POINTER(VlaWeightsW2A8), ci, vp,
                                   ctypes.POINTER(vp)],
        "vla_prefix_cache_bytes": [vp, ci, ci, ctypes.POINTER(ctypes.c_size_t)],
        "vla_prefix_kv_build": [vp, vp, ci, ci, vp, vp, vp],
        "vla_action_denoise": [vp, vp, vp, ci, ci, vp, vp, vp, vp],
        "vla_action_denoise_w2a8": [vp, vp, vp, ci, ci, vp, vp, vp, vp],
        "vla_policy_step_host": [vp, vp, ci, ci, vp, vp, vp],
        "vla_expert_poll_status": [vp, vp],
        "vla_expert_set_abort": [vp, ci],
        "vla_w2a8_quantize_rows": [vp, ci, ci, vp, vp, vp],
        "vla_w2a8_ternary_gemm": [vp, vp, vp, cf, ci, ci, ci, vp, vp, vp],
        "vla_expert_launch_count": [vp, ci, ci, ctypes.POINTER(ci)],
        "vla_expert_set_wait_limit": [vp, ctypes.c_ulonglong],
        "vla_expert_check_wait_timeout": [vp, vp],
        "vla_expert_w2a8_tap_bytes": [vp, ci, ctypes.POINTER(ctypes.c_size_t)],
        "vla_expert_set_w2a8_tap": [vp, ci, vp, ctypes.c_size_t],
        "vla_debug_gelu_forms": [vp, ci, vp, vp, vp],
        "vla_action_denoise_ex": [vp, vp, vp, ci, ci, ctypes.POINTER(VlaRequest), vp, vp, vp],
        "vla_noise_fill": [ctypes.c_ulonglong, ctypes.c_size_t, vp, vp],
        "vla_expert_select_ffn": [vp, vp, ci, vp],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ci
    L.vla_expert_destroy.argtypes = [vp]
    L.vla_expert_destroy.restype = None
    L.vla_status_string.argtypes = [ci]
    L.vla_status_string.restype = ctypes.c_char_p
    L.vla_version.argtypes = []
    L.vla_version.restype = ctypes.c_char_p
    L.vla_last_error.argtypes = []
    L.vla_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(status: int, where: str):
    if status != VLA_OK:
        detail = lib().vla_last_error().decode(errors="replace")
        raise VlaError(status, f"{where} [{detail}]" if detail else where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(dt: str):
    return torch.float32 if dt == "f32" else torch.bfloat16


def upload_weights(w: dict, dtype: str, w2a8: bool, device="cuda") -> dict:
    """numpy weight dict (workload layout) -> contiguous device tensors.

    Dense weights become the config dtype; packed ternary codes stay uint8 and
    per-tensor scales fp32.  Values are transferred, not changed (bf16 inputs
    are already bf16-representable)."""
    out = {}
    for k, v in w.items():
        if k not in DENSE_FIELDS and k not in W2A8_FIELDS and k not in ("beta_wk_pre", "beta_wv_pre"):
            continue
        t = torch.from_numpy(v)
        if t.dtype == torch.float32 and not k.startswith("beta_"):
            t = t.to(_dtype(dtype))
        out[k] = t.contiguous().to(device)
    return out


class Expert:
    """An expert handle (vla_expert*): fixed shapes, solver length and weights."""

    def __init__(self, cfg, weights: dict, max_batch: int | None = None, max_prefix: int | None = None,
                 flags: int = 0, n_steps: int | None = None, stream=None):
        self.cfg = cfg
        self.w2a8 = bool(cfg.w2a8)
        self.S = cfg.S if n_steps is None else n_steps
        self.dtype = _dtype(cfg.dtype)
        c = VlaConfig(n_layers=cfg.L, width=cfg.D, mlp_width=cfg.F, n_q_heads=cfg.n_q, n_kv_heads=cfg.n_kv,
                      head_dim=cfg.d_h, vlm_hidden=cfg.d_vlm, action_dim=cfg.d_a, horizon=cfg.H, time_dim=cfg.d_t,
                      max_batch=max_batch or cfg.B, max_prefix=max_prefix or cfg.P,
                      dtype=DTYPE_F32 if cfg.dtype == "f32" else DTYPE_BF16, rms_eps=cfg.eps, flags=flags,
                      schedule=1 if getattr(cfg, "reverse", False) else 0,
                      cross_every=int(getattr(cfg, "cross_every", 0)))
        self._c = c
        h = ctypes.c_void_p()
        if self.w2a8:
            fields = {n: weights[n].data_ptr() for n in W2A8_FIELDS if n in weights}
            if weights["wk_pre"].dtype == torch.uint8:  # ternary prefix maps
                fields.update(wk_pre_t=weights["wk_pre"].data_ptr(), wv_pre_t=weights["wv_pre"].data_ptr(),
                              beta_wk_pre=weights["beta_wk_pre"].data_ptr(),
                              beta_wv_pre=weights["beta_wv_pre"].data_ptr(), wk_pre=0, wv_pre=0)
            ws = VlaWeightsW2A8(**fields, beta_group=int(getattr(cfg, "beta_group", 0)))
            st = lib().vla_expert_create_w2a8(ctypes.byref(c), ctypes.byref(ws), self.S, _stream(stream),
                                              ctypes.byref(h))
        else:
            ws = VlaWeights(**{n: weights[n].data_ptr() for n in DENSE_FIELDS})
            st = lib().vla_expert_create(ctypes.byref(c), ctypes.byref(ws), self.S, _stream(stream),
                                         ctypes.byref(h))
        _check(st, "vla_expert_create")
        self._h = h

    # -- cache ------------------------------------------------------------
    def cache_bytes(self, B: int, P: int) -> int:
        n = ctypes.c_size_t()
        _check(lib().vla_prefix_cache_bytes(self._h, B, P, ctypes.byref(n)), "vla_prefix_cache_bytes")
        return n.value

    def alloc_cache(self, B: int, P: int):
        """K_C [L, B, n_kv, P, d_h] and V_C stored transposed [L, B, n_kv, d_h, P8]
        (P8 = P rounded up to a multiple of 8)."""
        c = self.cfg
        p8 = (P + 7) // 8 * 8
        return (torch.empty((c.L, B, c.n_kv, P, c.d_h), dtype=self.dtype, device="cuda"),
                torch.empty((c.L, B, c.n_kv, c.d_h, p8), dtype=self.dtype, device="cuda"))

    def prefix_kv_build(self, Z, Kc, Vc, stream=None):
        B, P = Z.shape[0], Z.shape[1]
        _check(lib().vla_prefix_kv_build(self._h, _ptr(Z), B, P, _ptr(Kc), _ptr(Vc), _stream(stream)),
               "vla_prefix_kv_build")

    # -- solver -----------------------------------------------------------
    def denoise(self, Kc, Vc, noise, actions=None, vel_tap=None, stream=None):
        B = noise.shape[0]
        P = Kc.shape[3]  # K_C is [L, B, n_kv, P, d_h]
        if actions is None:
            actions = torch.empty_like(noise)
        fn = lib().vla_action_denoise_w2a8 if self.w2a8 else lib().vla_action_denoise
        _check(fn(self._h, _ptr(Kc), _ptr(Vc), B, P, _ptr(noise), _ptr(actions), _ptr(vel_tap), _stream(stream)),
               "vla_action_denoise")
        return actions

    def denoise_ex(self, Kc, Vc, B, prefix_mask=None, noise=None, seed=0, noise_out=None, actions=None,
                   vel_tap=None, stream=None):
        """Eq. 1 with request options: prefix_mask uint32 [B, ceil(P/32)]
        (device), noise (device) or None for in-library noise from `seed`."""
        c = self.cfg
        P = Kc.shape[3]
        if actions is None:
            actions = torch.empty((B, c.H, c.d_a), dtype=torch.float32, device="cuda")
        req = VlaRequest(prefix_mask_dev=None if prefix_mask is None else prefix_mask.data_ptr(),
                         noise_dev=None if noise is None else noise.data_ptr(), seed=int(seed),
                         noise_out_dev=None if noise_out is None else noise_out.data_ptr())
        _check(lib().vla_action_denoise_ex(self._h, _ptr(Kc), _ptr(Vc), B, P, ctypes.byref(req), _ptr(actions),
                                           _ptr(vel_tap), _stream(stream)), "vla_action_denoise_ex")
        return actions

    def policy_step_host(self, Z_host, noise_host, actions_host, stream=None):
        B, P = Z_host.shape[0], Z_host.shape[1]
        _check(lib().vla_policy_step_host(self._h, _ptr(Z_host), B, P, _ptr(noise_host), _ptr(actions_host),
                                          _stream(stream)), "vla_policy_step_host")
        return actions_host

    def select_ffn(self, idx=None, stream=None):
        """Evaluate only the FFN neurons idx (int32 [L, F_sel] on the device);
        None restores the full MLP."""
        if idx is None:
            _check(lib().vla_expert_select_ffn(self._h, None, 0, _stream(stream)), "vla_expert_select_ffn")
        else:
            _check(lib().vla_expert_select_ffn(self._h, _ptr(idx), idx.shape[1], _stream(stream)),
                   "vla_expert_select_ffn")

    def launch_count(self, B: int, P: int) -> int:
        n = ctypes.c_int()
        _check(lib().vla_expert_launch_count(self._h, B, P, ctypes.byref(n)), "vla_expert_launch_count")
        return n.value

    def poll_status(self, stream=None) -> int:
        return lib().vla_expert_poll_status(self._h, _stream(stream))

    def set_abort(self, flag: bool):
        _check(lib().vla_expert_set_abort(self._h, 1 if flag else 0), "vla_expert_set_abort")

    def set_wait_limit(self, ns: int):
        _check(lib().vla_expert_set_wait_limit(self._h, int(ns)), "vla_expert_set_wait_limit")

    def check_wait_timeout(self, stream=None):
        _check(lib().vla_expert_check_wait_timeout(self._h, _stream(stream)), "vla_expert_check_wait_timeout")

    # -- W2A8 diagnostic tap ----------------------------------------------
    TAP_NAMES = ("h_in", "u_a", "c_a", "al_a", "acc_qkv", "q", "k_s", "v_sT", "o", "c_o", "al_o", "acc_o", "h_mid",
                 "u_m", "c_m", "al_m", "acc_up", "g", "c_d", "al_d", "acc_d", "h_out")

    def set_w2a8_tap(self, step: int | None, B: int | None = None):
        """Start recording solver step `step` of later W2A8 calls (None stops).
        Returns the raw uint8 device buffer; decode it with w2a8_tap_views()."""
        if step is None:
            _check(lib().vla_expert_set_w2a8_tap(self._h, 0, None, 0), "vla_expert_set_w2a8_tap")
            self._tap = None
            return None
        n = ctypes.c_size_t()
        _check(lib().vla_expert_w2a8_tap_bytes(self._h, self._c.max_batch, ctypes.byref(n)),
               "vla_expert_w2a8_tap_bytes")
        buf = torch.zeros(n.value, dtype=torch.uint8, device="cuda")
        _check(lib().vla_expert_set_w2a8_tap(self._h, step, _ptr(buf), n.value), "vla_expert_set_w2a8_tap")
        self._tap = buf
        return buf

    def w2a8_tap_views(self, B: int) -> list:
        """Per layer, a dict of host numpy arrays in the layout vla.h documents."""
        c = self.cfg
        T, D, F = B * c.H, c.D, c.F
        Q, KV = c.n_q * c.d_h, c.n_kv * c.d_h
        Hp = (c.H + 7) // 8 * 8
        f32, bf, i32 = torch.float32, torch.bfloat16, torch.int32
        shapes = [(f32, (T, D)), (f32, (T, D)), (bf, (T, D)), (f32, (T,)), (i32, (T, Q + 2 * KV)),
                  (bf, (B, c.n_q, c.H, c.d_h)), (bf, (B, c.n_kv, c.H, c.d_h)), (bf, (B, c.n_kv, c.d_h, Hp)),
                  (f32, (T, Q)), (bf, (T, Q)), (f32, (T,)), (i32, (T, D)), (f32, (T, D)),
                  (f32, (T, D)), (bf, (T, D)), (f32, (T,)), (i32, (T, F)), (f32, (T, F)), (bf, (T, F)),
                  (f32, (T,)), (i32, (T, D)), (f32, (T, D))]
        n = ctypes.c_size_t()
        _check(lib().vla_expert_w2a8_tap_bytes(self._h, B, ctypes.byref(n)), "vla_expert_w2a8_tap_bytes")
        per_layer = n.value // c.L
        raw = self._tap.cpu()
        out = []
        for l in range(c.L):
            off = l * per_layer
            rec = {}
            for name, (dt, shp) in zip(self.TAP_NAMES, shapes):
                nb = int(np_prod(shp)) * torch.tensor([], dtype=dt).element_size()
                t = raw[off:off + nb].view(dt).reshape(shp)
                rec[name] = t.float().numpy() if dt == bf else t.numpy()
                off += (nb + 255) // 256 * 256
            out.append(rec)
        return out

    def close(self):
        if getattr(self, "_h", None):
            lib().vla_expert_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def np_prod(shape):
    n = 1
    for d in shape:
        n *= int(d)
    return n


def noise_fill(seed: int, n: int, stream=None):
    """The library's seeded X^0 stream: n fp32 normals on the device."""
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    _check(lib().vla_noise_fill(int(seed), n, _ptr(out), _stream(stream)), "vla_noise_fill")
    return out


def gelu_forms(x, stream=None):
    """(erff GeLU, many-token epilogue GeLU) of an fp32 device tensor."""
    n = x.numel()
    exact = torch.empty_like(x)
    fast = torch.empty_like(x)
    _check(lib().vla_debug_gelu_forms(_ptr(x), n, _ptr(exact), _ptr(fast), _stream(stream)), "vla_debug_gelu_forms")
    return exact, fast


def quantize_rows(x, stream=None):
    """Eq. (4) activation quantiser on the GPU: x fp32 [M, K] -> (int8 [M, K], fp32 alpha [M])."""
    M, K = x.shape
    a = torch.empty((M, K), dtype=torch.int8, device=x.device)
    alpha = torch.empty((M,), dtype=torch.float32, device=x.device)
    _check(lib().vla_w2a8_quantize_rows(_ptr(x), M, K, _ptr(a), _ptr(alpha), _stream(stream)),
           "vla_w2a8_quantize_rows")
    return a, alpha


def ternary_gemm(a, alpha, q_packed, beta: float, want_acc: bool = True, stream=None):
    """Eq. (4) scaled ternary product on the GPU -> (bf16 y [M, N], int32 acc [M, N] or None)."""
    M, K = a.shape
    N = q_packed.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    acc = torch.empty((M, N), dtype=torch.int32, device=a.device) if want_acc else None
    _check(lib().vla_w2a8_ternary_gemm(_ptr(a), _ptr(alpha), _ptr(q_packed), float(beta), M, N, K, _ptr(y),
                                       _ptr(acc), _stream(stream)), "vla_w2a8_ternary_gemm")
    return y, acc
