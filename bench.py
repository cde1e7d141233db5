#!/usr/bin/env python
"""Benchmark of the prefix-cached flow-matching action expert on GB300.

One step = one whole request of the hot path over one batch of synthetic
input: the prefix K/V cache build (Eq. 2 of "vla.cpp: A Unified Inference
Runtime for Vision-Language-Action Models", §III-B) followed by the S-step
Euler solve of the action chunk (Eq. 1, §III-A), i.e. L_model = P + S E of
Eq. (3).  Metric: action chunks/s (and batch-1 ms per chunk, us per solver
step, fraction of the HBM roofline for the solver).

Default workload: the full-size bf16 expert at batch 1 (P = 816 prefix tokens
of width 2048, 18 layers of width 1024, MLP 4096, 8 query / 1 KV heads of
size 256, H = 50 actions x 32 dims, S = 10 steps).

Multi-GPU: observations are independent, so N ranks run N replicas with no
collective on the data path (weak scaling); the only collectives are the
timing barrier and the max over ranks.

`--impl reference` times the CPU oracle (fp64 numpy, the parity reference)
on the host cores on the same workload, one chunk per step.
"""

from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import CONFIGS, make_observations, make_weights  # noqa: E402

METRIC = "action chunks/s & batch-1 ms per chunk; per-step µs and % of HBM/tensor roofline"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_seed(seed: int, rank: int) -> int:
    """Seed of a replica's observations: every rank solves its own inputs."""
    return seed + 1000 * rank


def max_over_ranks(dist, values, device):
    """Element-wise max of a list of floats over all ranks (the slowest rank
    sets the job's time); the values themselves without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world_size: int, units_per_rank: int, ms: float) -> float:
    """Units every rank processed per second of the slowest rank's time."""
    return world_size * units_per_rank / (ms * 1e-3)


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def _lib_hash() -> str:
    """Hash of the library's CUDA/C++ sources with comments and blank lines
    removed: a change to a kernel changes it, a change to a comment does not."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "prefix_cached_flow_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if not f.endswith((".cu", ".cuh", ".h", ".cpp", ".c")):
            continue  # sources only: stray files (editor backups, caches) do not count
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.split("\n")]
        h.update(f.encode() + b"\0" + "\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def _traffic_from_profile(workload: str):
    """DRAM bytes per solver launch from the committed ncu summary, if it was
    taken on the current sources (else None)."""
    p = os.path.join(ROOT, "profiles", f"solver_{workload}_traffic.txt")
    try:
        kv = {}
        with open(p) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("library_sources_sha256_16") != _lib_hash():
            return None
        return float(kv["dram_bytes_per_solver_launch"])
    except Exception:
        return None


def algorithmic_bytes_per_step(cfg) -> float:
    """Bytes one Euler step must move at least: every token-dependent weight
    once plus the K/V cache once (activations and the time table excluded)."""
    wb = 2 if cfg.dtype == "bf16" else 4
    if cfg.w2a8:
        per_layer = ((cfg.qdim + 2 * cfg.kvdim) * cfg.D + cfg.D * cfg.qdim + 2 * cfg.D * cfg.F) // 4
        weights = cfg.L * per_layer + 2 * cfg.D * cfg.d_a * 2
    else:
        weights = cfg.token_dependent_params() * wb
    kv = 2 * cfg.L * cfg.B * cfg.n_kv * cfg.P * cfg.d_h * wb
    return float(weights + kv)


def algorithmic_flops_per_step(cfg) -> float:
    """Tensor-core work of one Euler step: every token-dependent linear map
    (2 T N K, ternary MACs counted at the bf16 rate) plus the joint attention
    (4 T n_q (P + H) d_h per layer)."""
    T = cfg.B * cfg.H
    lin = 2.0 * T * cfg.token_dependent_params()
    attn = 4.0 * T * cfg.n_q * (cfg.P + cfg.H) * cfg.d_h * cfg.L
    return lin + attn


def config_dict(cfg, ws=1):
    """The `config` object of a bench line (the same keys on both arms)."""
    return {"workload": cfg.name, "B": cfg.B, "P": cfg.P, "S": cfg.S, "L": cfg.L, "D": cfg.D, "F": cfg.F,
            "heads": f"{cfg.n_q}q/{cfg.n_kv}kv x {cfg.d_h}", "H": cfg.H, "d_a": cfg.d_a,
            "d_vlm": cfg.d_vlm, "global_batch": ws * cfg.B, "parallelism": f"replicas x{ws}",
            "l2": "flushed (256 MiB write) between timed steps"}


def roofline(cfg, denoise_ms, traffic=None):
    """Roofline of the solver launch: algorithmic bytes (or tensor FLOP) of
    the S steps over its measured time, against the measured peak."""
    hbm, tflops, tflops_sus, src = _peaks()
    solver_bytes = cfg.S * algorithmic_bytes_per_step(cfg)
    solver_flops = cfg.S * algorithmic_flops_per_step(cfg)
    # The solver launch runs for milliseconds back to back: the sustained
    # tensor peak applies to it.  Bound = whichever roof takes longer.
    if solver_flops / (tflops_sus * 1e12) > solver_bytes / (hbm * 1e9):
        roof = {"bound": "tensor", "achieved": solver_flops / (denoise_ms * 1e-3) / 1e12, "peak": tflops_sus,
                "unit": "TFLOP/s", "algorithmic_flops_per_launch": solver_flops,
                "peak_note": "bf16 sustained"}
    else:
        roof = {"bound": "hbm", "achieved": solver_bytes / (denoise_ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof.update({"traffic": traffic, "algorithmic_bytes_per_launch": solver_bytes, "peak_source": src})
    return roof


def prefix_roofline(cfg, prefix_ms):
    """The prefix K/V build (one GEMM over every layer): tensor-bound."""
    _, tflops, _, src = _peaks()
    flops = 2.0 * cfg.B * cfg.P * cfg.d_vlm * cfg.L * 2 * cfg.kvdim
    ach = flops / (prefix_ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": ach, "peak": tflops, "unit": "TFLOP/s", "frac": ach / tflops,
            "algorithmic_flops_per_launch": flops, "peak_note": "bf16 burst", "peak_source": src}


def time_request(ex, Zt, Kc, Vc, nt, act, steps, flush, stream):
    """CUDA-event times (ms) of the prefix build and the solve, per step, with
    an L2 flush between timed steps (outside the events)."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush.random_(0, 255)
        e0, e1, e2 = ev[i]
        e0.record(stream)
        ex.prefix_kv_build(Zt, Kc, Vc)
        e1.record(stream)
        ex.denoise(Kc, Vc, nt, act)
        e2.record(stream)
    torch.cuda.synchronize()
    prefix_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    denoise_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    return prefix_ms, denoise_ms


def sub_workload(name, steps, flush, stream):
    """Device-timed numbers of one more workload (same method as the main line)."""
    import torch

    import prefix_cached_flow_gb300 as V
    cfg = CONFIGS[name]
    w = make_weights(cfg)
    Z, noise = make_observations(cfg, cfg.B)
    ex = V.Expert(cfg, V.upload_weights(w, cfg.dtype, cfg.w2a8), max_batch=cfg.B, max_prefix=cfg.P)
    del w
    dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    Zt = torch.from_numpy(Z).to(dt).cuda()
    nt = torch.from_numpy(noise).cuda()
    act = torch.empty_like(nt)
    Kc, Vc = ex.alloc_cache(cfg.B, cfg.P)
    for _ in range(3):
        ex.prefix_kv_build(Zt, Kc, Vc)
        ex.denoise(Kc, Vc, nt, act)
    torch.cuda.synchronize()
    prefix_ms, denoise_ms = time_request(ex, Zt, Kc, Vc, nt, act, steps, flush, stream)
    status = ex.poll_status()
    out = {"config": config_dict(cfg), "value": cfg.B / ((prefix_ms + denoise_ms) * 1e-3), "unit": "chunks/s",
           "ms_per_request": prefix_ms + denoise_ms, "prefix_build_ms": prefix_ms, "denoise_ms": denoise_ms,
           "us_per_solver_step": denoise_ms * 1e3 / cfg.S, "roofline": roofline(cfg, denoise_ms),
           "prefix_roofline": prefix_roofline(cfg, prefix_ms),
           "gpu_launches_per_request": 1 + ex.launch_count(cfg.B, cfg.P), "steps": steps,
           "device_status": status}
    ex.close()
    return out


def cpu_oracle_chunk(cfg, w, Z, noise):
    import oracle as O
    Kc, Vc = O.prefix_kv(Z.astype(np.float64), w, cfg)
    if cfg.w2a8:
        return O.denoise_w2a8(noise.astype(np.float64), Kc, Vc, w, cfg)[0]
    return O.denoise(noise.astype(np.float64), Kc, Vc, w, cfg)[0]


def _host_threads() -> int:
    """Threads the oracle's BLAS uses: its thread variable if set, else the
    cores this process may run on."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return int(v)
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _cpu_model(info: str | None = None) -> str:
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: the
    implementer / part codes), else the machine type."""
    try:
        if info is None:
            with open("/proc/cpuinfo") as f:
                info = f.read()
        for key in ("model name", "Model name"):
            m = re.search(rf"^{key}\s*:\s*(.+)$", info, flags=re.M)
            if m:
                return m.group(1).strip()
        imp = re.search(r"^CPU implementer\s*:\s*(\S+)", info, flags=re.M)
        part = re.search(r"^CPU part\s*:\s*(\S+)", info, flags=re.M)
        if imp and part:
            return f"{platform.machine()} implementer {imp.group(1)} part {part.group(1)}"
    except OSError:
        pass
    return platform.machine()


def cpu_baseline(cfg, w, Z, noise, budget_s=10.0):
    """Oracle throughput on the host cores on a bounded sample: whole chunks
    of observation 0, repeated until ~budget_s of CPU work."""
    c1 = cfg.replace(B=1)
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        cpu_oracle_chunk(c1, w, Z[:1], noise[:1])
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > budget_s:
            break
    mean = sum(times) / len(times)
    return {"value": 1.0 / mean, "unit": "chunks/s", "cores": _host_threads(), "cpu": _cpu_model(), "kind": "oracle",
            "sample": f"{len(times)} whole chunk(s) (prefix K/V + {cfg.S} Euler steps) of observation 0 of "
                      f"{cfg.name}, fp64 numpy/OpenBLAS, {mean * 1e3:.0f} ms per chunk"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    cfg = CONFIGS[args.workload]
    if args.solver_steps:
        cfg = cfg.replace(S=args.solver_steps)
    w = make_weights(cfg)
    if cfg.w2a8:
        import oracle as O
        w = O.with_unpacked(w)
    Z, noise = make_observations(cfg, 1)
    c1 = cfg.replace(B=1)
    for _ in range(args.warmup):
        cpu_oracle_chunk(c1, w, Z, noise)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_oracle_chunk(c1, w, Z, noise)
    dt = (time.perf_counter() - t0) / args.steps
    value = 1.0 / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "chunks/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(config_dict(cfg.replace(B=1)), note="one observation per step"),
        "cpu_baseline": {"value": value, "unit": "chunks/s", "cores": _host_threads(), "cpu": _cpu_model(),
                         "kind": "oracle",
                         "sample": f"{args.steps} whole chunks of observation 0 of {cfg.name} (prefix K/V + "
                                   f"{cfg.S} Euler steps), fp64 numpy/OpenBLAS"},
        "e2e": {"value": value, "unit": "chunks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def eq3_sweep(cfg, dev_w, Zt, nt, steps=(1, 2, 4, 8, 16), reps=20):
    """Solver-step sweep of the latency model L(T) = P + T E ("vla.cpp", §III-B
    Eq. (3)): P = prefix K/V build, E = one Euler step, fitted by least squares
    over T, and the speedup over recomputing the conditioning every step,
    T (P + E) / (P + T E)."""
    import torch

    import prefix_cached_flow_gb300 as V
    rows = []
    for S in steps:
        ex = V.Expert(cfg, dev_w, max_batch=cfg.B, max_prefix=cfg.P, n_steps=S)
        Kc, Vc = ex.alloc_cache(cfg.B, cfg.P)
        act = torch.empty_like(nt)
        for _ in range(3):
            ex.prefix_kv_build(Zt, Kc, Vc)
            ex.denoise(Kc, Vc, nt, act)
        torch.cuda.synchronize()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        tp = td = 0.0
        for _ in range(reps):
            e[0].record()
            ex.prefix_kv_build(Zt, Kc, Vc)
            e[1].record()
            ex.denoise(Kc, Vc, nt, act)
            e[2].record()
            torch.cuda.synchronize()
            tp += e[0].elapsed_time(e[1])
            td += e[1].elapsed_time(e[2])
        rows.append((S, tp / reps, td / reps))
        ex.close()
    Ts = np.array([r[0] for r in rows], dtype=np.float64)
    L = np.array([r[1] + r[2] for r in rows])
    A = np.stack([np.ones_like(Ts), Ts], axis=1)
    (P_fit, E_fit), *_ = np.linalg.lstsq(A, L, rcond=None)
    P_meas = float(np.mean([r[1] for r in rows]))
    return {
        "T": [int(t) for t in Ts], "prefix_ms": [round(r[1], 4) for r in rows],
        "solve_ms": [round(r[2], 4) for r in rows], "fit_P_ms": float(P_fit), "fit_E_ms": float(E_fit),
        "prefix_ms_measured": P_meas,
        "speedup_vs_recompute": [float(t * (P_meas + E_fit) / (P_meas + t * E_fit)) for t in Ts],
    }


def run_ours(args):
    import torch

    import prefix_cached_flow_gb300 as V

    ws, rank, local = _dist()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if not os.path.exists(V.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    cfg = CONFIGS[args.workload]
    if args.solver_steps:
        cfg = cfg.replace(S=args.solver_steps)
    B = cfg.B
    w = make_weights(cfg)
    Z, noise = make_observations(cfg.replace(seed=replica_seed(cfg.seed, rank)), B)
    ex = V.Expert(cfg, V.upload_weights(w, cfg.dtype, cfg.w2a8), max_batch=B, max_prefix=cfg.P)
    dt = torch.float32 if cfg.dtype == "f32" else torch.bfloat16
    Zt = torch.from_numpy(Z).to(dt).cuda()
    nt = torch.from_numpy(noise).cuda()
    act = torch.empty_like(nt)
    Kc, Vc = ex.alloc_cache(B, cfg.P)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        ex.prefix_kv_build(Zt, Kc, Vc)
        ex.denoise(Kc, Vc, nt, act)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert ex.poll_status() == 0

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    prefix_ms, denoise_ms = time_request(ex, Zt, Kc, Vc, nt, act, args.steps, flush, stream)
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    status = ex.poll_status()
    step_ms = prefix_ms + denoise_ms
    step_ms, prefix_ms, denoise_ms = max_over_ranks(dist, [step_ms, prefix_ms, denoise_ms], "cuda")

    # End to end through the public host-buffer call: H2D of Z and noise, the
    # whole request, D2H of the chunk, every step.
    Zh = torch.from_numpy(Z).to(dt).pin_memory()
    nh = torch.from_numpy(noise).pin_memory()
    ah = torch.empty_like(nh).pin_memory()
    for _ in range(3):
        ex.policy_step_host(Zh, nh, ah)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ex.policy_step_host(Zh, nh, ah)
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    (e2e_ms,) = max_over_ranks(dist, [e2e_ms], "cuda")

    roof = roofline(cfg, denoise_ms, _traffic_from_profile(cfg.name))
    roof["kernel"] = "solver launch (all S steps)"
    launches = args.steps * (1 + ex.launch_count(B, cfg.P))
    line = {
        "metric": METRIC,
        "value": whole_job_rate(ws, B, step_ms),
        "unit": "chunks/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": config_dict(cfg, ws),
        "ms_per_chunk": step_ms / 1.0,
        "prefix_build_ms": prefix_ms,
        "denoise_ms": denoise_ms,
        "us_per_solver_step": denoise_ms * 1e3 / cfg.S,
        "roofline": roof,
        "prefix_roofline": prefix_roofline(cfg, prefix_ms),
        "e2e": {"value": whole_job_rate(ws, B, e2e_ms), "unit": "chunks/s",
                "h2d_bytes_per_step": int(Zh.numel() * Zh.element_size() + nh.numel() * 4),
                "d2h_bytes_per_step": int(ah.numel() * 4)},
        "gpu_launches": launches,
        "clocks": clocks,
        "device_status": status,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, w, Z, noise)
    if not args.only and rank == 0 and ws == 1:
        line["eq3"] = eq3_sweep(cfg, V.upload_weights(w, cfg.dtype, cfg.w2a8), Zt, nt)
        subs = {}
        for name in ("full_bf16_b64", "w2a8_b1", "w2a8_b16"):
            if name != cfg.name:
                subs[name] = sub_workload(name, max(5, min(args.steps, 10)), flush, stream)
        line["workloads"] = subs
    if rank == 0:
        print(json.dumps(line), flush=True)
    ex.close()
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="full_bf16_b1", choices=sorted(CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", action="store_true",
                    help="time the chosen workload alone (no Eq. (3) sweep, no other workloads)")
    ap.add_argument("--solver-steps", type=int, default=0,
                    help="override the workload's number of Euler steps S (0: the workload's own)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
