"""The benchmark's algorithmic work per Euler step, against figures worked out
by hand from the workload shapes (no GPU needed).

The roofline fractions the benchmark reports divide these numbers by the
measured time, so a mistake here (a map left out, a K/V head miscounted, the
ternary weights counted at 16 bits) would silently scale every fraction.
Shapes follow "vla.cpp: A Unified Inference Runtime for Vision-Language-Action
Models" (§III-B: one cached K/V per layer, re-read every step; §III-D: 2-bit
packed ternary weights), with the configurations' sizes.
"""

import importlib.util
import os

import pytest

from workloads import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_full_size_step_bytes(bench):
    # 18 layers x (QKV 2560x1024 + O 1024x2048 + up 4096x1024 + down 1024x4096)
    # bf16, plus W_in and W_out (1024 x 32 each), plus the K/V cache read once:
    # 18 x 2 x 816 x 256 values per tensor pair, bf16.
    weights = (18 * (2560 * 1024 + 1024 * 2048 + 4096 * 1024 + 1024 * 4096) + 2 * 1024 * 32) * 2
    cache = 2 * 18 * 816 * 256 * 2
    assert weights == 471_990_272
    assert bench.algorithmic_bytes_per_step(CONFIGS["full_bf16_b1"]) == weights + cache
    assert abs((weights + cache) / 1e6 - 487.03) < 0.01


def test_batched_step_flops(bench):
    # 3200 tokens: 2 T (token-dependent parameters) + attention 4 T n_q (P + H) d_h per layer
    T = 64 * 50
    params = 18 * (2560 * 1024 + 1024 * 2048 + 4096 * 1024 + 1024 * 4096) + 2 * 1024 * 32
    attn = 4 * T * 8 * (816 + 50) * 256 * 18
    flops = 2 * T * params + attn
    assert bench.algorithmic_flops_per_step(CONFIGS["full_bf16_b64"]) == flops
    assert abs(flops / 1e12 - 1.919) < 0.001


def test_w2a8_step_bytes_count_two_bits_per_weight(bench):
    # 24 layers x (QKV 3072x2048 + O 2048x2048 + up 5632x2048 + down 2048x5632)
    # at 2 bits, W_in / W_out in bf16 (2048 x 7 each), K/V cache 24 x 2 x 4 x
    # 512 x 128 bf16 per observation
    ternary = 24 * (3072 * 2048 + 2048 * 2048 + 5632 * 2048 + 2048 * 5632) // 4
    dense = 2 * 2048 * 7 * 2
    cache = 2 * 24 * 4 * 512 * 128 * 2
    assert bench.algorithmic_bytes_per_step(CONFIGS["w2a8_b1"]) == ternary + dense + cache
    assert abs((ternary + dense) / 1e6 - 201.38) < 0.01
    assert abs(cache / 1e6 - 25.17) < 0.01
    # batch 16: every observation has its own cache, the weights are shared
    b16 = bench.algorithmic_bytes_per_step(CONFIGS["w2a8_b16"])
    assert b16 == ternary + dense + 16 * cache


def test_roofline_picks_the_longer_roof(bench):
    cfg = CONFIGS["full_bf16_b1"]
    roof = bench.roofline(cfg, 7.5)  # a 7.5 ms solve of 10 steps
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert abs(roof["achieved"] - 10 * bench.algorithmic_bytes_per_step(cfg) / 7.5e-3 / 1e9) < 1e-6
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-12
    roof64 = bench.roofline(CONFIGS["full_bf16_b64"], 26.0)
    assert roof64["bound"] == "tensor" and roof64["unit"] == "TFLOP/s"


def test_traffic_record_is_used_only_for_the_sources_it_was_taken_on(bench, tmp_path, monkeypatch):
    # A DRAM-traffic record names the hash of the library sources it was
    # captured on; the bench reports it only while the sources hash the same.
    csrc = tmp_path / "prefix_cached_flow_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("// a kernel\n__global__ void k() { int x = 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = tmp_path / "profiles" / "solver_w_traffic.txt"
    rec.write_text(f"dram_bytes_per_solver_launch: 123456\nlibrary_sources_sha256_16: {bench._lib_hash()}\n")
    assert bench._traffic_from_profile("w") == 123456.0
    # comments, blank lines and stray non-source files do not change the hash
    (csrc / "k.cu").write_text("// the same kernel, reworded comment\n\n__global__ void k() { int x = 1; }  // x\n")
    (csrc / "k.cu~").write_bytes(b"\xff\xfe binary backup")
    assert bench._traffic_from_profile("w") == 123456.0
    # a code change does
    (csrc / "k.cu").write_text("__global__ void k() { int x = 2; }\n")
    assert bench._traffic_from_profile("w") is None
    # no record: None
    assert bench._traffic_from_profile("other") is None


def test_cpu_model_reads_x86_and_arm_cpuinfo(bench):
    assert bench._cpu_model("processor\t: 0\nmodel name\t: Some Xeon @ 2.70GHz\n") == "Some Xeon @ 2.70GHz"
    arm = "processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU part\t: 0xd4f\n"
    assert bench._cpu_model(arm).endswith("implementer 0x41 part 0xd4f")
    assert bench._cpu_model("") == bench.platform.machine()
    assert bench._host_threads() >= 1
