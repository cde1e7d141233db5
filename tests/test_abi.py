"""Host-side checks of the C ABI: the library loads, exports every entry
point that include/vla.h declares, and rejects bad arguments synchronously
(before touching a device)."""

import ctypes
import os
import re

import pytest

import prefix_cached_flow_gb300 as V

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "vla.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(vla_[a-z0-9_]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(V.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return V.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "vla_prefix_kv_build" in names and "vla_action_denoise_w2a8" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(V.EXPORTED) <= set(names)


def test_status_strings(lib):
    for s in range(9):
        assert lib.vla_status_string(s)
    assert lib.vla_version() == b"0.1.0"


def test_null_arguments_rejected_without_device(lib):
    out = ctypes.c_void_p()
    assert lib.vla_expert_create(None, None, 4, None, ctypes.byref(out)) == 1
    assert lib.vla_expert_create_w2a8(None, None, 4, None, ctypes.byref(out)) == 1
    assert lib.vla_prefix_kv_build(None, None, 1, 1, None, None, None) == 1
    assert lib.vla_action_denoise(None, None, None, 1, 1, None, None, None, None) == 1
    assert lib.vla_action_denoise_w2a8(None, None, None, 1, 1, None, None, None, None) == 1
    assert lib.vla_policy_step_host(None, None, 1, 1, None, None, None) == 1
    assert lib.vla_expert_poll_status(None, None) == 1
    assert lib.vla_expert_set_abort(None, 1) == 1
    assert lib.vla_w2a8_quantize_rows(None, 1, 1, None, None, None) == 1
    assert lib.vla_w2a8_ternary_gemm(None, None, None, 1.0, 1, 1, 64, None, None, None) == 1
    n = ctypes.c_size_t()
    assert lib.vla_prefix_cache_bytes(None, 1, 1, ctypes.byref(n)) == 1
    lib.vla_expert_destroy(None)


def _cfg(**kw):
    base = dict(n_layers=2, width=128, mlp_width=512, n_q_heads=4, n_kv_heads=1, head_dim=32, vlm_hidden=128,
                action_dim=7, horizon=8, time_dim=256, max_batch=1, max_prefix=64, dtype=V.DTYPE_BF16,
                rms_eps=1e-6, flags=0)
    base.update(kw)
    return V.binding.VlaConfig(**base)


def _dummy_weights():
    # 16-byte aligned non-null host addresses: validation order rejects the
    # config before any pointer is dereferenced.
    buf = (ctypes.c_uint8 * 64)()
    addr = (ctypes.addressof(buf) + 15) & ~15
    return buf, V.binding.VlaWeights(**{n: addr for n in V.binding.DENSE_FIELDS})


@pytest.mark.parametrize("kw,code", [
    (dict(n_layers=0), 1), (dict(n_q_heads=4, n_kv_heads=3), 2), (dict(time_dim=255), 2),
    (dict(dtype=7), 1), (dict(width=100), 3), (dict(rms_eps=0.0), 1), (dict(max_batch=0), 1)])
def test_config_validation(lib, kw, code):
    keep, w = _dummy_weights()
    out = ctypes.c_void_p()
    c = _cfg(**kw)
    assert lib.vla_expert_create(ctypes.byref(c), ctypes.byref(w), 4, None, ctypes.byref(out)) == code
    assert not out.value


def test_bad_solver_length_and_misaligned_pointer(lib):
    keep, w = _dummy_weights()
    out = ctypes.c_void_p()
    c = _cfg()
    assert lib.vla_expert_create(ctypes.byref(c), ctypes.byref(w), 0, None, ctypes.byref(out)) == 1
    w.wq = w.wq + 1
    assert lib.vla_expert_create(ctypes.byref(c), ctypes.byref(w), 4, None, ctypes.byref(out)) == 1


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/vla.h is a C header (no C++ or torch types): a C99 program that
    includes it and takes the address of every declared entry point compiles
    with -Wall -Werror and links against the built library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = _declared()
    src = tmp_path / "abi_check.c"
    body = "\n".join(f"  p[{i}] = (fn){n};" for i, n in enumerate(names))
    src.write_text('#include "vla.h"\n#include <stdio.h>\n'
                   f"typedef void (*fn)(void);\nint main(void) {{\n  fn p[{len(names)}];\n{body}\n"
                   f"  for (int i = 0; i < {len(names)}; ++i) if (!p[i]) return 1;\n"
                   '  printf("%s\\n", vla_status_string(VLA_OK));\n  return 0;\n}\n')
    libdir = os.path.dirname(V.LIB_PATH)
    exe = tmp_path / "abi_check"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-lvla", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    # the program runs without a GPU: it only resolves symbols and reads a string
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip(), r.stderr
