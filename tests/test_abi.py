"""The C ABI without a GPU: the library loads, exports every declared entry
point, agrees with a C compiler on struct layout, and rejects bad arguments on
the host before launching anything.  Also checks that the oracle and the CUDA
path share no code."""
import ctypes
import glob
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from smc_speculative_decoding_gb300 import build, binding
    build.build()
    return binding.lib()


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if not m.group(0).lstrip().startswith(("#", "typedef")):
                names.append(m.group(1))
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"smc_step", "smc_resample", "kv_blocktable_remap", "sps_verify"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_abi_version_and_strerror(lib):
    from smc_speculative_decoding_gb300 import binding
    assert binding.smc_abi_version() == 1
    for code in (0, -1, -2, -3, -4, -5, 1, 2, 4, 8, 16, 32, 64, 3):
        assert binding.smc_strerror(code)


def test_struct_layout_matches_c_compiler(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    from smc_speculative_decoding_gb300.binding import smc_params, smc_kv, smc_step_opts
    src = tmp_path / "layout.c"
    fields_p = [f[0] for f in smc_params._fields_]
    fields_k = [f[0] for f in smc_kv._fields_]
    fields_o = [f[0] for f in smc_step_opts._fields_]
    body = ['#include <stdio.h>', '#include <stddef.h>', '#include "smcsd.h"', 'int main(void){',
            'printf("%zu %zu %zu\\n", sizeof(smc_params), sizeof(smc_kv), sizeof(smc_step_opts));']
    body += [f'printf("p {f} %zu\\n", offsetof(smc_params, {f}));' for f in fields_p]
    body += [f'printf("k {f} %zu\\n", offsetof(smc_kv, {f}));' for f in fields_k]
    body += [f'printf("o {f} %zu\\n", offsetof(smc_step_opts, {f}));' for f in fields_o]
    body += ['return 0;}']
    src.write_text("\n".join(body))
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", f"-I{ROOT}/include", str(src), "-o",
                    str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    sp, sk, so = map(int, out[0].split())
    assert sp == ctypes.sizeof(smc_params) and sk == ctypes.sizeof(smc_kv)
    assert so == ctypes.sizeof(smc_step_opts)
    for line in out[1:]:
        if not line:
            continue
        kind, name, off = line.split()
        cls = {"p": smc_params, "k": smc_kv, "o": smc_step_opts}[kind]
        assert getattr(cls, name).offset == int(off), name


def test_header_compiles_as_c_and_cxx(tmp_path):
    for cc, ext in (("gcc", "c"), ("g++", "cpp")):
        exe = shutil.which(cc)
        if exe is None:
            continue
        src = tmp_path / f"h.{ext}"
        src.write_text('#include "smcsd.h"\nint main(void){ return smc_abi_version() < 0; }\n')
        subprocess.run([exe, "-Wall", "-Werror", f"-I{ROOT}/include", "-c", str(src), "-o",
                        str(tmp_path / f"h_{ext}.o")], check=True, capture_output=True)


def test_host_validation_without_gpu(lib):
    from smc_speculative_decoding_gb300 import binding as bd
    P = bd.smc_params
    fake = ctypes.c_void_p(0x1000)
    ws = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    bad_shapes = [P(1, 0, 3, 64, 0, 1.0, 0.5, 0, 0), P(1, 257, 3, 64, 0, 1.0, 0.5, 0, 0),
                  P(1, 4, 0, 64, 0, 1.0, 0.5, 0, 0), P(1, 4, 3, 0, 0, 1.0, 0.5, 0, 0),
                  P(1, 4, 3, 64, 0, -1.0, 0.5, 0, 0), P(1, 4, 3, 64, 0, float("nan"), 0.5, 0, 0)]
    for p in bad_shapes:
        assert lib.smc_workspace_bytes(ctypes.byref(p), None) == 0
        rc = lib.smc_step(ctypes.byref(p), *[fake] * 8, None, ws, 1 << 30, None)
        assert rc == -1
    good = P(2, 4, 3, 64, 0, 1.0, 0.5, 0, 0)
    need = lib.smc_workspace_bytes(ctypes.byref(good), None)
    assert need > 0 and need % 256 == 0
    assert lib.smc_step(None, *[fake] * 8, None, ws, need, None) == -1
    bad_dtype = P(2, 4, 3, 64, 7, 1.0, 0.5, 0, 0)
    assert lib.smc_step(ctypes.byref(bad_dtype), *[fake] * 8, None, ws, need, None) == -2
    assert lib.smc_step(ctypes.byref(good), *[fake] * 8, None, ws, need - 1, None) == -3
    assert lib.smc_step(ctypes.byref(good), *[fake] * 8, None, ctypes.c_void_p(0x10010), need,
                        None) == -3
    assert lib.smc_step(ctypes.byref(good), fake, None, *[fake] * 6, None, ws, need, None) == -1
    # sps_verify requires N == 1 and alpha == 1
    assert lib.sps_verify(ctypes.byref(good), *[fake] * 5, ws, need, None) == -1
    # kv_blocktable_remap needs a KV struct and n_append >= 0
    assert lib.kv_blocktable_remap(ctypes.byref(good), None, fake, fake, 1, ws, need, None) == -1
    kv = bd.smc_kv(*[0x2000] * 7, 8, 16, 64)
    assert lib.kv_blocktable_remap(ctypes.byref(good), ctypes.byref(kv), fake, fake, -1, ws,
                                   1 << 30, None) == -1
    assert lib.smc_device_status(None, 0, None, None) == -1
    # smc_step_ex: temperature must be positive and finite, reserved zero
    for t, tp, r in ((0.0, 1.0, 0), (-1.0, 1.0, 0), (float("inf"), 1.0, 0),
                     (float("nan"), 1.0, 0), (1e-45, 1.0, 0), (1.0, 1.0, 3), (1.0, 0.0, 0),
                     (1.0, 1.5, 0), (1.0, float("nan"), 0)):
        opts = bd.smc_step_opts(None, t, tp, (ctypes.c_int32 * 2)(r, 0))
        assert lib.smc_step_ex(ctypes.byref(good), ctypes.byref(opts), *[fake] * 8, None, ws,
                               need, None) == -1
    # top_p < 1 needs alpha == 1
    power = P(2, 4, 3, 64, 0, 4.0, 0.5, 0, 0)
    opts = bd.smc_step_opts(None, 1.0, 0.9, (ctypes.c_int32 * 2)(0, 0))
    assert lib.smc_step_ex(ctypes.byref(power), ctypes.byref(opts), *[fake] * 8, None, ws,
                           need, None) == -1
    # sps_verify_ex: no log-potential (one particle), the same temperature and
    # top_p rules
    sps_p = P(2, 1, 3, 64, 0, 1.0, 0.5, 0, 0)
    sps_need = lib.smc_workspace_bytes(ctypes.byref(sps_p), None)
    opts = bd.smc_step_opts(fake, 1.0, 1.0, (ctypes.c_int32 * 2)(0, 0))
    assert lib.sps_verify_ex(ctypes.byref(sps_p), *[fake] * 5, ctypes.byref(opts), ws, sps_need,
                             None) == -1
    for t, tp, r in ((0.0, 1.0, 0), (float("inf"), 1.0, 0), (1.0, 0.0, 0), (1.0, 1.5, 0),
                     (1.0, 1.0, 1)):
        opts = bd.smc_step_opts(None, t, tp, (ctypes.c_int32 * 2)(r, 0))
        assert lib.sps_verify_ex(ctypes.byref(sps_p), *[fake] * 5, ctypes.byref(opts), ws,
                                 sps_need, None) == -1
    assert lib.sps_verify_ex(ctypes.byref(good), *[fake] * 5, None, ws, need, None) == -1
    # smc_draft_sample: a position below 0 or a missing output
    assert lib.smc_draft_sample(ctypes.byref(good), fake, -1, fake, ws, need, None) == -1
    assert lib.smc_draft_sample(ctypes.byref(good), fake, 0, None, ws, need, None) == -1
    # smc_kv_usage needs the KV struct and both outputs
    assert lib.smc_kv_usage(ctypes.byref(good), None, fake, fake, None) == -1
    assert lib.smc_kv_usage(ctypes.byref(good), ctypes.byref(kv), None, fake, None) == -1
    # the row-timing hook takes both events or neither
    assert lib.smc_set_row_timing_events(fake, None) == -1
    assert lib.smc_set_row_timing_events(None, fake) == -1
    assert lib.smc_set_row_timing_events(None, None) == 0
    # the step clock needs a counter and a positive capacity with its stamps
    lib.smc_set_step_clock.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
    assert lib.smc_set_step_clock(fake, None, 4) == -1
    assert lib.smc_set_step_clock(fake, fake, 0) == -1
    assert lib.smc_set_step_clock(None, None, 0) == 0
    # the wait self-test: a buffer of two words, kind 0 or 1, a positive limit
    lib.smc_selftest_bounded_wait.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_void_p]
    assert lib.smc_selftest_bounded_wait(None, 64, 0, 10, None) == -1
    assert lib.smc_selftest_bounded_wait(fake, 4, 0, 10, None) == -1
    assert lib.smc_selftest_bounded_wait(fake, 64, 2, 10, None) == -1
    assert lib.smc_selftest_bounded_wait(fake, 64, 1, 0, None) == -1


def test_oracle_and_cuda_path_share_no_code():
    pkg = os.path.join(ROOT, "smc_speculative_decoding_gb300")
    for f in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True) + \
            glob.glob(os.path.join(pkg, "csrc", "*")):
        text = open(f, errors="ignore").read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), \
            f"{f} imports the oracle"
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        text = open(f).read()
        assert "smc_speculative_decoding_gb300" not in text, f"{f} imports the product"
