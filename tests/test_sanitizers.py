"""The oracle and the library's host code under AddressSanitizer and
UndefinedBehaviorSanitizer (no GPU).

Builds tests/sanitize_driver.cpp against the oracle's C source and against
every translation unit of the CUDA library, all host code compiled with
-fsanitize=address,undefined (device code is compiled as usual), and runs it.
The driver exercises the oracle's entry points on small problems with their
edge cases and the C ABI's argument checks and host-only planner; any
sanitizer report aborts it.
"""
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

from paged_gqa_decode_attention_gb300 import build as pda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SAN = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all",
       "-fno-omit-frame-pointer", "-g"]


def _run(cmd, cwd=None):
    res = subprocess.run(cmd, capture_output=True, text=True, cwd=cwd)
    if res.returncode != 0:
        raise AssertionError(f"{' '.join(cmd[:3])} ... failed:\n{res.stdout[-4000:]}\n"
                             f"{res.stderr[-4000:]}")
    return res


def test_oracle_and_host_library_under_asan_ubsan(tmp_path):
    if shutil.which("gcc") is None or shutil.which("g++") is None:
        pytest.skip("no gcc")
    try:
        nvcc = pda_build.nvcc_path()
    except RuntimeError:
        pytest.skip("no nvcc")
    cuda_home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    out = str(tmp_path)
    objs = []
    oracle_o = os.path.join(out, "oracle.o")
    _run(["gcc", "-std=c11", "-O1", "-ffp-contract=off", "-fno-fast-math", *SAN, "-c",
          os.path.join(ROOT, "oracle", "paged_attn_oracle.c"), "-o", oracle_o])
    objs.append(oracle_o)

    def compile_tu(src):
        obj = os.path.join(out, os.path.basename(src) + ".o")
        _run([nvcc, *pda_build.ARCH, "-O1", "-std=c++17", "-I", pda_build.INCLUDE, "-I",
              pda_build.CSRC, *[a for f in SAN for a in ("-Xcompiler", f)], "-c", src, "-o",
              obj])
        return obj

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        objs += list(ex.map(compile_tu, pda_build.sources()))
    driver = os.path.join(out, "sanitize_driver")
    _run(["g++", "-std=c++17", "-O1", *SAN, "-I", pda_build.INCLUDE,
          os.path.join(ROOT, "tests", "sanitize_driver.cpp"), *objs,
          "-L", os.path.join(cuda_home, "lib64"), "-lcudart_static", "-ldl", "-lpthread", "-lrt",
          "-lm", "-o", driver])
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0:protect_shadow_gap=0",
               UBSAN_OPTIONS="print_stacktrace=1")
    res = subprocess.run([driver], capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0, res.stdout[-4000:] + res.stderr[-4000:]
    assert "0 failure(s)" in res.stdout
