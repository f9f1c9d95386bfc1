"""AddressSanitizer + UndefinedBehaviorSanitizer runs on the CPU (no GPU):
the oracle's C code on small seeded inputs, and the library's host-side
argument checks (the CUDA sources' host code built with the sanitizers; the
device code is built as PTX only, which the checks never reach)."""
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SAN = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all",
       "-fno-omit-frame-pointer"]
NVCC_SAN = [f for flag in SAN for f in ("-Xcompiler", flag)]
ENV = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:protect_shadow_gap=0:abort_on_error=0",
           UBSAN_OPTIONS="print_stacktrace=1")


def _run(cmd, env=None):
    r = subprocess.run(cmd, capture_output=True, text=True, env=env)
    assert r.returncode == 0, f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
    return r


def test_oracle_under_asan_ubsan(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    exe = str(tmp_path / "oracle_driver")
    _run(["gcc", "-std=c11", "-O1", "-g", *SAN, "-ffp-contract=off",
          "-I", os.path.join(ROOT, "oracle"), "-o", exe,
          os.path.join(ROOT, "tests", "sanitize", "oracle_driver.c"),
          os.path.join(ROOT, "oracle", "rvq_oracle.c"), "-lm"])
    r = _run([exe], env=ENV)
    assert "oracle driver done" in r.stdout


def test_library_host_checks_under_asan_ubsan(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    csrc = os.path.join(ROOT, "moe_expert_ffn_router_gb300", "csrc")
    srcs = sorted(os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith(".cu"))
    flags = ["-gencode", "arch=compute_103a,code=compute_103a", "-O1", "-std=c++17",
             "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
             *NVCC_SAN]

    def compile_one(src):
        obj = str(tmp_path / (os.path.basename(src)[:-3] + ".o"))
        _run([nvcc, *flags, "-c", src, "-o", obj])
        return obj

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    exe = str(tmp_path / "host_checks")
    _run([nvcc, "-gencode", "arch=compute_103a,code=compute_103a", "-I",
          os.path.join(ROOT, "include"), *NVCC_SAN, "-o", exe,
          os.path.join(ROOT, "tests", "sanitize", "host_checks.c"), *objs])
    r = _run([exe], env=ENV)
    assert "host checks done" in r.stdout
