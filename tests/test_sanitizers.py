"""AddressSanitizer + UndefinedBehaviorSanitizer builds of the host code, run on the CPU.

* The oracle (oracle/kv8_oracle.c) with a driver that calls every function on small inputs and edge
  cases (tests/sanitize/oracle_driver.c).
* The C ABI's host side: every library source compiled with the sanitizers (device code is unaffected)
  and a driver (tests/sanitize/abi_driver.cpp) run with all GPUs hidden, so no kernel can start.  It
  checks host validation (KV8_EINVAL / KV8_EWORKSPACE) and that a well-formed call whose launch the
  CUDA runtime refuses returns KV8_ECUDA -- a launch failure injected on the host, with no GPU fault.
Any sanitizer report makes the run exit non-zero.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SAN = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-g"]
ENV = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:protect_shadow_gap=0:abort_on_error=0",
           UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")


def _run(cmd, env=None, timeout=600):
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=timeout)
    assert r.returncode == 0, f"{' '.join(cmd)}\nstdout:\n{r.stdout[-4000:]}\nstderr:\n{r.stderr[-6000:]}"
    return r


def _gcc_has_sanitizers(tmp):
    src = os.path.join(tmp, "probe.c")
    open(src, "w").write("int main(void){return 0;}\n")
    r = subprocess.run(["gcc", *SAN, src, "-o", os.path.join(tmp, "probe")], capture_output=True)
    return r.returncode == 0


def test_oracle_under_asan_ubsan(tmp_path):
    if not shutil.which("gcc") or not _gcc_has_sanitizers(str(tmp_path)):
        pytest.skip("gcc with the address / undefined sanitizers is not available")
    exe = str(tmp_path / "oracle_asan")
    _run(["gcc", "-std=c11", "-O1", "-fopenmp", "-ffp-contract=off", *SAN,
          os.path.join(ROOT, "oracle", "kv8_oracle.c"), os.path.join(ROOT, "tests", "sanitize", "oracle_driver.c"),
          "-lm", "-o", exe])
    env = dict(ENV, OMP_NUM_THREADS="2",
               # the OpenMP runtime keeps thread pools alive at exit: leaks there are not the oracle's
               ASAN_OPTIONS="detect_leaks=0:abort_on_error=0")
    r = _run([exe], env=env)
    assert "oracle driver ok" in r.stdout


def test_c_abi_host_side_under_asan_ubsan(tmp_path):
    from fp8_latent_kv_gb300 import build as kvbuild
    try:
        nvcc = kvbuild._nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    if not _gcc_has_sanitizers(str(tmp_path)):
        pytest.skip("gcc with the address / undefined sanitizers is not available")
    flags = ["-gencode", "arch=compute_103a,code=sm_103a", "-O1", "-std=c++17", "--expt-relaxed-constexpr",
             "-I", os.path.join(ROOT, "include"), "-I", kvbuild.CSRC, "-Xcompiler", ",".join(SAN)]
    srcs = sorted(glob.glob(os.path.join(kvbuild.CSRC, "*.cu"))) + [
        os.path.join(ROOT, "tests", "sanitize", "abi_driver.cpp")]
    objs = []
    procs = []
    for s in srcs:
        o = str(tmp_path / (os.path.basename(s) + ".o"))
        objs.append(o)
        procs.append((s, subprocess.Popen([nvcc, *flags, "-c", s, "-o", o], stdout=subprocess.PIPE,
                                          stderr=subprocess.PIPE, text=True)))
    for s, p in procs:
        out, err = p.communicate(timeout=600)
        assert p.returncode == 0, f"nvcc failed on {s}:\n{err[-4000:]}"
    cudart = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
    exe = str(tmp_path / "abi_asan")
    _run(["g++", *SAN, *objs, "-L" + cudart, "-lcudart_static", "-ldl", "-lpthread", "-lrt", "-o", exe])
    env = dict(ENV, CUDA_VISIBLE_DEVICES="")  # no device can be seen: nothing can launch
    r = _run([exe], env=env)
    assert "abi driver ok" in r.stdout
