"""The host code under AddressSanitizer and UndefinedBehaviorSanitizer (CPU
only; the WARP page's rule of sanitizing host-side parsers and validation):

  * libgdn.so rebuilt with -fsanitize=address,undefined on its host code, and a
    C driver (tests/sanitize/abi_driver.c) that sends every entry point bad
    arguments -- every call must return the documented status before touching a
    device, with no sanitizer report;
  * the C oracle (oracle/gdn_oracle.c) built the same way and run by
    tests/sanitize/oracle_driver.c on cases that walk its edge paths (empty and
    one-token sequences, beta at 0 and 1, strong decay, a zero q head).

Both builds go to tests/sanitize/_build (not tracked)."""
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.join(ROOT, "tests", "sanitize")
BUILD = os.path.join(HERE, "_build")
CSRC = os.path.join(ROOT, "gated_deltanet_linear_decode_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
SAN = "-fsanitize=address,undefined"
ENV = {**os.environ, "ASAN_OPTIONS": "detect_leaks=0:halt_on_error=1:abort_on_error=0",
       "UBSAN_OPTIONS": "halt_on_error=1:print_stacktrace=1"}


def _have(tool):
    return shutil.which(tool) is not None


def _gcc_has_sanitizers():
    if not _have("gcc"):
        return False
    lib = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    return os.path.isabs(lib) and os.path.exists(lib)


def _run(cmd, **kw):
    r = subprocess.run(cmd, capture_output=True, text=True, **kw)
    assert r.returncode == 0, f"{' '.join(cmd)}\n{r.stdout[-4000:]}\n{r.stderr[-4000:]}"
    return r


@pytest.mark.skipif(not _gcc_has_sanitizers(), reason="gcc with AddressSanitizer runtime not available")
def test_oracle_under_sanitizers():
    os.makedirs(BUILD, exist_ok=True)
    exe = os.path.join(BUILD, "oracle_driver")
    _run(["gcc", "-O1", "-g", "-std=c11", SAN, "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-fopenmp",
          "-ffp-contract=off", os.path.join(ROOT, "oracle", "gdn_oracle.c"), os.path.join(HERE, "oracle_driver.c"),
          "-lm", "-o", exe])
    r = _run([exe], env=ENV, timeout=300)
    assert r.stdout.strip().endswith("ok"), r.stdout


@pytest.mark.skipif(not (_gcc_has_sanitizers() and _have("nvcc")), reason="needs nvcc and gcc sanitizer runtimes")
def test_abi_validation_under_sanitizers():
    os.makedirs(BUILD, exist_ok=True)
    host = f"-fPIC,-g,-fno-omit-frame-pointer,{SAN.replace(',', ',-fsanitize=')}"
    srcs = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".san.o")
        _run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O1", "-std=c++17", "--expt-relaxed-constexpr",
              "-Xcompiler", host, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj])
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    lib = os.path.join(BUILD, "libgdn_san.so")
    cudalib = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(shutil.which("nvcc")))), "lib64")
    _run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-Xcompiler", host, *objs, "-o", lib,
          "-L", cudalib, "-lcublasLt", "-Xlinker", "-rpath", "-Xlinker", cudalib])
    exe = os.path.join(BUILD, "abi_driver")
    _run(["gcc", "-O1", "-g", "-std=c11", SAN, "-fno-sanitize-recover=all", "-I", INCLUDE,
          os.path.join(HERE, "abi_driver.c"), "-L", BUILD, "-lgdn_san", "-Wl,-rpath," + BUILD, "-o", exe])
    r = _run([exe], env=ENV, timeout=300)
    assert r.stdout.strip().endswith("ok"), r.stdout
