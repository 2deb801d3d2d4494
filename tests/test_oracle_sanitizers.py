"""The oracle under AddressSanitizer and UBSan (host only).

mita_oracle.cpp is compiled with -fsanitize=address,undefined into a
temporary library, and every pin of tests/oracle_pins.py runs against it in
a child process with the sanitizer runtime preloaded (a Python process has
to load it first). Any out-of-bounds access, use after free or undefined
behaviour (overflow, bad shift, misaligned load) aborts the child with a
report, which fails the test.
"""
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r"""
import sys
sys.path.insert(0, {tests!r})
sys.path.insert(0, {root!r})
import oracle, oracle_pins
orc = oracle.Oracle({lib!r})
names = [n for n in dir(oracle_pins) if n.startswith("pin_")]
for n in names:
    getattr(oracle_pins, n)(orc)
print("pins:", len(names))
"""


def _asan_runtime():
    gxx = shutil.which("g++")
    if not gxx:
        return None
    path = subprocess.run([gxx, "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    return path if os.path.isabs(path) and os.path.exists(path) else None


def test_oracle_pins_under_asan_and_ubsan(tmp_path):
    runtime = _asan_runtime()
    if runtime is None:
        pytest.skip("no g++ with AddressSanitizer here")
    lib = str(tmp_path / "liboracle_san.so")
    subprocess.check_call(["g++", "-O1", "-g", "-std=c++17", "-fopenmp", "-shared", "-fPIC",
                           "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined",
                           "-fno-omit-frame-pointer", os.path.join(ROOT, "oracle", "mita_oracle.cpp"), "-o", lib])
    env = dict(os.environ, LD_PRELOAD=runtime, ASAN_OPTIONS="detect_leaks=0",
               UBSAN_OPTIONS="halt_on_error=1:print_stacktrace=1", OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-c", CHILD.format(tests=HERE, root=ROOT, lib=lib)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-4000:])
    assert "pins: 17" in r.stdout, r.stdout
