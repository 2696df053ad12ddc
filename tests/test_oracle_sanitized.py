"""The oracle itself, run under AddressSanitizer and UndefinedBehaviorSanitizer:
the fast pins against a sanitized build of oracle/mix_oracle.c, in a child
process with the sanitizer runtimes preloaded.  Any out-of-bounds access or
undefined operation in the checker (a shift of a negative value, a signed
overflow) ends the child with a report."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import os, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, os.path.join({root!r}, "tests"))
import oracle
oracle._LIB = {lib!r}
oracle.lib()
import test_oracle_pins as T
for pin in T.FAST_PINS:
    pin(oracle)
print("pins ok")
"""


def _runtime(name):
    p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_pins_clean_under_asan_and_ubsan():
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not (asan and ubsan):
        pytest.skip("gcc sanitizer runtimes not installed")
    out = os.path.join(ROOT, "_build", "oracle_sanitized")
    os.makedirs(out, exist_ok=True)
    lib = os.path.join(out, f"liborcmix_san.{os.getpid()}.so")
    subprocess.run(["gcc", "-O1", "-g", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                    "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer",
                    "-o", lib, os.path.join(ROOT, "oracle", "mix_oracle.c"), "-lm"], check=True)
    try:
        env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0", LD_PRELOAD=f"{asan}:{ubsan}")
        r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT, lib=lib)], env=env, cwd=ROOT,
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0 and "pins ok" in r.stdout, (r.stdout + r.stderr)[-4000:]
        assert "runtime error" not in r.stderr, r.stderr[-4000:]
    finally:
        os.remove(lib)
