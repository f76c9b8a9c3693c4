"""The fp64 oracle compiled with AddressSanitizer and UndefinedBehaviorSanitizer
(gcc) and run over every entry point, weight format and router mode on small
layers: no out-of-bounds access, use after free or undefined arithmetic."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
DRIVER = os.path.join(HERE, "oracle_sanitize_driver.c")


def test_oracle_under_address_and_undefined_behaviour_sanitizers(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    exe = str(tmp_path / "oracle_sanitized")
    r = subprocess.run([gcc, "-std=c11", "-O1", "-g", "-fno-omit-frame-pointer", "-fopenmp",
                        "-fsanitize=address,undefined", "-fno-sanitize-recover=all", DRIVER, "-o", exe, "-lm"],
                       capture_output=True, text=True)
    if r.returncode != 0 and "asan" in r.stderr.lower():
        pytest.skip("sanitizer runtimes not installed: " + r.stderr.splitlines()[-1])
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=0:abort_on_error=0", UBSAN_OPTIONS="print_stacktrace=1",
               OMP_NUM_THREADS="2")
    run = subprocess.run([exe], env=env, capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "runtime error" not in run.stderr and "AddressSanitizer" not in run.stderr, run.stderr
    assert run.stdout.strip().endswith("ok")
