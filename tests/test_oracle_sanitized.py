"""The CPU oracle (and the seeded generator that feeds it) under
AddressSanitizer and UndefinedBehaviorSanitizer: `sanitize_driver.c` calls
every oracle entry point on small inputs; any out-of-bounds access, leak,
signed overflow or other undefined behaviour aborts the run.  The binary is
built in tests/_build (git-ignored)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_oracle_under_asan_and_ubsan():
    cc = shutil.which("gcc")
    if cc is None:
        pytest.skip("gcc not found")
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, f"sanitize_driver_{os.getpid()}")
    cmd = [cc, "-std=c11", "-O1", "-g", "-fsanitize=address,undefined",
           "-fno-sanitize-recover=all", "-fno-omit-frame-pointer", "-fopenmp", "-Wall", "-Wextra",
           "-Werror", "-o", exe, os.path.join(HERE, "sanitize_driver.c"),
           os.path.join(ROOT, "oracle", "ptq_oracle.c"), os.path.join(ROOT, "synth", "gen.c"),
           "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and "sanitize" in (r.stderr or "") and "cannot find" in r.stderr:
        pytest.skip("no sanitizer runtime: " + r.stderr.strip().splitlines()[-1])
    assert r.returncode == 0, r.stderr
    try:
        env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=1",
                   UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
        run = subprocess.run([exe], capture_output=True, text=True, timeout=600, env=env)
        assert run.returncode == 0, run.stdout + run.stderr
        assert "sanitized oracle run: ok" in run.stdout
    finally:
        os.remove(exe)
