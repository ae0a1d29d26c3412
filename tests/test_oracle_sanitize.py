"""The oracle under AddressSanitizer and UndefinedBehaviorSanitizer (CPU only).

oracle/dflash2_oracle.c is compiled single-threaded (its OpenMP pragmas
ignored) with -fsanitize=address,undefined (no
recovery: the first finding aborts) together with tests/oracle_sanitize.c, a
driver that calls every oracle function on small seeded inputs and on the
degenerate and rejected cases; the run must exit 0 with no sanitizer report.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _sanitizers_available(tmp):
    src = os.path.join(tmp, "probe.c")
    with open(src, "w") as f:
        f.write("int main(void){return 0;}\n")
    r = subprocess.run(["gcc", "-fsanitize=address,undefined", src, "-o",
                        os.path.join(tmp, "probe")], capture_output=True)
    return r.returncode == 0


def test_oracle_clean_under_asan_ubsan(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    tmp = str(tmp_path)
    if not _sanitizers_available(tmp):
        pytest.skip("gcc without the address/undefined sanitizer runtimes")
    exe = os.path.join(tmp, "oracle_sanitize")
    cmd = ["gcc", "-std=c11", "-O1", "-g", "-fno-omit-frame-pointer", "-fno-fast-math",
           "-ffp-contract=off", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
           "-Wall", "-Wextra", "-Werror", "-Wno-unknown-pragmas",
           os.path.join(ROOT, "oracle", "dflash2_oracle.c"),
           os.path.join(HERE, "oracle_sanitize.c"), "-lm", "-o", exe]
    subprocess.run(cmd, check=True)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=1",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    r = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "oracle sanitize ok" in r.stdout
    assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr
