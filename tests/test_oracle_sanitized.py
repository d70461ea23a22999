"""The oracle's C under AddressSanitizer and UndefinedBehaviorSanitizer.

The pins of tests/test_oracle_pins.py run once more, in a child process, against a build of
nf4_oracle.c with -fsanitize=address,undefined and no recovery: an out-of-bounds or freed-memory
access, a signed overflow, an invalid shift or a misaligned load in the oracle aborts the run."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _runtime(name):
    p = subprocess.run(["gcc", f"-print-file-name={name}"], capture_output=True, text=True).stdout.strip()
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_pins_under_asan_and_ubsan(tmp_path):
    if os.environ.get("ORACLE_LIB"):
        pytest.skip("this process already runs another build of the oracle")
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not (asan and ubsan):
        pytest.skip("gcc has no sanitizer runtimes here")
    so = tmp_path / "liboracle_asan.so"
    subprocess.check_call(["gcc", "-O1", "-g", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer",
                           "-fPIC", "-shared", "-Wall", "-o", str(so), os.path.join(ROOT, "oracle", "nf4_oracle.c"),
                           "-lm"])
    env = dict(os.environ, ORACLE_LIB=str(so), LD_PRELOAD=f"{asan}:{ubsan}",
               ASAN_OPTIONS="detect_leaks=0", UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    # the sanitized oracle (and the sanitizer runtime) are the ones the child process loads
    probe = ("import oracle; oracle.lib(); m = open('/proc/self/maps').read(); "
             "assert 'liboracle_asan.so' in m and 'libasan' in m, 'sanitized oracle not loaded'")
    subprocess.run([sys.executable, "-c", probe], env=env, cwd=ROOT, check=True, timeout=300)
    # --capture=sys: a sanitizer report (written to file descriptor 2) reaches the output below
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider", "--capture=sys"], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert " passed" in r.stdout
