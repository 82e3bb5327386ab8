"""The oracle's C code under AddressSanitizer and UndefinedBehaviorSanitizer.

The pins of test_oracle.py (all but the planted mistakes, which build their own
copies of the oracle) run in a subprocess against a sanitized build of
w4a16_oracle.c: an out-of-bounds access, a use of freed memory, a signed overflow, a
bad shift or a misaligned load anywhere the pins reach ends that run with an error.
The sanitizer runtimes have to be loaded before the interpreter starts, hence the
subprocess and LD_PRELOAD; Python's own allocations are not leak-checked."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_SRC = os.path.join(ROOT, "oracle", "w4a16_oracle.c")


def _runtime(name):
    try:
        p = subprocess.run(["gcc", "-print-file-name=" + name], capture_output=True, text=True).stdout.strip()
    except OSError:
        return None
    return p if os.path.isabs(p) and os.path.exists(p) else None


def test_oracle_pins_run_clean_under_sanitizers():
    asan, ubsan = _runtime("libasan.so"), _runtime("libubsan.so")
    if not (asan and ubsan):
        pytest.skip("gcc's sanitizer runtimes are not installed")
    with tempfile.TemporaryDirectory() as d:
        lib = os.path.join(d, "liboracle_sanitized.so")
        subprocess.check_call(["gcc", "-O1", "-g", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fsanitize=address,undefined", "-fno-omit-frame-pointer",
                               "-fno-sanitize-recover=undefined", "-o", lib,
                               ORACLE_SRC, "-lm"])
        runner = ("import sys, pytest, oracle\n"
                  "oracle.build = lambda force=False: %r\n"
                  "sys.exit(pytest.main(['-q', '-x', '-s', '-p', 'no:cacheprovider', '-k', 'not planted_mistakes', %r]))\n"
                  % (lib, os.path.join(ROOT, "tests", "test_oracle.py")))
        # a sanitizer report ends the run with its own exit code (86: address, 87: undefined)
        env = dict(os.environ, LD_PRELOAD=asan + ":" + ubsan, ASAN_OPTIONS="detect_leaks=0:exitcode=86",
                   UBSAN_OPTIONS="halt_on_error=1:exitcode=87:print_stacktrace=1", PYTHONPATH=ROOT)
        r = subprocess.run([sys.executable, "-c", runner], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=900)
        assert r.returncode == 0, ("exit code %d" % r.returncode, r.stdout[-3000:], r.stderr[-3000:])
        assert " passed" in r.stdout
