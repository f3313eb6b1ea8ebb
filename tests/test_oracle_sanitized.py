"""The oracle built with ASan and UBSan runs its pins without a report (CPU only).

The sanitized library is loaded in a child interpreter with the ASan runtime preloaded; any
out-of-bounds access, leak-free misuse or undefined behaviour in the oracle aborts the child."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r})
from oracle import build as obuild
from oracle.oracle import Oracle
from tests import oracle_pins as P
o = Oracle(path=obuild.build(sanitize=True, openmp=False, out_dir={out!r}))
for pin in P.ALL_PINS:
    pin(o)
print("sanitized pins ok", len(P.ALL_PINS))
"""


def test_oracle_pins_under_asan_ubsan(tmp_path):
    libasan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    if not libasan or not os.path.exists(libasan):
        pytest.skip("no ASan runtime for this compiler")
    env = dict(os.environ)
    env["LD_PRELOAD"] = libasan
    env["ASAN_OPTIONS"] = "detect_leaks=0:abort_on_error=1"
    env["UBSAN_OPTIONS"] = "halt_on_error=1:print_stacktrace=1"
    code = CHILD.format(root=ROOT, out=str(tmp_path))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-4000:]
    assert "sanitized pins ok" in r.stdout
