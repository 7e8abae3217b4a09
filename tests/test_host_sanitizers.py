"""The C oracle and the library's host-only parts under AddressSanitizer and
UndefinedBehaviorSanitizer.  CPU only.

Each side is rebuilt with -fsanitize=address,undefined into a scratch directory. A child
pytest run, with the sanitizer runtime preloaded, then repeats the checks against it:
- every oracle pin, against the sanitized oracle;
- the tier manager's parity and usage-file checks, against the sanitized host library
  (tier manager and status strings).

An invalid access, an overflow or an undefined operation ends the child with an error. Leak
detection is off, because the Python interpreter itself does not free everything at exit.
"""
import os
import subprocess
import sys

import pytest

from int4_routed_expert_quantize_gb300 import _build
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _sanitizer_env(**extra):
    libasan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True,
                             text=True).stdout.strip()
    if not os.path.isabs(libasan) or not os.path.exists(libasan):
        pytest.skip("gcc has no AddressSanitizer runtime here")
    env = dict(os.environ)
    env.update(LD_PRELOAD=libasan, ASAN_OPTIONS="detect_leaks=0:exitcode=97",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1:exitcode=98", **extra)
    return env


def _child_pytest(env, *targets):
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        *targets], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    assert "passed" in r.stdout and "ERROR: AddressSanitizer" not in tail, tail
    assert "runtime error:" not in tail, tail


def test_oracle_pins_under_sanitizers(tmp_path):
    so = str(tmp_path / "liboracle_san.so")
    O.build(out=so, sanitize=True)
    _child_pytest(_sanitizer_env(COLI_ORACLE_SO=so), "tests/test_oracle_pins.py")


def test_tier_manager_under_sanitizers(tmp_path):
    so = str(tmp_path / "libcoli_tier_san.so")
    _build.build_host(so, sanitize=True)
    _child_pytest(_sanitizer_env(COLI_TIER_HOST_SO=so), "tests/test_tier_parity.py")
