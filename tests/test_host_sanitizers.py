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


def test_planted_mistakes_stay_memory_safe(tmp_path):
    """every planted mistake of the C oracle only changes values: built with the sanitizers,
    its guard pins fail by assertion, never by an invalid access or undefined operation"""
    from concurrent.futures import ThreadPoolExecutor

    from . import test_oracle_mutants as M
    sos = {}

    def build(n):
        so = str(tmp_path / f"liboracle_m{n}_san.so")
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
                               "-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined",
                               "-fno-sanitize-recover=undefined", M.write_mutant(n, tmp_path),
                               "-o", so, "-lm"])
        sos[n] = so

    with ThreadPoolExecutor(max_workers=8) as ex:
        list(ex.map(build, sorted(M.MUTANTS)))
    plan = {n: (sos[n], M.MUTANTS[n][1]) for n in sorted(M.MUTANTS)}
    code = (f"import sys\nsys.path.insert(0, {ROOT!r})\n"
            "from oracle import oracle as O\n"
            "from tests import test_oracle_pins as P\n"
            f"for n, (so, guards) in {plan!r}.items():\n"
            "    O.SO, O._lib = so, None\n"
            "    for g in guards:\n"
            "        try:\n"
            "            getattr(P, g)()\n"
            "        except AssertionError:\n"
            "            pass\n"
            "print('all mutants ran')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_sanitizer_env(),
                       capture_output=True, text=True, timeout=600)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0 and "all mutants ran" in r.stdout, tail
    assert "ERROR: AddressSanitizer" not in tail and "runtime error:" not in tail, tail
