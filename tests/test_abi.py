"""The C-ABI library builds, loads and exports every function the headers under include/ declare;
argument validation that needs no GPU.  CPU only (no kernel is launched)."""
import ctypes
import shutil
import subprocess

import pytest

from int4_routed_expert_quantize_gb300 import _build, coli


@pytest.fixture(scope="module")
def built():
    if shutil.which("nvcc") is None:
        pytest.skip("nvcc not available")
    if _build.is_stale():  # a fresh build (e.g. by __graft_entry__.build()) is reused
        _build.build()
    coli._lib = None
    return coli.lib()


def test_exports_match_header(built):
    names = coli.header_functions()
    assert len(names) >= 13
    out = subprocess.run(["nm", "-D", "--defined-only", _build.SO], capture_output=True, text=True,
                         check=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines() if ln.strip()})
    assert exported == names  # every declared function, and nothing else
    for n in names:
        assert hasattr(built, n)


def test_strerror_and_record_bytes(built):
    for st in (0, -1, -2, -3, -4, -5, -6, -7):
        assert built.coli_moe_strerror(st)
    assert coli.expert_record_bytes(6144, 2048) == 18_915_328


def _create(**kw):
    base = dict(d=512, f=256, n_experts=32, top_k=4, n_shared=1, qblock=32, max_tokens=4,
                routed_scale=1.0, rms_eps=1e-6, has_norm=0)
    base.update(kw)
    cfg = coli.Config(**base)
    h = ctypes.c_void_p()
    rc = coli.lib().coli_moe_create(ctypes.byref(cfg), ctypes.byref(h))
    if rc == 0:
        coli.lib().coli_moe_destroy(h)
    return rc, h.value


@pytest.mark.parametrize("kw,expect", [
    (dict(qblock=16), -1), (dict(n_experts=0), -1), (dict(top_k=0), -1), (dict(top_k=33, n_experts=64), -1),
    (dict(top_k=40, n_experts=32), -1), (dict(n_shared=2), -1), (dict(max_tokens=0), -1),
    (dict(max_tokens=5000), -1), (dict(rms_eps=-1.0), -1), (dict(routed_scale=float("inf")), -1),
    (dict(d=500), -6), (dict(d=192), -6), (dict(f=2560), -6), (dict(d=16384), -6),
])
def test_create_rejects_bad_config(built, kw, expect):
    rc, h = _create(**kw)
    assert rc == expect and h is None


def test_null_arguments(built):
    L = coli.lib()
    assert L.coli_moe_create(None, None) == -1
    h = ctypes.c_void_p()
    assert L.coli_moe_create(None, ctypes.byref(h)) == -1 and h.value is None
    assert L.coli_moe_forward(None, None, 1, None, None) == -1
    assert L.coli_moe_load_router(None, None, None, None, None) == -1
    assert L.coli_moe_load_experts(None, 0, 1, None, None, None) == -1
    assert L.coli_quantize_act_q8(None, 33, None, None, None) == -1
    assert L.coli_quantize_act_q8(None, 0, None, None, None) == 0
    assert L.coli_quantize_i4_rows(None, 4, 7, None, None, None) == -1
    assert L.coli_moe_status(None, None) == -1
    assert L.coli_moe_inject_fault(None, 1) == -1
    assert L.coli_moe_set_prefill_min(None, 64) == -1
    assert L.coli_moe_launches(None, 1) == -1
    L.coli_moe_destroy(None)


def test_create_without_gpu_reports_cuda_error(built):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = _create()
    assert rc == -4 and h is None


def test_binding_constants_match_the_headers():
    """status codes, tier classes and counters in the binding are the headers' #defines"""
    import glob
    import os
    import re
    text = "".join(open(h).read() for h in glob.glob(os.path.join(_build.INCLUDE, "*.h")))
    defs = {m.group(1): int(m.group(2)) for m in
            re.finditer(r"^#define\s+(COLI_\w+)\s+\(?(-?\d+)\)?", text, re.M)}
    for code, name in coli.STATUS.items():
        assert defs[name] == code, name
    assert {v for k, v in defs.items() if re.fullmatch(r"COLI_E[A-Z]+|COLI_OK", k)} == set(coli.STATUS)
    assert coli.ETIMEOUT == defs["COLI_ETIMEOUT"]
    assert coli.FAULT_SKIP_ARRIVAL == defs["COLI_FAULT_SKIP_ARRIVAL"]
    assert defs["COLI_TIER_N_STATS"] == len(coli.TIER_STATS)
    from oracle.tier import LRU_HIT, MISS, PIN_HIT
    assert (defs["COLI_TIER_PIN_HIT"], defs["COLI_TIER_LRU_HIT"], defs["COLI_TIER_MISS"]) == (PIN_HIT, LRU_HIT, MISS)
