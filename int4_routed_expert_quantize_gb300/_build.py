"""Build of libcoli_moe.so: nvcc for sm_103a (the host-only tier manager through nvcc's host
compiler), one object per source compiled in parallel."""
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
SO = os.path.join(PKG, "libcoli_moe.so")
SOURCES = ["pack.cu", "route.cu", "expert_decode.cu", "gateup_w4.cu", "down_w4.cu", "gateup_w8.cu",
           "down_w8.cu", "gateup_w2.cu", "down_w2.cu", "expert_fused.cu", "expert_prefill.cu",
           "runtime.cu", "noalloc.cu", "tier.cpp", "status.cpp"]
HOST_SOURCES = ["tier.cpp", "status.cpp"]  # the parts that need no CUDA


def nvcc_flags(arch="sm_103a"):
    cc = arch.split("_")[1]
    return ["-O3", "-std=c++17", f"-gencode=arch=compute_{cc},code={arch}", "-lineinfo",
            "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def is_stale():
    """True when the library is missing or older than a source or header it is built from"""
    if not os.path.exists(SO):
        return True
    built = os.path.getmtime(SO)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)] + [os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > built for p in deps if os.path.isfile(p))


def build(arch="sm_103a", verbose=False, extra=()):
    os.makedirs(BUILD, exist_ok=True)
    flags = nvcc_flags(arch) + list(extra)

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = ["nvcc"] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        subprocess.check_call(cmd)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    subprocess.check_call(["nvcc", "-shared", "-cudart", "static", "-Xlinker",
                           "--version-script=" + os.path.join(CSRC, "exports.map"), "-o", SO] + objs)
    return SO


def build_host(out, sanitize=False):
    """Build the host-only parts (tier manager, status strings) with g++ into `out`; with
    `sanitize`, under AddressSanitizer and UndefinedBehaviorSanitizer (for tests)."""
    flags = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-I", INCLUDE, "-I", CSRC]
    if sanitize:
        flags += ["-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined",
                  "-fno-sanitize-recover=undefined"]
    subprocess.check_call(flags + [os.path.join(CSRC, f) for f in HOST_SOURCES] + ["-o", out])
    return out
