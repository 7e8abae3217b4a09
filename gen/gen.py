"""ctypes front-end of the counter-based generator (coli_gen.h).

Host fills come from libcoli_gen_host.so (gcc, -ffp-contract=off), device fills from
libcoli_gen_dev.so (nvcc, sm_103a).  Both produce the same bits for the same key and index.
"""
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SO = os.path.join(HERE, "libcoli_gen_host.so")
DEV_SO = os.path.join(HERE, "libcoli_gen_dev.so")

T_X, T_ROUTER, T_GATE, T_UP, T_DOWN, T_GAMMA, T_PERM, T_PICK = range(8)

_u64, _u32, _f32, _vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_float, ctypes.c_void_p


def build(cuda=True, arch="sm_103a"):
    """Compile the host generator, and the device one when `cuda` is set."""
    subprocess.check_call(
        ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11",
         os.path.join(HERE, "gen_host.c"), "-o", HOST_SO])
    if cuda:
        cc = arch.split("_")[1]
        subprocess.check_call(
            ["nvcc", "-O3", "-std=c++17", f"-gencode=arch=compute_{cc},code={arch}",
             "-Xcompiler", "-fPIC", "-shared", os.path.join(HERE, "gen_dev.cu"), "-o", DEV_SO])


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_SO):
            build(cuda=False)
        lib = ctypes.CDLL(HOST_SO)
        lib.cg_fill_normal_host.argtypes = [_vp, _u64, _u64, _u32, _u32, _u32, _u64, _f32]
        lib.cg_fill_uniform_affine_host.argtypes = [_vp, _u64, _u64, _u32, _u32, _u32, _u64, _f32, _f32]
        lib.cg_fill_draws_host.argtypes = [_vp, _u64, _u64, _u32, _u32, _u32, _u64]
        lib.cg_draw_raw_host.argtypes = [_u64, _u64]
        lib.cg_draw_raw_host.restype = _u64
        _host = lib
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_SO):
            raise RuntimeError("device generator not built: run __graft_entry__.build()")
        lib = ctypes.CDLL(DEV_SO)
        lib.cg_fill_normal_dev.argtypes = [_vp, _u64, _u64, _u32, _u32, _u32, _u64, _f32, _vp]
        lib.cg_fill_normal_dev.restype = ctypes.c_int
        lib.cg_fill_uniform_affine_dev.argtypes = [_vp, _u64, _u64, _u32, _u32, _u32, _u64, _f32, _f32, _vp]
        lib.cg_fill_uniform_affine_dev.restype = ctypes.c_int
        _dev = lib
    return _dev


def normal_host(shape, seed, layer, tensor, slot, idx0=0, sigma=1.0):
    out = np.empty(shape, dtype=np.float32)
    _host_lib().cg_fill_normal_host(out.ctypes.data, out.size, seed, layer, tensor, slot, idx0, sigma)
    return out


def uniform_affine_host(shape, seed, layer, tensor, slot, lo, span, idx0=0):
    out = np.empty(shape, dtype=np.float32)
    _host_lib().cg_fill_uniform_affine_host(out.ctypes.data, out.size, seed, layer, tensor, slot,
                                            idx0, lo, span)
    return out


def draws_host(n, seed, layer, tensor, slot, idx0=0):
    out = np.empty(n, dtype=np.uint64)
    _host_lib().cg_fill_draws_host(out.ctypes.data, n, seed, layer, tensor, slot, idx0)
    return out


def draw_raw_host(key, n):
    return int(_host_lib().cg_draw_raw_host(key, n))


def normal_dev(out, seed, layer, tensor, slot, idx0=0, sigma=1.0, stream=0):
    """Fill the contiguous float32 CUDA tensor `out` in place."""
    rc = _dev_lib().cg_fill_normal_dev(out.data_ptr(), out.numel(), seed, layer, tensor, slot, idx0,
                                       sigma, stream)
    if rc:
        raise RuntimeError("cg_fill_normal_dev failed")
    return out


def uniform_affine_dev(out, seed, layer, tensor, slot, lo, span, idx0=0, stream=0):
    rc = _dev_lib().cg_fill_uniform_affine_dev(out.data_ptr(), out.numel(), seed, layer, tensor, slot,
                                               idx0, lo, span, stream)
    if rc:
        raise RuntimeError("cg_fill_uniform_affine_dev failed")
    return out
