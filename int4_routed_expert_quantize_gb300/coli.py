"""Thin ctypes binding of libcoli_moe.so (include/coli_moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.  If the shared library is missing the import of
`lib()` raises: there is no CPU fallback.
"""
import ctypes
import glob
import os
import re
import sys

import numpy as np

import torch

from . import _build

_i, _f, _vp, _i64 = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int64

STATUS = {0: "COLI_OK", -1: "COLI_EINVAL", -2: "COLI_ENOMEM", -3: "COLI_ESTATE", -4: "COLI_ECUDA",
          -5: "COLI_ETIMEOUT", -6: "COLI_EUNSUPPORTED", -7: "COLI_EIO"}
HEADER = os.path.join(_build.INCLUDE, "coli_moe.h")
ETIMEOUT = -5
FAULT_SKIP_ARRIVAL = 1  # coli_moe_inject_fault: the next fused forward leaves CTA 0 out of its barrier


class ColiError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({lib().coli_moe_strerror(status).decode()})")


class Config(ctypes.Structure):
    _fields_ = [("d", _i), ("f", _i), ("n_experts", _i), ("top_k", _i), ("n_shared", _i),
                ("qblock", _i), ("max_tokens", _i), ("routed_scale", _f), ("rms_eps", _f),
                ("has_norm", _i), ("wbits", _i), ("hbm_slots", _i)]


class TierConfig(ctypes.Structure):
    _fields_ = [("n_layers", _i), ("n_experts", _i), ("n_pin", _i), ("n_lru", _i)]


DUMP_FIELDS = ["xn", "qx", "dx", "logits", "scores", "ids", "w", "n_union", "union_ids", "offsets",
               "pair_token", "pair_rank", "inv", "g", "u", "h", "qh", "dh", "e", "Ag", "Au", "Ad"]


class Dump(ctypes.Structure):
    _fields_ = [(n, _vp) for n in DUMP_FIELDS]


_lib = None


def header_functions():
    """names of the functions the headers under include/ declare"""
    text = "".join(open(h).read() for h in sorted(glob.glob(os.path.join(_build.INCLUDE, "*.h"))))
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(coli_\w+)\s*\(", text, re.M)))


def _bind_host(L):
    """argument types of the host-only entry points (tier manager, status strings)"""
    _ip = ctypes.POINTER(_i)
    L.coli_tier_create.argtypes = [ctypes.POINTER(TierConfig), ctypes.POINTER(_vp)]
    L.coli_tier_destroy.argtypes = [_vp]
    L.coli_tier_destroy.restype = None
    L.coli_tier_lookup.argtypes = [_vp, _i, _vp, _i, _vp, _vp, _vp, _vp, _ip, _vp, _vp, _ip]
    L.coli_tier_prefetch.argtypes = [_vp, _i, _vp, _i, _vp, _vp, _ip, _vp, _vp, _ip]
    L.coli_tier_repin.argtypes = [_vp, _i, _vp, _vp, _ip, _vp, _vp, _ip]
    L.coli_tier_autopin.argtypes = [_vp, _i, _vp, _vp, _ip, _vp, _vp, _ip]
    L.coli_tier_decay.argtypes = [_vp]
    L.coli_tier_session_heat.argtypes = [_vp, _i, _vp]
    L.coli_tier_state.argtypes = [_vp, _i, _vp, _ip, _vp, _ip, _vp]
    L.coli_tier_heat.argtypes = [_vp, _i, _vp]
    L.coli_tier_set_heat.argtypes = [_vp, _i, _vp]
    L.coli_tier_stats.argtypes = [_vp, _vp]
    L.coli_tier_config_of.argtypes = [_vp, ctypes.POINTER(TierConfig)]
    L.coli_tier_save_usage.argtypes = [_vp, ctypes.c_char_p]
    L.coli_tier_load_usage.argtypes = [_vp, ctypes.c_char_p]
    L.coli_moe_strerror.argtypes = [_i]
    L.coli_moe_strerror.restype = ctypes.c_char_p


def _bind_layer(L):
    """argument types of the layer's entry points"""
    L.coli_moe_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(_vp)]
    L.coli_moe_destroy.argtypes = [_vp]
    L.coli_moe_destroy.restype = None
    L.coli_moe_load_router.argtypes = [_vp, _vp, _vp, _vp, _vp]
    L.coli_moe_load_experts.argtypes = [_vp, _i, _i, _vp, _vp, _vp]
    L.coli_moe_forward.argtypes = [_vp, _vp, _i, _vp, _vp]
    L.coli_moe_forward_debug.argtypes = [_vp, _vp, _i, _vp, ctypes.POINTER(Dump), _vp]
    L.coli_moe_forward_host.argtypes = [_vp, _vp, _i, _vp, _vp]
    L.coli_moe_forward_profiled.argtypes = [_vp, _vp, _i, _vp, ctypes.POINTER(_vp), _i, _vp]
    L.coli_moe_stack_forward.argtypes = [ctypes.POINTER(_vp), _i, _vp, _i, _vp]
    L.coli_moe_status.argtypes = [_vp, _vp]
    L.coli_moe_expert_record_bytes.argtypes = [_i, _i]
    L.coli_moe_expert_record_bytes.restype = _i64
    L.coli_moe_expert_record_bytes_w.argtypes = [_i, _i, _i]
    L.coli_moe_expert_record_bytes_w.restype = _i64
    L.coli_quantize_i8_rows.argtypes = [_vp, _i64, _i, _vp, _vp, _vp]
    L.coli_quantize_i2_rows.argtypes = [_vp, _i64, _i, _vp, _vp, _vp]
    L.coli_moe_launches.argtypes = [_vp, _i]
    L.coli_moe_inject_fault.argtypes = [_vp, _i]
    L.coli_moe_set_prefill_min.argtypes = [_vp, _i]
    L.coli_quantize_i4_rows.argtypes = [_vp, _i64, _i, _vp, _vp, _vp]
    L.coli_quantize_act_q8.argtypes = [_vp, _i64, _vp, _vp, _vp]
    L.coli_route_noalloc.argtypes = [_vp, _i, _vp, _vp, _i, _i, _i, _f, _vp, _vp, _vp]
    L.coli_moe_forward_tiered.argtypes = [_vp, _vp, _i, _vp, _i, _vp, _vp]
    L.coli_moe_prefetch_tiered.argtypes = [_vp, _vp, _i, _vp, _i, _vp]
    L.coli_moe_repin_tiered.argtypes = [_vp, _vp, _i, _i, _vp]
    L.coli_moe_tier_copies.argtypes = [_vp, ctypes.POINTER(_i64), ctypes.POINTER(_i64)]


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_build.SO):
            raise RuntimeError(f"{_build.SO} is missing: build the CUDA extension first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(_build.SO)
        _bind_host(L)
        _bind_layer(L)
        _lib = L
    return _lib


def use_host_library(path):
    """Bind a host-only build of the tier manager (_build.build_host) in place of the full
    library: for the tier calls alone, e.g. a sanitizer run.  The layer calls are absent."""
    global _lib
    L = ctypes.CDLL(path)
    _bind_host(L)
    _lib = L
    return L


def _check(rc, where):
    if rc != 0:
        raise ColiError(rc, where)


def _ptr(a):
    """device or host address of a torch tensor / numpy array (None -> NULL)"""
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        if not a.is_contiguous():
            raise ValueError("the library takes contiguous tensors")
        return a.data_ptr()
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("the library takes C-contiguous arrays")
    return a.ctypes.data


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else stream


def expert_record_bytes(d, f, wbits=4):
    return int(lib().coli_moe_expert_record_bytes_w(d, f, wbits))


class MoeLayer:
    """One routed-expert MoE layer (int4 experts, or int8 / int2 with wbits) resident on the
    current CUDA device."""

    def __init__(self, d, f, n_experts, top_k, n_shared=1, max_tokens=4, routed_scale=1.0,
                 rms_eps=1e-6, has_norm=False, wbits=4, hbm_slots=0):
        self.cfg = Config(d, f, n_experts, top_k, n_shared, 32, max_tokens, routed_scale, rms_eps,
                          int(has_norm), wbits, hbm_slots)
        self.wbits, self.hbm_slots = wbits, hbm_slots
        h = _vp()
        _check(lib().coli_moe_create(ctypes.byref(self.cfg), ctypes.byref(h)), "coli_moe_create")
        self.h = h
        self.d, self.f, self.E, self.K, self.n_shared = d, f, n_experts, top_k, n_shared
        self.max_tokens, self.has_norm = max_tokens, has_norm

    @classmethod
    def for_workload(cls, wl, max_tokens=None, hbm_slots=0):
        return cls(wl.d, wl.f, wl.E, wl.K, wl.n_shared, max_tokens or wl.T, 1.0, wl.rms_eps,
                   wl.has_norm, wl.wbits, hbm_slots)

    def forward_tiered(self, tier, layer, x, y=None, stream=None):
        """forward of a tiered layer with the tier manager placing its experts
        (coli_moe_forward_tiered)"""
        if y is None:
            y = torch.empty_like(x)
        _check(lib().coli_moe_forward_tiered(self.h, tier.h, layer, _ptr(x), x.shape[0], _ptr(y),
                                             _stream(stream)), "coli_moe_forward_tiered")
        return y

    def prefetch_tiered(self, tier, layer, ids, stream=None):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        _check(lib().coli_moe_prefetch_tiered(self.h, tier.h, layer, ids.ctypes.data, ids.size,
                                              _stream(stream)), "coli_moe_prefetch_tiered")

    def repin_tiered(self, tier, layer, by_usage=False, stream=None):
        _check(lib().coli_moe_repin_tiered(self.h, tier.h, layer, int(by_usage), _stream(stream)),
               "coli_moe_repin_tiered")

    def tier_copies(self):
        """(records, bytes) copied from host memory into the HBM slots since creation"""
        r, b = _i64(), _i64()
        _check(lib().coli_moe_tier_copies(self.h, ctypes.byref(r), ctypes.byref(b)), "coli_moe_tier_copies")
        return r.value, b.value

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            lib().coli_moe_destroy(self.h)
            self.h = _vp()

    def __del__(self):
        if sys.is_finalizing():  # the process is exiting: no native calls during teardown
            return
        try:
            self.close()
        except Exception:
            pass

    def load_router(self, W_r, bias=None, gamma=None, stream=None):
        _check(lib().coli_moe_load_router(self.h, _ptr(W_r), _ptr(bias), _ptr(gamma), _stream(stream)),
               "coli_moe_load_router")

    def load_experts(self, first, count, packed, scales, stream=None):
        _check(lib().coli_moe_load_experts(self.h, first, count, _ptr(packed), _ptr(scales),
                                           _stream(stream)), "coli_moe_load_experts")

    def forward(self, x, y=None, stream=None):
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        _check(lib().coli_moe_forward(self.h, _ptr(x), T, _ptr(y), _stream(stream)), "coli_moe_forward")
        return y

    def forward_profiled(self, x, y, events, stream=None):
        """forward recording 4 torch.cuda.Event objects: before/after routing, after gate/up,
        after down"""
        for e in events:  # torch creates the CUDA event on its first record
            if not e.cuda_event:
                e.record()
        arr = (_vp * len(events))(*[e.cuda_event for e in events])
        _check(lib().coli_moe_forward_profiled(self.h, _ptr(x), x.shape[0], _ptr(y), arr, len(events),
                                               _stream(stream)), "coli_moe_forward_profiled")
        return y

    def forward_host(self, x, y, stream=None):
        _check(lib().coli_moe_forward_host(self.h, _ptr(x), x.shape[0], _ptr(y), _stream(stream)),
               "coli_moe_forward_host")
        return y

    def forward_debug(self, x, want_A=False, stream=None):
        """forward plus every intermediate, as torch tensors on the device"""
        T, d, f, E, K = x.shape[0], self.d, self.f, self.E, self.K
        P = T * K + (T if self.n_shared else 0)
        dev = x.device
        f32, i32, i8 = torch.float32, torch.int32, torch.int8
        shapes = dict(xn=((T, d), f32), qx=((T, d), i8), dx=((T, d // 32), f32),
                      logits=((T, E), f32), scores=((T, E), f32), ids=((T, K), i32),
                      w=((T, K), f32), n_union=((1,), i32), union_ids=((E + 1,), i32),
                      offsets=((E + 2,), i32), pair_token=((P,), i32), pair_rank=((P,), i32),
                      inv=((T, K), i32), g=((P, f), f32), u=((P, f), f32), h=((P, f), f32),
                      qh=((P, f), i8), dh=((P, f // 32), f32), e=((P, d), f32))
        if want_A:
            shapes.update(Ag=((P, f, d // 32), i32), Au=((P, f, d // 32), i32),
                          Ad=((P, d, f // 32), i32))
        out = {k: torch.zeros(s, dtype=t, device=dev) for k, (s, t) in shapes.items()}
        dump = Dump(**{k: v.data_ptr() for k, v in out.items()})
        y = torch.empty_like(x)
        _check(lib().coli_moe_forward_debug(self.h, _ptr(x), T, _ptr(y), ctypes.byref(dump),
                                            _stream(stream)), "coli_moe_forward_debug")
        out["y"] = y
        return out

    def status(self, stream=None):
        return int(lib().coli_moe_status(self.h, _stream(stream)))

    def set_prefill_min(self, min_tokens):
        """batches of at least min_tokens (>= 2) take the tensor-core path, smaller ones the
        decode kernels in one pass of up to 8 tokens or chunks of 8 (coli_moe_set_prefill_min)"""
        _check(lib().coli_moe_set_prefill_min(self.h, min_tokens), "coli_moe_set_prefill_min")

    def inject_fault(self, fault):
        """failure-path test knob (coli_moe_inject_fault): 1 = the next fused one-token forward
        leaves CTA 0 out of the grid barrier, so its bounded waits run out"""
        _check(lib().coli_moe_inject_fault(self.h, fault), "coli_moe_inject_fault")

    def launches(self, T):
        """kernel launches one forward of T tokens makes"""
        n = int(lib().coli_moe_launches(self.h, T))
        if n < 0:
            raise ColiError(n, "coli_moe_launches")
        return n


def stack_forward(layers, x, stream=None):
    arr = (_vp * len(layers))(*[l.h.value for l in layers])
    _check(lib().coli_moe_stack_forward(arr, len(layers), _ptr(x), x.shape[0], _stream(stream)),
           "coli_moe_stack_forward")
    return x


def quantize_i4_rows(w, packed=None, scales=None, stream=None):
    rows, cols = w.shape
    if packed is None:
        packed = torch.empty((rows, cols // 2), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty(rows, dtype=torch.float32, device=w.device)
    _check(lib().coli_quantize_i4_rows(_ptr(w), rows, cols, _ptr(packed), _ptr(scales), _stream(stream)),
           "coli_quantize_i4_rows")
    return packed, scales


def quantize_i8_rows(w, q=None, scales=None, stream=None):
    """int8 rows (one code per byte) and one f32 scale per row (coli_quantize_i8_rows)"""
    rows, cols = w.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.int8, device=w.device)
    if scales is None:
        scales = torch.empty(rows, dtype=torch.float32, device=w.device)
    _check(lib().coli_quantize_i8_rows(_ptr(w), rows, cols, _ptr(q), _ptr(scales), _stream(stream)),
           "coli_quantize_i8_rows")
    return q, scales


def quantize_i2_rows(w, packed=None, scales=None, stream=None):
    """int2 rows (four codes per byte) and one f32 scale per row (coli_quantize_i2_rows)"""
    rows, cols = w.shape
    if packed is None:
        packed = torch.empty((rows, cols // 4), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty(rows, dtype=torch.float32, device=w.device)
    _check(lib().coli_quantize_i2_rows(_ptr(w), rows, cols, _ptr(packed), _ptr(scales), _stream(stream)),
           "coli_quantize_i2_rows")
    return packed, scales


def quantize_rows(w, wbits, out=None, scales=None, stream=None):
    """rows of `wbits` bits per weight into `out` (a uint8 view of the record's bytes)"""
    if wbits == 4:
        return quantize_i4_rows(w, out, scales, stream)
    if wbits == 8:
        return quantize_i8_rows(w, None if out is None else out.view(torch.int8), scales, stream)
    if wbits == 2:
        return quantize_i2_rows(w, out, scales, stream)
    raise ValueError(f"no {wbits}-bit rows")


def route_noalloc(x, W_r, K, bias=None, routed_scale=1.0, stream=None):
    """top-K ids and weights of the tokens x [T,d] (device) under router W_r [E,d] (device),
    through the entry point that allocates nothing"""
    T, d = x.shape
    E = W_r.shape[0]
    ids = torch.empty((T, K), dtype=torch.int32, device=x.device)
    w = torch.empty((T, K), dtype=torch.float32, device=x.device)
    _check(lib().coli_route_noalloc(_ptr(x), T, _ptr(W_r), _ptr(bias), E, d, K, routed_scale,
                                    _ptr(ids), _ptr(w), _stream(stream)), "coli_route_noalloc")
    return ids, w


def quantize_act_q8(x, stream=None):
    q = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    d = torch.empty(x.shape[:-1] + (x.shape[-1] // 32,), dtype=torch.float32, device=x.device)
    _check(lib().coli_quantize_act_q8(_ptr(x), x.numel(), _ptr(q), _ptr(d), _stream(stream)),
           "coli_quantize_act_q8")
    return q, d


TIER_STATS = ("pin_hits", "lru_hits", "misses", "evictions", "prefetch_fetches", "prefetch_used",
              "prefetch_wasted", "repin_fetches")


class Tier:
    """Expert residency tiers of n_layers MoE layers (include/coli_tier.h): host-side decisions
    of which expert records sit in which HBM slots; the caller moves the data."""

    def __init__(self, n_layers, n_experts, n_pin, n_lru):
        self.cfg = TierConfig(n_layers, n_experts, n_pin, n_lru)
        h = _vp()
        _check(lib().coli_tier_create(ctypes.byref(self.cfg), ctypes.byref(h)), "coli_tier_create")
        self.h = h
        self.n_layers, self.n_experts, self.n_pin, self.n_lru = n_layers, n_experts, n_pin, n_lru

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            lib().coli_tier_destroy(self.h)
            self.h = _vp()

    def __del__(self):
        if sys.is_finalizing():  # the process is exiting: no native calls during teardown
            return
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _ids(ids):
        return np.ascontiguousarray(ids, dtype=np.int32)

    def lookup(self, layer, ids):
        """-> dict(cls, slot, fetch_ids, fetch_slots, evict_ids, evict_slots) as int32 arrays"""
        ids = self._ids(ids)
        n = ids.size
        out = {k: np.empty(n, np.int32) for k in
               ("cls", "slot", "fetch_ids", "fetch_slots", "evict_ids", "evict_slots")}
        nf, ne = _i(), _i()
        _check(lib().coli_tier_lookup(self.h, layer, ids.ctypes.data, n, out["cls"].ctypes.data,
                                      out["slot"].ctypes.data, out["fetch_ids"].ctypes.data,
                                      out["fetch_slots"].ctypes.data, ctypes.byref(nf),
                                      out["evict_ids"].ctypes.data, out["evict_slots"].ctypes.data,
                                      ctypes.byref(ne)), "coli_tier_lookup")
        for k in ("fetch_ids", "fetch_slots"):
            out[k] = out[k][:nf.value]
        for k in ("evict_ids", "evict_slots"):
            out[k] = out[k][:ne.value]
        return out

    def prefetch(self, layer, ids):
        """-> dict(fetch_ids, fetch_slots, evict_ids, evict_slots)"""
        ids = self._ids(ids)
        n = ids.size
        out = {k: np.empty(n, np.int32) for k in ("fetch_ids", "fetch_slots", "evict_ids", "evict_slots")}
        nf, ne = _i(), _i()
        _check(lib().coli_tier_prefetch(self.h, layer, ids.ctypes.data, n,
                                        out["fetch_ids"].ctypes.data, out["fetch_slots"].ctypes.data,
                                        ctypes.byref(nf), out["evict_ids"].ctypes.data,
                                        out["evict_slots"].ctypes.data, ctypes.byref(ne)),
               "coli_tier_prefetch")
        for k in ("fetch_ids", "fetch_slots"):
            out[k] = out[k][:nf.value]
        for k in ("evict_ids", "evict_slots"):
            out[k] = out[k][:ne.value]
        return out

    def _pin(self, fn, layer):
        m = max(self.n_pin, 1)
        out = {k: np.empty(m, np.int32) for k in ("fetch_ids", "fetch_slots", "drop_ids", "drop_slots")}
        nf, nd = _i(), _i()
        _check(getattr(lib(), fn)(self.h, layer, out["fetch_ids"].ctypes.data,
                                  out["fetch_slots"].ctypes.data, ctypes.byref(nf),
                                  out["drop_ids"].ctypes.data, out["drop_slots"].ctypes.data,
                                  ctypes.byref(nd)), fn)
        for k in ("fetch_ids", "fetch_slots"):
            out[k] = out[k][:nf.value]
        for k in ("drop_ids", "drop_slots"):
            out[k] = out[k][:nd.value]
        return out

    def repin(self, layer):
        """live repin by session heat -> dict(fetch_ids, fetch_slots, drop_ids, drop_slots)"""
        return self._pin("coli_tier_repin", layer)

    def autopin(self, layer):
        """start-up pinning by usage heat -> dict(fetch_ids, fetch_slots, drop_ids, drop_slots)"""
        return self._pin("coli_tier_autopin", layer)

    def decay(self):
        """halve every layer's session heat"""
        _check(lib().coli_tier_decay(self.h), "coli_tier_decay")

    def session_heat(self, layer):
        h = np.empty(self.n_experts, np.int64)
        _check(lib().coli_tier_session_heat(self.h, layer, h.ctypes.data), "coli_tier_session_heat")
        return h

    def state(self, layer):
        """-> (pinned ascending, LRU list most recent first, slot_of[n_experts])"""
        pinned = np.empty(max(self.n_pin, 1), np.int32)
        lru = np.empty(self.n_lru, np.int32)
        slot_of = np.empty(self.n_experts, np.int32)
        npin, nlru = _i(), _i()
        _check(lib().coli_tier_state(self.h, layer, pinned.ctypes.data, ctypes.byref(npin),
                                     lru.ctypes.data, ctypes.byref(nlru), slot_of.ctypes.data),
               "coli_tier_state")
        return pinned[:npin.value], lru[:nlru.value], slot_of

    def heat(self, layer):
        h = np.empty(self.n_experts, np.int64)
        _check(lib().coli_tier_heat(self.h, layer, h.ctypes.data), "coli_tier_heat")
        return h

    def set_heat(self, layer, heat):
        heat = np.ascontiguousarray(heat, dtype=np.int64)
        if heat.size != self.n_experts:
            raise ValueError(f"heat needs {self.n_experts} counts, got {heat.size}")
        _check(lib().coli_tier_set_heat(self.h, layer, heat.ctypes.data), "coli_tier_set_heat")

    def stats(self):
        st = np.empty(len(TIER_STATS), np.int64)
        _check(lib().coli_tier_stats(self.h, st.ctypes.data), "coli_tier_stats")
        return dict(zip(TIER_STATS, (int(v) for v in st)))

    def save_usage(self, path):
        _check(lib().coli_tier_save_usage(self.h, os.fsencode(path)), "coli_tier_save_usage")

    def load_usage(self, path):
        _check(lib().coli_tier_load_usage(self.h, os.fsencode(path)), "coli_tier_load_usage")
