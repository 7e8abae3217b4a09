"""ctypes front-end of the plain C oracle (oracle.c).  TEST INFRASTRUCTURE ONLY.

Used by tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg; the product
library never imports it.  Weights come from the shared seeded generator (gen/) and are
quantised here by the oracle's own int4 packer.
"""
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.environ.get("COLI_ORACLE_SO") or os.path.join(HERE, "liboracle.so")  # a sanitized build may stand in
QB = 32

_i, _f, _vp, _i64 = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int64


class Cfg(ctypes.Structure):
    _fields_ = [("d", _i), ("f", _i), ("n_experts", _i), ("top_k", _i), ("n_shared", _i),
                ("qblock", _i), ("routed_scale", _f), ("rms_eps", _f), ("has_norm", _i),
                ("wbits", _i)]


_DUMP_FIELDS = ["xn", "qx", "dx", "logits", "scores", "ids", "w", "n_union", "union_ids", "offsets",
                "pair_token", "pair_rank", "inv", "g", "u", "h", "qh", "dh", "e", "Ag", "Au", "Ad"]


class Dump(ctypes.Structure):
    _fields_ = [(n, _vp) for n in _DUMP_FIELDS]


def build(openmp=True, out=None, sanitize=False):
    """Compile oracle.c into `out` (default: the library the tests load); with `sanitize`,
    under AddressSanitizer and UndefinedBehaviorSanitizer."""
    flags = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math"]
    if openmp:
        flags.append("-fopenmp")
    if sanitize:
        flags += ["-g", "-fno-omit-frame-pointer", "-fsanitize=address,undefined",
                  "-fno-sanitize-recover=undefined"]
    subprocess.check_call(flags + [os.path.join(HERE, "oracle.c"), "-o", out or SO, "-lm"])


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(SO):
            build()
        L = ctypes.CDLL(SO)
        L.orc_quantize_i4_rows.argtypes = [_vp, _i64, _i, _vp, _vp]
        L.orc_i4_get.argtypes = [_vp, _i]
        L.orc_i4_get.restype = _i
        L.orc_pack_i4_row.argtypes = [_vp, _i, _vp]
        L.orc_quantize_q8.argtypes = [_vp, _i64, _vp, _vp]
        L.orc_exp.argtypes = [_f]
        L.orc_exp.restype = _f
        L.orc_exp_n.argtypes = [_vp, _vp, _i64]
        L.orc_sigmoid.argtypes = [_f]
        L.orc_sigmoid.restype = _f
        L.orc_silu_mul.argtypes = [_f, _f]
        L.orc_silu_mul.restype = _f
        L.orc_pairwise32.argtypes = [_vp]
        L.orc_pairwise32.restype = _f
        L.orc_canon_dot.argtypes = [_vp, _vp, _i]
        L.orc_canon_dot.restype = _f
        L.orc_canon_blocksum.argtypes = [_vp, _vp, _i]
        L.orc_canon_blocksum.restype = _f
        L.orc_block_dot.argtypes = [_vp, _vp, _i]
        L.orc_block_dot.restype = ctypes.c_int32
        L.orc_i4_matvec.argtypes = [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp]
        L.orc_quantize_i8_rows.argtypes = [_vp, _i64, _i, _vp, _vp]
        L.orc_i8_block_dot.argtypes = [_vp, _vp, _i]
        L.orc_i8_block_dot.restype = ctypes.c_int32
        L.orc_i8_matvec.argtypes = [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp]
        L.orc_i2_get.argtypes = [_vp, _i]
        L.orc_i2_get.restype = _i
        L.orc_pack_i2_row.argtypes = [_vp, _i, _vp]
        L.orc_quantize_i2_rows.argtypes = [_vp, _i64, _i, _vp, _vp]
        L.orc_i2_block_dot.argtypes = [_vp, _vp, _i]
        L.orc_i2_block_dot.restype = ctypes.c_int32
        L.orc_i2_matvec.argtypes = [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp]
        L.orc_topk.argtypes = [_vp, _i, _i, _vp]
        L.orc_route_token.argtypes = [_vp, _vp, _vp, _i, _i, _i, _f, _vp, _vp, _vp, _vp]
        L.orc_rmsnorm.argtypes = [_vp, _vp, _i, _f, _vp]
        L.orc_union_bucket.argtypes = [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]
        L.orc_union_bucket.restype = _i
        L.orc_expert_ffn_bits.argtypes = [_i, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                                          _vp, _vp]
        L.orc_expert_ffn_bits.restype = _i
        L.orc_expert_ffn.argtypes = [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _vp, _vp]
        L.orc_moe_forward.argtypes = [ctypes.POINTER(Cfg), _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                                      _vp, ctypes.POINTER(Dump)]
        L.orc_moe_forward.restype = _i
        L.orc_moe_dequant64.argtypes = [ctypes.POINTER(Cfg), _vp, _i, _vp, _vp, _vp, _vp, _vp, _vp]
        L.orc_moe_dequant64.restype = _i
        L.orc_num_threads.restype = _i
        L.orc_set_num_threads.argtypes = [_i]
        L.orc_set_num_threads.restype = None
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def cfg_of(wl, routed_scale=1.0, wbits=4):
    return Cfg(wl.d, wl.f, wl.E, wl.K, wl.n_shared, QB, routed_scale, wl.rms_eps, int(wl.has_norm),
               wbits)


# ---------------- formats ----------------

def quantize_i4_rows(w):
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    packed = np.empty((rows, cols // 2), dtype=np.uint8)
    scales = np.empty(rows, dtype=np.float32)
    lib().orc_quantize_i4_rows(w.ctypes.data, rows, cols, packed.ctypes.data, scales.ctypes.data)
    return packed, scales


def quantize_i8_rows(w):
    """int8 rows (one code per byte) and one f32 scale per row"""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    q = np.empty((rows, cols), dtype=np.int8)
    scales = np.empty(rows, dtype=np.float32)
    lib().orc_quantize_i8_rows(w.ctypes.data, rows, cols, q.ctypes.data, scales.ctypes.data)
    return q, scales


def quantize_i2_rows(w):
    """int2 rows (four codes per byte) and one f32 scale per row"""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    packed = np.empty((rows, cols // 4), dtype=np.uint8)
    scales = np.empty(rows, dtype=np.float32)
    lib().orc_quantize_i2_rows(w.ctypes.data, rows, cols, packed.ctypes.data, scales.ctypes.data)
    return packed, scales


def quantize_q8(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.empty(x.shape, dtype=np.int8)
    d = np.empty(x.shape[:-1] + (x.shape[-1] // QB,), dtype=np.float32)
    lib().orc_quantize_q8(x.ctypes.data, x.size, q.ctypes.data, d.ctypes.data)
    return q, d


def exp(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    lib().orc_exp_n(x.ctypes.data, y.ctypes.data, x.size)
    return y


def canon_dot(a, b):
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    return lib().orc_canon_dot(a.ctypes.data, b.ctypes.data, a.size)


def canon_blocksum(d, A):
    d = np.ascontiguousarray(d, dtype=np.float32)
    A = np.ascontiguousarray(A, dtype=np.int32)
    return lib().orc_canon_blocksum(d.ctypes.data, A.ctypes.data, d.size)


def pairwise32(p):
    p = np.ascontiguousarray(p, dtype=np.float32)
    assert p.size == 32
    return lib().orc_pairwise32(p.ctypes.data)


def i4_matvec(W, s, cols, qx, dx, want_A=False):
    rows = W.shape[0]
    out = np.empty(rows, dtype=np.float32)
    A = np.empty((rows, cols // QB), dtype=np.int32) if want_A else None
    lib().orc_i4_matvec(W.ctypes.data, s.ctypes.data, rows, cols, qx.ctypes.data, dx.ctypes.data,
                        out.ctypes.data, _p(A))
    return out, A


def i8_matvec(W, s, cols, qx, dx, want_A=False):
    W = np.ascontiguousarray(W, dtype=np.int8)
    rows = W.shape[0]
    out = np.empty(rows, dtype=np.float32)
    A = np.empty((rows, cols // QB), dtype=np.int32) if want_A else None
    lib().orc_i8_matvec(W.ctypes.data, s.ctypes.data, rows, cols, qx.ctypes.data, dx.ctypes.data,
                        out.ctypes.data, _p(A))
    return out, A


def i2_matvec(W, s, cols, qx, dx, want_A=False):
    W = np.ascontiguousarray(W, dtype=np.uint8)
    rows = W.shape[0]
    out = np.empty(rows, dtype=np.float32)
    A = np.empty((rows, cols // QB), dtype=np.int32) if want_A else None
    lib().orc_i2_matvec(W.ctypes.data, s.ctypes.data, rows, cols, qx.ctypes.data, dx.ctypes.data,
                        out.ctypes.data, _p(A))
    return out, A


def expert_ffn_bits(bits, rec, sc, d, f, qx, dx):
    """one expert with int8 / int4 / int2 rows on one token -> dict(qh, dh, e, g, u, h)"""
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    sc = np.ascontiguousarray(sc, dtype=np.float32)
    out = dict(qh=np.empty(f, dtype=np.int8), dh=np.empty(f // QB, dtype=np.float32),
               e=np.empty(d, dtype=np.float32), g=np.empty(f, dtype=np.float32),
               u=np.empty(f, dtype=np.float32), h=np.empty(f, dtype=np.float32))
    rc = lib().orc_expert_ffn_bits(bits, rec.ctypes.data, sc.ctypes.data, d, f, qx.ctypes.data,
                                   dx.ctypes.data, *(out[k].ctypes.data for k in
                                                     ("qh", "dh", "e", "g", "u", "h")))
    if rc != 0:
        raise ValueError(f"no {bits}-bit rows")
    return out


def topk(sel, K):
    sel = np.ascontiguousarray(sel, dtype=np.float32)
    ids = np.empty(K, dtype=np.int32)
    lib().orc_topk(sel.ctypes.data, sel.size, K, ids.ctypes.data)
    return ids


def rmsnorm(x, gamma, eps):
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    lib().orc_rmsnorm(x.ctypes.data, gamma.ctypes.data, x.size, eps, out.ctypes.data)
    return out


def route_token(Wr, bias, x, K, routed_scale=1.0):
    E, d = Wr.shape
    logits = np.empty(E, dtype=np.float32)
    scores = np.empty(E, dtype=np.float32)
    ids = np.empty(K, dtype=np.int32)
    w = np.empty(K, dtype=np.float32)
    lib().orc_route_token(Wr.ctypes.data, _p(bias), x.ctypes.data, E, d, K, routed_scale,
                          logits.ctypes.data, scores.ctypes.data, ids.ctypes.data, w.ctypes.data)
    return logits, scores, ids, w


def union_bucket(ids, E, n_shared):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, K = ids.shape
    P = T * K + (T if n_shared else 0)
    union_ids = np.empty(E + 1, dtype=np.int32)
    offsets = np.empty(E + 2, dtype=np.int32)
    pair_token = np.empty(P, dtype=np.int32)
    pair_rank = np.empty(P, dtype=np.int32)
    inv = np.empty((T, K), dtype=np.int32)
    nu = lib().orc_union_bucket(ids.ctypes.data, T, K, E, n_shared, union_ids.ctypes.data,
                                offsets.ctypes.data, pair_token.ctypes.data, pair_rank.ctypes.data,
                                inv.ctypes.data)
    return dict(n_union=nu, union_ids=union_ids[:nu], offsets=offsets[:nu + 1],
                pair_token=pair_token, pair_rank=pair_rank, inv=inv)


def expert_ffn(rec, sc, d, f, qx, dx, want_A=False):
    qh = np.empty(f, dtype=np.int8)
    dh = np.empty(f // QB, dtype=np.float32)
    e = np.empty(d, dtype=np.float32)
    g = np.empty(f, dtype=np.float32)
    u = np.empty(f, dtype=np.float32)
    h = np.empty(f, dtype=np.float32)
    Ag = np.empty((f, d // QB), dtype=np.int32) if want_A else None
    Au = np.empty((f, d // QB), dtype=np.int32) if want_A else None
    Ad = np.empty((d, f // QB), dtype=np.int32) if want_A else None
    lib().orc_expert_ffn(rec.ctypes.data, sc.ctypes.data, d, f, qx.ctypes.data, dx.ctypes.data,
                         qh.ctypes.data, dh.ctypes.data, e.ctypes.data, g.ctypes.data, u.ctypes.data,
                         h.ctypes.data, _p(Ag), _p(Au), _p(Ad))
    return dict(qh=qh, dh=dh, e=e, g=g, u=u, h=h, Ag=Ag, Au=Au, Ad=Ad)


# ---------------- expert records from the generator ----------------

def expert_record_from_float(gate, up, down, wbits=4):
    """[gate | up | down] packed codes (int4 nibbles, int8 bytes or int2 fields, by the oracle's
    own packers) and [s_g | s_u | s_d] scales, the three matrices of an expert stored adjacently"""
    quant = {4: quantize_i4_rows, 8: quantize_i8_rows, 2: quantize_i2_rows}[wbits]
    parts = [quant(m) for m in (gate, up, down)]
    rec = np.concatenate([np.ascontiguousarray(p).view(np.uint8).ravel() for p, _ in parts])
    sc = np.concatenate([s for _, s in parts])
    return rec, sc


def expert_record(wl, layer, expert):
    from gen import workloads
    return expert_record_from_float(*workloads.expert_float_host(wl, layer, expert),
                                    wbits=getattr(wl, "wbits", 4))


# ---------------- full layer ----------------

def forward(wl, x, Wr, bias, gamma, recs, want_dump=True, want_A=False, want_y64=True,
            routed_scale=1.0, wbits=4):
    """recs: dict expert id -> (rec, sc) for at least every selected expert and the shared one;
    wbits: the records' code width (4, or 8 / 2 for int8 / int2 experts, without the per-block
    accumulator dumps)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    T, d = x.shape
    E, K, f = wl.E, wl.K, wl.f
    P = T * K + (T if wl.n_shared else 0)
    if want_A and wbits != 4:
        raise ValueError("per-block accumulators are dumped for int4 experts only")
    cfg = cfg_of(wl, routed_scale, wbits)
    y = np.empty((T, d), dtype=np.float32)
    y64 = np.empty((T, d), dtype=np.float64) if want_y64 else None
    recp = (ctypes.c_void_p * (E + 1))()
    scp = (ctypes.c_void_p * (E + 1))()
    for k, (r, s) in recs.items():
        recp[k] = r.ctypes.data
        scp[k] = s.ctypes.data
    out = {}
    dump = None
    if want_dump:
        shapes = dict(xn=((T, d), np.float32), qx=((T, d), np.int8), dx=((T, d // QB), np.float32),
                      logits=((T, E), np.float32), scores=((T, E), np.float32),
                      ids=((T, K), np.int32), w=((T, K), np.float32), n_union=((1,), np.int32),
                      union_ids=((E + 1,), np.int32), offsets=((E + 2,), np.int32),
                      pair_token=((P,), np.int32), pair_rank=((P,), np.int32),
                      inv=((T, K), np.int32), g=((P, f), np.float32), u=((P, f), np.float32),
                      h=((P, f), np.float32), qh=((P, f), np.int8), dh=((P, f // QB), np.float32),
                      e=((P, d), np.float32))
        if want_A:
            shapes.update(Ag=((P, f, d // QB), np.int32), Au=((P, f, d // QB), np.int32),
                          Ad=((P, d, f // QB), np.int32))
        for k, (shp, dt) in shapes.items():
            out[k] = np.zeros(shp, dtype=dt)
        dump = Dump(**{k: out[k].ctypes.data for k in out})
    rc = lib().orc_moe_forward(ctypes.byref(cfg), x.ctypes.data, T, Wr.ctypes.data, _p(bias),
                               _p(gamma), recp, scp, y.ctypes.data, _p(y64),
                               ctypes.byref(dump) if dump is not None else None)
    if rc:
        raise RuntimeError("orc_moe_forward failed (missing expert weights?)")
    out["y"] = y
    out["y64"] = y64
    if want_dump:
        nu = int(out["n_union"][0])
        out["union_ids"] = out["union_ids"][:nu]
        out["offsets"] = out["offsets"][:nu + 1]
    return out


def dequant64(wl, xn, ids, w, recs, x_resid=None):
    xn = np.ascontiguousarray(xn, dtype=np.float32)
    T = xn.shape[0]
    y = np.empty((T, wl.d), dtype=np.float64)
    recp = (ctypes.c_void_p * (wl.E + 1))()
    scp = (ctypes.c_void_p * (wl.E + 1))()
    for k, (r, s) in recs.items():
        recp[k] = r.ctypes.data
        scp[k] = s.ctypes.data
    rc = lib().orc_moe_dequant64(ctypes.byref(cfg_of(wl)), xn.ctypes.data, T,
                                 np.ascontiguousarray(ids, dtype=np.int32).ctypes.data,
                                 np.ascontiguousarray(w, dtype=np.float32).ctypes.data, recp, scp,
                                 _p(x_resid), y.ctypes.data)
    if rc:
        raise RuntimeError("orc_moe_dequant64 failed")
    return y


def route_only(wl, x, Wr, bias, gamma):
    """(xn, ids [T,K], w [T,K]) for each token: RMSNorm when the layer has one, then the router"""
    T = x.shape[0]
    xn = np.empty_like(x)
    ids = np.empty((T, wl.K), dtype=np.int32)
    w = np.empty((T, wl.K), dtype=np.float32)
    for t in range(T):
        xn[t] = rmsnorm(x[t], gamma, wl.rms_eps) if wl.has_norm else x[t]
        _, _, ids[t], w[t] = route_token(Wr, bias, np.ascontiguousarray(xn[t]), wl.K)
    return xn, ids, w


class Layer:
    """One synthetic layer on the oracle side: router inputs plus an on-demand cache of expert
    records (only the experts a batch touches are generated and quantised)."""

    def __init__(self, wl, layer=0):
        from gen import workloads
        self.wl, self.layer = wl, layer
        self.Wr = workloads.router_host(wl, layer)
        self.bias = workloads.bias_host(wl, layer)
        self.gamma = workloads.gamma_host(wl, layer) if wl.has_norm else None
        self.recs = {}

    def ensure(self, experts):
        for e in experts:
            e = int(e)
            if e not in self.recs:
                self.recs[e] = expert_record(self.wl, self.layer, e)

    def forward(self, x, **kw):
        _, ids, _ = route_only(self.wl, x, self.Wr, self.bias, self.gamma)
        need = set(np.unique(ids).tolist())
        if self.wl.n_shared:
            need.add(self.wl.E)
        self.ensure(sorted(need))
        kw.setdefault("wbits", getattr(self.wl, "wbits", 4))
        return forward(self.wl, x, self.Wr, self.bias, self.gamma, self.recs, **kw)
