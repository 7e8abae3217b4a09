"""GPU parity of expert layers with int8 rows and with int2 rows ("colibrì 架构概述" §3.1: int8
rows for the dense part and the MTP head, quantize_rows and dot_i8i8; int2 packed rows,
pack_int2 and matmul_i2, experimental), against the CPU oracle with the same code width:
the device packers bit for bit, every stage of the layer bit for bit (fp32 stages follow the
canonical order on both sides), the output within 1e-4 of the oracle's fp64 evaluation, and the
int32 block dots of sampled rows against brute-force sums over the decoded codes.  All calls go
through the C ABI."""
import numpy as np
import pytest
import torch

from gen import workloads as W
from int4_routed_expert_quantize_gb300 import coli, synthetic
from oracle import oracle as O

from .gpu_util import normwise_rel, to_np
from .test_gpu_parity import TOL, _compare_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _rows():
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((130, 512)) * rng.uniform(1e-3, 5, (130, 1))).astype(np.float32)
    w[3] = 0.0
    w[4, :] = 1e-30
    w[5, ::3] = -2.5
    w[6, 7] = 3.0e38
    return w


def test_int8_row_packer_bit_exact():
    w = _rows()
    q, s = coli.quantize_i8_rows(torch.from_numpy(w).cuda())
    oq, os_ = O.quantize_i8_rows(w)
    assert np.array_equal(to_np(q), oq)
    assert np.array_equal(to_np(s).view(np.uint32), os_.view(np.uint32))


def test_int2_row_packer_bit_exact():
    w = _rows()
    pk, s = coli.quantize_i2_rows(torch.from_numpy(w).cuda())
    opk, os_ = O.quantize_i2_rows(w)
    assert np.array_equal(to_np(pk), opk)
    assert np.array_equal(to_np(s).view(np.uint32), os_.view(np.uint32))


def test_record_bytes_of_every_width():
    for wb in (4, 8, 2):
        assert coli.expert_record_bytes(6144, 2048, wb) == 3 * 6144 * 2048 * wb // 8 + 4 * (2 * 2048 + 6144)
    assert W.WORKLOADS["glm_i8_decode_t1"].expert_bytes == 37_789_696


def _codes(rec, wl, which):
    """decoded codes [rows, cols] of the gate (0), up (1) or down (2) matrix of a canonical record"""
    d, f, wb = wl.d, wl.f, wl.wbits
    rows, cols = (f, d) if which < 2 else (d, f)
    mat = f * d * wb // 8
    raw = rec[which * mat:(which + 1) * mat].reshape(rows, cols * wb // 8)
    if wb == 8:
        return raw.view(np.int8).astype(np.int64)
    fields = np.stack([(raw >> (2 * k)) & 3 for k in range(4)], axis=-1).reshape(rows, cols).astype(np.int64)
    return np.where(fields >= 2, fields - 4, fields)


def _check_block_dots(L, OL, x, rows=(0, 5, 31, 100)):
    """Ag, Au and Ad of sampled rows against brute-force sums over the decoded codes"""
    wl = OL.wl
    g = L.forward_debug(torch.from_numpy(x).cuda(), want_A=True)
    torch.cuda.synchronize()
    o = OL.forward(x)
    Ag, Au, Ad = (to_np(g[k]) for k in ("Ag", "Au", "Ad"))
    nu = int(to_np(g["n_union"])[0])
    offs = to_np(g["offsets"])[:nu + 1]
    uids = to_np(g["union_ids"])[:nu]
    pt = to_np(g["pair_token"])
    for s_ in range(nu):
        rec, _ = OL.recs[int(uids[s_])]
        Wg, Wu, Wd = (_codes(rec, wl, k) for k in range(3))
        for p in range(offs[s_], offs[s_ + 1]):
            qx = o["qx"][pt[p]].astype(np.int64).reshape(-1, 32)
            qh = o["qh"][p].astype(np.int64).reshape(-1, 32)
            for r in rows:
                if r < wl.f:
                    assert np.array_equal(Ag[p, r], (Wg[r].reshape(-1, 32) * qx).sum(axis=1))
                    assert np.array_equal(Au[p, r], (Wu[r].reshape(-1, 32) * qx).sum(axis=1))
                if r < wl.d:
                    assert np.array_equal(Ad[p, r], (Wd[r].reshape(-1, 32) * qh).sum(axis=1))


@pytest.fixture(scope="module", params=[8, 2])
def tiny_w(request):
    wl = W.WORKLOADS[f"tiny_i{request.param}_t1"]
    L = synthetic.build_layer(wl, max_tokens=16)
    yield wl, L, O.Layer(wl)
    L.close()


@pytest.mark.parametrize("T,token0", [(1, 0), (3, 40), (8, 7)])
def test_tiny_width_layer_all_stages(tiny_w, T, token0):
    wl, L, OL = tiny_w
    assert L.launches(T) == 3  # the decode kernels for every batch size of these widths
    _compare_layer(L, OL, W.x_host(wl, T, token0), want_A=False)


def test_tiny_width_block_dots_brute_force(tiny_w):
    wl, L, OL = tiny_w
    _check_block_dots(L, OL, W.x_host(wl, 2, 70))


def test_tiny_width_chunked_production(tiny_w):
    """11 tokens: a chunk of 8 and one of 3, production instances, against the oracle"""
    wl, L, OL = tiny_w
    x = W.x_host(wl, 11, token0=500)
    y = to_np(L.forward(torch.from_numpy(x).cuda()))
    o = OL.forward(x, want_dump=False)
    assert np.array_equal(y, o["y"])
    assert normwise_rel(y, o["y64"]) <= TOL


@pytest.mark.parametrize("wb", [8, 2])
def test_glm_width_layer(wb):
    """the GLM-shaped layer with int8 or int2 experts: one token (all stages), then a 4-token
    batch with the shared selection bias through the production kernels"""
    wl = W.WORKLOADS[f"glm_i{wb}_decode_t1"]
    L = synthetic.build_layer(wl, max_tokens=4)
    OL = O.Layer(wl)
    g, _ = _compare_layer(L, OL, W.x_host(wl, 1, 3), want_A=False)
    assert int(to_np(g["n_union"])[0]) == 9
    L.close()
    wv = W.Workload(f"glm_i{wb}_verify_t4", d=6144, f=2048, E=256, K=8, n_shared=1, T=4,
                    bias="overlap", wbits=wb)
    L = synthetic.build_layer(wv, max_tokens=4)
    OL = O.Layer(wv)
    x = W.x_host(wv, 4, 11)
    y = to_np(L.forward(torch.from_numpy(x).cuda()))
    o = OL.forward(x, want_dump=False)
    assert np.array_equal(y, o["y"])
    assert normwise_rel(y, o["y64"]) <= TOL
    L.close()
