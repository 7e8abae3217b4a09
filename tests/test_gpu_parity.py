"""GPU parity: every stage of the CUDA path against the CPU oracle on the same seeded inputs.

Bar (stated per check): bit-exact for integer work (q8 codes, int4 bytes, int32 block dots,
top-k ids, union/bucket) and -- because both sides follow the same canonical fp32 order of
operations -- for every fp32 stage too; the official output bar is max normwise relative
error <= 1e-4 against the oracle's fp64 evaluation of the same integer codes.
All calls go through the C ABI (libcoli_moe.so) via the ctypes binding.
"""
import numpy as np
import pytest
import torch

from gen import workloads as W
from int4_routed_expert_quantize_gb300 import coli, synthetic
from oracle import oracle as O

from .gpu_util import normwise_rel, to_np

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


# ------------------------------------------------------------------ formats ---------------

def test_quantize_i4_rows_bit_exact():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((300, 512)) * rng.uniform(1e-3, 5, (300, 1))).astype(np.float32)
    w[7] = 0.0
    w[8, :] = 1e-30
    w[9, ::2] = -3.5
    pk, sc = coli.quantize_i4_rows(torch.from_numpy(w).cuda())
    opk, osc = O.quantize_i4_rows(w)
    assert np.array_equal(to_np(pk), opk)
    assert np.array_equal(to_np(sc).view(np.uint32), osc.view(np.uint32))


def test_quantize_i4_generated_expert_bit_exact():
    wl = W.WORKLOADS["glm_decode_t1"]
    gate, _, down = W.expert_float_host(wl, 0, 17)
    for m in (gate, down):
        pk, sc = coli.quantize_i4_rows(torch.from_numpy(m).cuda())
        opk, osc = O.quantize_i4_rows(m)
        assert np.array_equal(to_np(pk), opk)
        assert np.array_equal(to_np(sc), osc)


def test_device_generator_matches_host():
    wl = W.WORKLOADS["glm_decode_t1"]
    g = torch.empty((wl.f, wl.d), device="cuda")
    u = torch.empty_like(g)
    dn = torch.empty((wl.d, wl.f), device="cuda")
    W.expert_float_dev(wl, 0, 5, g, u, dn)
    hg, hu, hd = W.expert_float_host(wl, 0, 5)
    assert np.array_equal(to_np(g), hg) and np.array_equal(to_np(u), hu) and np.array_equal(to_np(dn), hd)
    x = synthetic.x_tokens(wl, 3, token0=7)
    assert np.array_equal(to_np(x), W.x_host(wl, 3, token0=7))


def test_quantize_act_q8_bit_exact():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(32 * 999) * rng.uniform(1e-3, 100, 32 * 999)).astype(np.float32)
    x[64:96] = 0.0
    x[96] = 3.4e38
    q, d = coli.quantize_act_q8(torch.from_numpy(x).cuda())
    oq, od = O.quantize_q8(x)
    assert np.array_equal(to_np(q), oq) and np.array_equal(to_np(d), od)


# ------------------------------------------------------------------ whole layer -----------

def _compare_layer(L, OL, x, want_A):
    wl = OL.wl
    g = L.forward_debug(torch.from_numpy(x).cuda(), want_A=want_A)
    torch.cuda.synchronize()
    o = OL.forward(x, want_A=want_A)
    nu = int(to_np(g["n_union"])[0])
    assert nu == o["n_union"][0]
    exact = {k: to_np(g[k]) for k in ("xn", "qx", "dx", "logits", "scores", "ids", "w", "inv",
                                      "pair_token", "pair_rank", "g", "u", "h", "qh", "dh", "e")}
    exact["union_ids"] = to_np(g["union_ids"])[:nu]
    exact["offsets"] = to_np(g["offsets"])[:nu + 1]
    if want_A:
        for k in ("Ag", "Au", "Ad"):
            exact[k] = to_np(g[k])
    for k, v in exact.items():
        ov = o[k]
        assert v.shape == ov.shape, k
        assert np.array_equal(v.view(np.uint8), np.ascontiguousarray(ov).view(np.uint8)), \
            f"stage {k} differs from the oracle"
    y = to_np(g["y"])
    assert normwise_rel(y, o["y64"]) <= TOL
    assert np.array_equal(y, o["y"])
    return g, o


@pytest.fixture(scope="module")
def tiny():
    wl = W.WORKLOADS["tiny_t1"]
    L = synthetic.build_layer(wl, max_tokens=8)
    OL = O.Layer(wl)
    yield wl, L, OL
    L.close()


@pytest.mark.parametrize("T,token0", [(1, 0), (2, 5), (3, 100), (4, 9)])
def test_tiny_layer_all_stages(tiny, T, token0):
    wl, L, OL = tiny
    _compare_layer(L, OL, W.x_host(wl, T, token0), want_A=True)


def test_tiny_batch_invariance(tiny):
    wl, L, OL = tiny
    x = synthetic.x_tokens(wl, 4, token0=40)
    yb = to_np(L.forward(x))
    for t in range(4):
        y1 = to_np(L.forward(x[t:t + 1].contiguous()))
        assert np.array_equal(yb[t], y1[0])


def test_tiny_chunked_batch(tiny):
    """a 7-token batch in one union pass: each token still matches the oracle"""
    wl, L, OL = tiny
    x = W.x_host(wl, 7, token0=300)
    y = to_np(L.forward(torch.from_numpy(x).cuda()))
    o = OL.forward(x)
    assert np.array_equal(y, o["y"])
    assert normwise_rel(y, o["y64"]) <= TOL


def test_tiny_host_buffers(tiny):
    wl, L, OL = tiny
    x = torch.from_numpy(W.x_host(wl, 3, token0=77)).pin_memory()
    y = torch.empty_like(x).pin_memory()
    L.forward_host(x, y)
    ref = to_np(L.forward(x.cuda()))
    assert np.array_equal(y.numpy(), ref)
    assert L.status() == 0


def test_tiny_profiled_matches_forward(tiny):
    wl, L, OL = tiny
    x = synthetic.x_tokens(wl, 3, token0=55)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    y = torch.empty_like(x)
    L.forward_profiled(x, y, ev)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(y), to_np(L.forward(x)))
    assert all(ev[i].elapsed_time(ev[i + 1]) >= 0 for i in range(3))


def test_tiny_edge_cases(tiny):
    wl, L, OL = tiny
    x = synthetic.x_tokens(wl, 2)
    lib = coli.lib()
    assert lib.coli_moe_forward(L.h, x.data_ptr(), 0, x.data_ptr(), None) == 0  # T = 0: no-op
    assert lib.coli_moe_forward(L.h, x.data_ptr(), 9, x.data_ptr(), None) == -1  # T > max_tokens
    assert lib.coli_moe_forward(L.h, x.data_ptr(), -1, x.data_ptr(), None) == -1
    assert lib.coli_moe_forward(L.h, x.data_ptr(), 2, x.data_ptr(), None) == -1  # in place without norm
    y = torch.empty_like(x)
    assert lib.coli_moe_forward(L.h, x.data_ptr(), 2, x[1:].data_ptr(), None) == -1  # overlap
    assert lib.coli_moe_forward(L.h, x.data_ptr(), 2, y.data_ptr(), None) == 0
    assert lib.coli_moe_load_experts(L.h, 30, 5, x.data_ptr(), x.data_ptr(), None) == -1  # ids > E
    assert lib.coli_moe_forward(L.h, x.data_ptr() + 4, 1, y.data_ptr(), None) == -1  # misaligned x


def test_forward_before_load_is_state_error():
    L = coli.MoeLayer(512, 256, 32, 4, max_tokens=2)
    x = torch.zeros((1, 512), device="cuda")
    with pytest.raises(coli.ColiError) as ei:
        L.forward(x)
    assert ei.value.status == -3
    L.close()


def test_forced_all_experts_and_no_shared():
    """K = E (every expert selected) and a layer without the shared expert"""
    base = W.WORKLOADS["tiny_t1"]
    for wl in (W.Workload("tiny_dense", d=512, f=256, E=32, K=32, n_shared=1, T=2),
               W.Workload("tiny_noshared", d=512, f=256, E=32, K=4, n_shared=0, T=3)):
        L = synthetic.build_layer(wl, max_tokens=wl.T)
        OL = O.Layer(wl)
        _compare_layer(L, OL, W.x_host(wl, wl.T, 3), want_A=False)
        L.close()
    assert base.K == 4


def test_wide_selection_odd_expert_count():
    """E > 256 (the round-based top-K) with E not a multiple of 4 (scores loaded without the
    bulk copy), K = 6, T = 4 tokens, a zipf selection bias: every stage bit-exact"""
    wl = W.Workload("tiny_wide", d=256, f=128, E=301, K=6, n_shared=1, T=4, bias="zipf")
    L = synthetic.build_layer(wl, max_tokens=4)
    OL = O.Layer(wl)
    for T, token0 in ((1, 2), (4, 40)):
        _compare_layer(L, OL, W.x_host(wl, T, token0), want_A=False)
    L.close()


def test_selection_ties_go_to_the_lower_id():
    """Router rows copied so that two experts score exactly alike: once at the boundary of the
    top-K (an unselected lower id takes the last place) and once at the top (the two keep id
    order); both sides must make the same choices, and the ties must really occur"""
    wl = W.WORKLOADS["tiny_t1"]
    L = synthetic.build_layer(wl, max_tokens=4)
    OL = O.Layer(wl)
    x = W.x_host(wl, 2, 11)
    _, ids, _ = O.route_only(wl, x, OL.Wr, OL.bias, OL.gamma)
    last = int(ids[0][wl.K - 1])
    lower = [e for e in range(last) if e not in ids[0]]
    assert lower, "token 0 needs an unselected expert below its last pick"
    u = lower[0]
    top = int(ids[1][0])
    v = max(e for e in range(wl.E) if e not in ids[1] and e != u and e not in ids[0])
    Wr = OL.Wr.copy()
    Wr[u] = Wr[last]
    Wr[v] = Wr[top]
    OL.Wr = Wr
    L.load_router(torch.from_numpy(Wr).cuda(), OL.bias, OL.gamma)
    torch.cuda.synchronize()
    _, ids2, _ = O.route_only(wl, x, OL.Wr, OL.bias, OL.gamma)
    assert u in ids2[0] and last not in ids2[0]
    r_top, r_v = list(ids2[1]).index(top), list(ids2[1]).index(v)
    assert abs(r_top - r_v) == 1 and (r_top < r_v) == (top < v)
    _compare_layer(L, OL, x, want_A=False)
    L.close()


def test_norm_layer_in_place():
    wl = W.Workload("tiny_norm", d=512, f=256, E=32, K=4, n_shared=1, T=3, has_norm=True)
    L = synthetic.build_layer(wl, max_tokens=4)
    OL = O.Layer(wl)
    x = W.x_host(wl, 3, 21)
    _compare_layer(L, OL, x, want_A=False)
    xt = torch.from_numpy(x).cuda()
    L.forward(xt, xt)  # y = x + MoE(RMSNorm(x)) written over x
    assert np.array_equal(to_np(xt), OL.forward(x)["y"])
    L.close()


@pytest.fixture(scope="module")
def glm():
    wl = W.WORKLOADS["glm_decode_t1"]
    L = synthetic.build_layer(wl, max_tokens=4)
    OL = O.Layer(wl)
    yield wl, L, OL
    L.close()


def test_glm_decode_t1_all_stages(glm):
    wl, L, OL = glm
    g, o = _compare_layer(L, OL, W.x_host(wl, 1, 0), want_A=True)
    assert int(to_np(g["n_union"])[0]) == 9


def test_glm_decode_t1_more_tokens(glm):
    wl, L, OL = glm
    for tok in (1, 2, 63):
        _compare_layer(L, OL, W.x_host(wl, 1, tok), want_A=False)


def test_glm_verify_t4_union(glm):
    """T = 4 with the shared selection bias: the four biased experts are in every token's
    top-8, so the union reads them once for all four tokens"""
    wl = W.WORKLOADS["glm_verify_t4"]
    L = synthetic.build_layer(wl, max_tokens=4)
    OL = O.Layer(wl)
    g, o = _compare_layer(L, OL, W.x_host(wl, 4, 0), want_A=False)
    nu = int(to_np(g["n_union"])[0])
    offs = to_np(g["offsets"])[:nu + 1]
    sizes = np.diff(offs)
    assert (sizes[:-1] == 4).sum() >= 4  # biased experts shared by all tokens
    assert nu - 1 < 4 * wl.K  # union smaller than the pair count
    # the production kernel instances (the ones the verify benchmark times) on further batches
    for token0 in (4, 64, 400):
        x = W.x_host(wl, 4, token0)
        y = to_np(L.forward(torch.from_numpy(x).cuda()))
        ref = OL.forward(x, want_dump=False)
        assert np.array_equal(y, ref["y"]), token0
        assert normwise_rel(y, ref["y64"]) <= TOL
    assert L.status() == 0
    L.close()
