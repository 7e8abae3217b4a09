"""GPU parity of the tensor-core (batched) expert path against the CPU oracle, stage by stage,
and its bit-identity with the decode path for the same tokens."""
import numpy as np
import pytest
import torch

from gen import workloads as W
from int4_routed_expert_quantize_gb300 import synthetic
from oracle import oracle as O

from .gpu_util import normwise_rel, stage_report, to_np

pytestmark = pytest.mark.gpu
TOL = 1e-4
STAGES = ("xn", "qx", "dx", "logits", "scores", "ids", "w", "inv", "pair_token", "pair_rank",
          "g", "u", "h", "qh", "dh", "e")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _full_compare(L, OL, x, want_A):
    g = L.forward_debug(torch.from_numpy(x).cuda(), want_A=want_A)
    torch.cuda.synchronize()
    o = OL.forward(x, want_A=want_A)
    nu = int(to_np(g["n_union"])[0])
    assert nu == o["n_union"][0]
    gd = {k: to_np(g[k]) for k in STAGES}
    gd["union_ids"] = to_np(g["union_ids"])[:nu]
    gd["offsets"] = to_np(g["offsets"])[:nu + 1]
    keys = list(STAGES) + ["union_ids", "offsets"]
    if want_A:
        for k in ("Ag", "Au", "Ad"):
            gd[k] = to_np(g[k])
        keys += ["Ag", "Au", "Ad"]
    bad = stage_report(gd, o, keys)
    y = to_np(g["y"])
    err = normwise_rel(y, o["y64"])
    assert not bad, f"stages differing from the oracle: {bad}; y rel err {err:.3e}"
    assert err <= TOL
    assert np.array_equal(y, o["y"])
    return g, o


@pytest.fixture(scope="module")
def tiny32():
    wl = W.Workload("tiny_batch", d=512, f=256, E=32, K=4, n_shared=1, T=32)
    L = synthetic.build_layer(wl, max_tokens=32)
    L.set_prefill_min(5)  # these tests exercise the tensor-core path at small batches
    yield wl, L, O.Layer(wl)
    L.close()


@pytest.mark.parametrize("T,token0", [(5, 0), (16, 3), (32, 40)])
def test_tiny_tensor_core_path_all_stages(tiny32, T, token0):
    wl, L, OL = tiny32
    _full_compare(L, OL, W.x_host(wl, T, token0), want_A=True)


def test_tiny_tensor_core_matches_decode_path(tiny32):
    wl, L, OL = tiny32
    x = synthetic.x_tokens(wl, 24, token0=500)
    yb = to_np(L.forward(x))
    for t in (0, 7, 23):
        y1 = to_np(L.forward(x[t:t + 1].contiguous()))
        assert np.array_equal(yb[t], y1[0])


@pytest.fixture(scope="module")
def glm64():
    wl = W.Workload("glm_batch", d=6144, f=2048, E=256, K=8, n_shared=1, T=64)
    L = synthetic.build_layer(wl, max_tokens=64)
    L.set_prefill_min(5)  # these tests exercise the tensor-core path at small batches
    yield wl, L, O.Layer(wl)
    L.close()


def test_glm_tensor_core_path_all_stages(glm64):
    wl, L, OL = glm64
    _full_compare(L, OL, W.x_host(wl, 12, 0), want_A=True)


def test_glm_tensor_core_matches_decode_path(glm64):
    wl, L, OL = glm64
    x = synthetic.x_tokens(wl, 64, token0=1000)
    yb = to_np(L.forward(x))
    for t in (0, 31, 63):
        y1 = to_np(L.forward(x[t:t + 1].contiguous()))
        assert np.array_equal(yb[t], y1[0])
    assert L.status() == 0


def test_glm_batch_paths_agree(glm64):
    # the same 64-token batch through the tensor-core path and through chunked decode (the
    # default below the crossover): bit-identical outputs
    wl, L, OL = glm64
    x = synthetic.x_tokens(wl, 64, token0=2000)
    yt = to_np(L.forward(x))
    assert L.launches(64) == 8
    L.set_prefill_min(65)
    try:
        assert L.launches(64) == 3 * 8  # 8 chunks of 8 tokens, one union pass each
        yd = to_np(L.forward(x))
    finally:
        L.set_prefill_min(5)
    assert np.array_equal(yt, yd)
    assert L.status() == 0


@pytest.fixture(scope="module")
def prefill512():
    wl = W.WORKLOADS["glm_prefill_t512"]
    L = synthetic.build_layer(wl, max_tokens=512)
    yield wl, L, O.Layer(wl)
    L.close()


def test_prefill512_routing_union_and_sampled_outputs(prefill512):
    """the 512-token Zipf batch: every token's top-8, weights and the whole batch union match
    the oracle exactly; h codes and outputs of sampled tokens match too"""
    wl, L, OL = prefill512
    x = W.x_host(wl, 512)
    g = L.forward_debug(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    xn, ids, w = O.route_only(wl, x, OL.Wr, OL.bias, OL.gamma)
    assert np.array_equal(to_np(g["ids"]), ids)
    assert np.array_equal(to_np(g["w"]), w)
    ub = O.union_bucket(ids, wl.E, 1)
    nu = int(to_np(g["n_union"])[0])
    assert nu == ub["n_union"]
    assert np.array_equal(to_np(g["union_ids"])[:nu], ub["union_ids"])
    assert np.array_equal(to_np(g["offsets"])[:nu + 1], ub["offsets"])
    assert np.array_equal(to_np(g["pair_token"]), ub["pair_token"])
    assert np.array_equal(to_np(g["inv"]), ub["inv"])
    y = to_np(g["y"])
    qh = to_np(g["qh"])
    inv = ub["inv"]
    for t in (0, 1, 100, 255, 256, 411, 511):
        o = OL.forward(x[t:t + 1])
        assert np.array_equal(y[t], o["y"][0]), t
        assert normwise_rel(y[t], o["y64"][0]) <= TOL
        for k in range(wl.K):  # the pair's h codes, found through the batch union
            assert np.array_equal(qh[inv[t, k]], o["qh"][o["inv"][0, k]])
        assert np.array_equal(qh[wl.K * 512 + t], o["qh"][wl.K])  # shared expert pair
    assert L.status() == 0
