"""The routing entry point that allocates nothing, for callers that cannot call cudaMalloc
(for example a process whose device memory belongs to another allocator's pool).  Checked
through the C ABI against the layer's own routing (the ids and weights
coli_moe_forward_debug reports), bit for bit, on two calls in a row.  Kept in a file pytest
collects last."""
import numpy as np
import pytest
import torch

from gen import workloads as W
from int4_routed_expert_quantize_gb300 import coli, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


@pytest.mark.parametrize("name", ["tiny_t1", "glm_verify_t4"])
def test_route_noalloc_matches_layer_routing_twice(name):
    wl = W.WORKLOADS[name]
    layer = synthetic.build_layer(wl, max_tokens=4)
    Wr = torch.empty((wl.E, wl.d), dtype=torch.float32, device="cuda")
    W.router_dev(wl, 0, Wr)
    b = W.bias_host(wl, 0)
    bias = torch.from_numpy(b).cuda() if b is not None else None
    for call, (T, token0) in enumerate([(4, 0), (3, 77)]):
        x = synthetic.x_tokens(wl, T, token0=token0)
        ref = layer.forward_debug(x)
        ids, w = coli.route_noalloc(x, Wr, wl.K, bias=bias)
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), ref["ids"].cpu().numpy()), call
        assert np.array_equal(w.cpu().numpy(), ref["w"].cpu().numpy()), call
    layer.close()


def test_route_noalloc_ranks_non_finite_scores_like_the_layer():
    """selection biases of NaN and +-inf: both sides rank by the same order-preserving key, so
    the ids and weights still agree bit for bit, on two calls in a row"""
    wl = W.WORKLOADS["tiny_t1"]
    layer = synthetic.build_layer(wl, max_tokens=4)
    Wr = torch.empty((wl.E, wl.d), dtype=torch.float32, device="cuda")
    W.router_dev(wl, 0, Wr)
    b = np.zeros(wl.E, dtype=np.float32)
    b[3], b[5], b[7], b[20] = np.nan, -np.inf, np.inf, -np.nan
    layer.load_router(Wr, b)
    bias = torch.from_numpy(b).cuda()
    for call, (T, token0) in enumerate([(4, 11), (2, 40)]):
        x = synthetic.x_tokens(wl, T, token0=token0)
        ref = layer.forward_debug(x)
        ids, w = coli.route_noalloc(x, Wr, wl.K, bias=bias)
        torch.cuda.synchronize()
        assert np.array_equal(ids.cpu().numpy(), ref["ids"].cpu().numpy()), call
        assert np.array_equal(w.cpu().numpy().view(np.uint32), ref["w"].cpu().numpy().view(np.uint32)), call
    layer.close()


def test_route_noalloc_rejects_sizes_beyond_its_limits():
    x = torch.zeros((5, 512), device="cuda")
    Wr = torch.zeros((1100, 512), device="cuda")
    ids = torch.zeros((5, 40), dtype=torch.int32, device="cuda")
    wo = torch.zeros((5, 40), device="cuda")
    lib = coli.lib()

    def call(T, E, d, K):
        return lib.coli_route_noalloc(x.data_ptr(), T, Wr.data_ptr(), None, E, d, K, 1.0,
                                      ids.data_ptr(), wo.data_ptr(), None)

    assert call(5, 32, 512, 4) == -1      # more tokens than the scratch holds
    assert call(4, 1025, 512, 4) == -1    # more experts than the scratch holds
    assert call(4, 32, 500, 4) == -1      # width not a multiple of 128
    assert call(4, 32, 512, 33) == -1     # K above 32
    assert call(4, 8, 512, 9) == -1       # K above E
    assert call(0, 32, 512, 4) == 0       # nothing to do
    assert call(4, 1024, 512, 8) == 0     # the largest case fits exactly (4 x 1024 scores)
    torch.cuda.synchronize()
