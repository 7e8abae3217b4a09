"""GPU parity of the multi-layer stack (RMSNorm + residual between GLM-shaped layers) and of
the 512-token prefill batch with Zipf-skewed routing, against the CPU oracle."""
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


def _stack(n_layers, token0):
    wl = W.WORKLOADS["glm_stack16_t1"]
    layers = [synthetic.build_layer(wl, layer=l, max_tokens=1) for l in range(n_layers)]
    x0 = W.x_host(wl, 1, token0)
    xd = torch.from_numpy(x0).cuda()
    coli.stack_forward(layers, xd)
    torch.cuda.synchronize()
    got = to_np(xd)
    for L in layers:
        assert L.status() == 0
        L.close()
    del layers
    torch.cuda.empty_cache()
    x = x0
    for l in range(n_layers):
        x = O.Layer(wl, l).forward(x, want_dump=False, want_y64=False)["y"]
    return got, x


def test_stack_four_layers():
    got, ref = _stack(4, token0=0)
    assert np.array_equal(got, ref)
    assert normwise_rel(got, ref) <= TOL


@pytest.mark.slow
def test_stack_sixteen_layers_full():
    """the whole 16-layer, 77.8 GB resident stack, one token through every layer"""
    got, ref = _stack(16, token0=1)
    assert np.array_equal(got, ref)
    assert normwise_rel(got, ref) <= TOL


@pytest.fixture(scope="module")
def prefill():
    wl = W.WORKLOADS["glm_prefill_t512"]
    L = synthetic.build_layer(wl, max_tokens=512)
    OL = O.Layer(wl)
    yield wl, L, OL
    L.close()


def test_prefill_zipf_histogram(prefill):
    wl, L, OL = prefill
    x = W.x_host(wl, 512)
    _, ids, _ = O.route_only(wl, x, OL.Wr, OL.bias, OL.gamma)
    cnt = np.bincount(ids.ravel(), minlength=wl.E)
    assert 150 <= cnt.max() <= 260 and cnt.min() >= 0 and cnt.sum() == 512 * wl.K


def test_prefill_sampled_tokens(prefill):
    """the full 512-token batch on the GPU; 12 tokens spread over it recomputed by the oracle
    (each token's output depends on that token only)"""
    wl, L, OL = prefill
    x = W.x_host(wl, 512)
    y = to_np(L.forward(torch.from_numpy(x).cuda()))
    torch.cuda.synchronize()
    for t in (0, 1, 63, 64, 127, 200, 255, 256, 300, 401, 510, 511):
        o = OL.forward(x[t:t + 1], want_dump=False)
        assert np.array_equal(y[t], o["y"][0]), t
        assert normwise_rel(y[t], o["y64"][0]) <= TOL
    assert L.status() == 0
