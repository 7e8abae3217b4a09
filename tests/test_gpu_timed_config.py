"""GPU parity in the launch configuration the benchmark times.

The benchmark builds the GLM layer for one token and captures its forward once into a CUDA
graph. Each step it copies a new token into the static input and replays the graph. Here the
same configuration runs on the full GLM layer (d=6144, f=2048, 256 routed experts plus one
shared, top-8).

Each replayed output must equal, bit for bit:
- a direct forward of the same token, and
- the oracle's fp32 output.

It must also lie within the 1e-4 normwise bar of the oracle's fp64 evaluation.
"""
import numpy as np
import pytest
import torch

from gen import workloads as W
from int4_routed_expert_quantize_gb300 import synthetic
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


def test_glm_decode_t1_graph_replay_as_benchmarked():
    wl = W.WORKLOADS["glm_decode_t1"]
    L = synthetic.build_layer(wl, layer=0, max_tokens=wl.T)
    OL = O.Layer(wl)
    assert L.launches(1) == 2  # router + fused expert kernel, as timed
    xs = W.x_host(wl, 6, 100)  # six seeded tokens the other tests do not use
    xin = torch.empty((1, wl.d), dtype=torch.float32, device="cuda")
    y = torch.empty_like(xin)
    ydirect = torch.empty_like(xin)
    xin.copy_(torch.from_numpy(xs[:1]))
    # capture exactly as the benchmark does: a warm-up forward on a side stream, then the graph
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        L.forward(xin, y)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        L.forward(xin, y)
    torch.cuda.synchronize()
    for i in range(xs.shape[0]):
        xin.copy_(torch.from_numpy(xs[i:i + 1]))
        graph.replay()
        torch.cuda.synchronize()
        got = to_np(y).copy()
        L.forward(xin, ydirect)
        torch.cuda.synchronize()
        assert np.array_equal(got, to_np(ydirect)), f"token {i}: replay differs from a direct forward"
        o = OL.forward(xs[i:i + 1], want_dump=False)
        assert np.array_equal(got, o["y"]), f"token {i}: replay differs from the oracle"
        assert normwise_rel(got, o["y64"]) <= TOL
    assert L.status() == 0
    del graph
    L.close()
