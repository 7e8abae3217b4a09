"""GPU parity of the tensor-core (batched) expert path on layer shapes other than the GLM and
tiny ones ("colibrì 架构概述" §5, gate/up/SwiGLU/down; README batch union): lane groups of 1, 2
and 7 blocks per row, an odd number of 4-block bursts (on the down side: the path takes d a
multiple of 256), a layer without a shared expert, and tile edges where a slot's pairs end inside
a 32-pair tile.  Every stage is compared with the CPU oracle (integers bit for bit, fp32 stages in
the canonical order bit for bit), y with the oracle's fp64 evaluation within 1e-4.  All calls go
through the C ABI."""
import pytest
import torch

from gen import workloads as W
from int4_routed_expert_quantize_gb300 import synthetic
from oracle import oracle as O

from .test_gpu_prefill import _full_compare

pytestmark = pytest.mark.gpu

SHAPES = [
    # d=1280: 40 blocks per row, lane groups of 2, 10 bursts; f=640: groups of 1, 5 bursts
    W.Workload("pf_d1280_f640", d=1280, f=640, E=16, K=4, n_shared=1, T=40, bias="zipf"),
    # d=2048, f=1536: groups of 2 on both sides, no shared expert
    W.Workload("pf_d2048_f1536", d=2048, f=1536, E=16, K=2, n_shared=0, T=48),
    # d=7168: 224 blocks per row, lane groups of 7
    W.Workload("pf_d7168_f512", d=7168, f=512, E=8, K=2, n_shared=1, T=24, bias="zipf"),
]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


@pytest.mark.parametrize("wl", SHAPES, ids=[w.name for w in SHAPES])
def test_tensor_core_path_other_shapes(wl):
    L = synthetic.build_layer(wl, max_tokens=wl.T)
    try:
        L.set_prefill_min(2)
        assert L.launches(wl.T) == 8  # the batched tensor-core path
        OL = O.Layer(wl)
        for T, token0 in ((wl.T, 0), (wl.T - 3, 100)):
            _full_compare(L, OL, W.x_host(wl, T, token0), want_A=False)
        assert L.status() == 0
    finally:
        L.close()
