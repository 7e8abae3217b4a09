"""The host-buffer forward (coli_moe_forward_host) over many consecutive calls: token counts of
1-8 go through the handle's mapped staging and one cached CUDA graph per count, whose last kernel
raises a completion counter that the call waits on; larger counts copy directly.  Calls of
different counts, pageable and pinned buffers, and a call whose fused kernel's barrier wait runs
out (the failure knob, reported as COLI_ETIMEOUT) are interleaved; every other call's y must be
bit-identical to the device forward's and to the oracle's ("colibrì 架构概述" §5, moe step).
All calls go through the C ABI."""
import numpy as np
import pytest
import torch

from gen import workloads as W
from int4_routed_expert_quantize_gb300 import coli, synthetic
from oracle import oracle as O

from .gpu_util import to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def test_host_buffer_calls_in_sequence():
    wl = W.WORKLOADS["tiny_t1"]
    L = synthetic.build_layer(wl, max_tokens=16)
    OL = O.Layer(wl)
    try:
        counts = [1, 2, 1, 8, 3, 12, 1, 1, 5, 16, 2, 1]
        token0 = 0
        for call, T in enumerate(counts):
            x_np = W.x_host(wl, T, token0)
            token0 += T
            pinned = call % 2 == 0
            x = torch.from_numpy(x_np)
            y = torch.empty_like(x)
            if pinned:
                x, y = x.pin_memory(), y.pin_memory()
            if call == 6:
                # one token with the failure knob set: the fused kernel's barrier wait runs out
                L.inject_fault(coli.FAULT_SKIP_ARRIVAL)
                with pytest.raises(coli.ColiError) as ei:
                    L.forward_host(x, y)
                assert ei.value.status == coli.ETIMEOUT
                continue
            L.forward_host(x, y)
            ref = to_np(L.forward(x.cuda()))
            assert np.array_equal(y.numpy(), ref), (call, T)
            assert np.array_equal(y.numpy(), OL.forward(x_np, want_dump=False)["y"]), (call, T)
        assert L.status() == 0
    finally:
        L.close()
