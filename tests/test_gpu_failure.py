"""Failure path of the fused one-token expert kernel, the one kernel whose CTAs wait on each
other (its grid barrier between the gate/up and down phases).  A host-set knob leaves CTA 0's
arrival out, so every CTA's bounded wait at the barrier runs out (after about 2 s) and the
kernel finishes without its result: the handle's status word must say COLI_ETIMEOUT, and the
next forward on the same handle must be correct again.  No GPU fault and no hang is involved:
the waits give up by themselves and every CTA leaves the kernel normally."""
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


def test_fused_barrier_timeout_is_reported_and_the_handle_recovers():
    wl = W.WORKLOADS["tiny_t1"]
    layer = synthetic.build_layer(wl, max_tokens=4)
    try:
        assert layer.launches(1) == 2  # one token runs the fused expert kernel
        x = synthetic.x_tokens(wl, 1, token0=11)
        y_ok = torch.empty_like(x)
        layer.forward(x, y_ok)
        torch.cuda.synchronize()
        assert layer.status() == 0

        layer.inject_fault(coli.FAULT_SKIP_ARRIVAL)
        y_bad = torch.empty_like(x)
        layer.forward(x, y_bad)
        torch.cuda.synchronize()
        assert layer.status() == coli.ETIMEOUT
        assert layer.status() == 0  # reading the status cleared it

        y_again = torch.empty_like(x)
        layer.forward(x, y_again)
        torch.cuda.synchronize()
        assert layer.status() == 0
        assert torch.equal(y_again, y_ok)
    finally:
        layer.close()


def test_fault_knob_rejects_unknown_codes_and_clears():
    wl = W.WORKLOADS["tiny_t1"]
    layer = synthetic.build_layer(wl, max_tokens=4)
    try:
        with pytest.raises(coli.ColiError):
            layer.inject_fault(7)
        layer.inject_fault(coli.FAULT_SKIP_ARRIVAL)
        layer.inject_fault(0)  # cleared again: the next forward is normal
        x = synthetic.x_tokens(wl, 1, token0=12)
        y = torch.empty_like(x)
        layer.forward(x, y)
        torch.cuda.synchronize()
        assert layer.status() == 0
    finally:
        layer.close()
