"""GPU tests of the device side of the expert residency tiers ("colibrì 架构概述" §4, the expert
cache and scheduling layer; §5, pin -> LRU -> load; README "統一記憶體階層"): a tiered layer
keeps every record in pinned host memory and only some of them in HBM slots, and where an
expert sits must change the speed only.  A Zipf-routed token stream runs through a layer with
fewer slots than experts, with lookahead prefetch and repinning mixed in; every output must be
bit-identical to the all-resident layer's and to the oracle's.  All calls go through the C ABI."""
import numpy as np
import pytest
import torch

from gen import workloads as W
from int4_routed_expert_quantize_gb300 import coli, synthetic
from oracle import oracle as O

from .gpu_util import normwise_rel, to_np
from .test_gpu_parity import TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


TINY_ZIPF = W.Workload("tiny_zipf", d=512, f=256, E=32, K=4, n_shared=1, T=2, bias="zipf")


def test_tiered_stream_is_bit_identical_to_resident():
    wl = TINY_ZIPF
    Lr = synthetic.build_layer(wl, max_tokens=8)
    Lt = synthetic.build_layer(wl, max_tokens=8, hbm_slots=12)
    tier = coli.Tier(1, wl.E, 4, 8)
    OL = O.Layer(wl)
    xs = W.x_host(wl, 200, token0=1000)
    pos = 0
    for call in range(60):
        T = (1, 2, 1, 3)[call % 4]
        x = xs[pos:pos + T]
        pos += T
        xt = torch.from_numpy(x).cuda()
        yt = to_np(Lt.forward_tiered(tier, 0, xt))
        yr = to_np(Lr.forward(xt))
        assert np.array_equal(yt, yr), call
        if call % 10 == 0:
            assert np.array_equal(yt, OL.forward(x, want_dump=False)["y"]), call
        if call % 7 == 3:
            # lookahead: the oracle's routing of the next call's tokens, as a router would predict
            _, ids, _ = O.route_only(wl, xs[pos:pos + 2], OL.Wr, OL.bias, OL.gamma)
            Lt.prefetch_tiered(tier, 0, sorted(set(ids.ravel().tolist()))[:8])
        if call == 30:
            Lt.repin_tiered(tier, 0)  # live repin by session heat
            tier.decay()
    torch.cuda.synchronize()
    st = tier.stats()
    assert st["misses"] > 0 and st["evictions"] > 0 and st["lru_hits"] > 0 and st["pin_hits"] > 0
    assert st["prefetch_fetches"] > 0
    recs, nbytes = Lt.tier_copies()
    assert recs >= st["misses"] and nbytes == recs * wl.expert_bytes
    assert Lt.status() == 0
    Lt.close()
    Lr.close()
    tier.close()


def test_tiered_glm_layer_against_oracle():
    """the GLM-shaped layer with 40 slots (8 pinned, 32 LRU): one-token forwards (the fused
    kernel) and an 8-token batch (two chunks of 4, the most a 32-slot LRU can take at K = 8)"""
    wl = W.WORKLOADS["glm_verify_t8"]
    Lt = synthetic.build_layer(wl, max_tokens=8, hbm_slots=40)
    tier = coli.Tier(1, wl.E, 8, 32)
    OL = O.Layer(wl)
    for T, token0 in ((1, 0), (1, 1), (8, 2), (1, 2), (4, 30)):
        x = W.x_host(wl, T, token0)
        y = to_np(Lt.forward_tiered(tier, 0, torch.from_numpy(x).cuda()))
        o = OL.forward(x, want_dump=False)
        assert np.array_equal(y, o["y"]), (T, token0)
        assert normwise_rel(y, o["y64"]) <= TOL
    Lt.repin_tiered(tier, 0, by_usage=True)  # start-up pinning by usage heat, then more tokens
    for token0 in (40, 41):
        x = W.x_host(wl, 1, token0)
        y = to_np(Lt.forward_tiered(tier, 0, torch.from_numpy(x).cuda()))
        assert np.array_equal(y, OL.forward(x, want_dump=False)["y"])
    assert Lt.status() == 0
    Lt.close()
    tier.close()


def test_tiered_layer_rules():
    """a tier of another shape is refused; a plain forward before any placement reads no
    outside memory and reports COLI_ESTATE through the status word"""
    wl = TINY_ZIPF
    Lt = synthetic.build_layer(wl, max_tokens=4, hbm_slots=12)
    x = synthetic.x_tokens(wl, 1)
    for bad in (coli.Tier(1, wl.E, 4, 9), coli.Tier(1, wl.E + 1, 4, 8), coli.Tier(1, wl.E, 4, 8)):
        layer = 1 if bad.n_lru == 8 and bad.n_experts == wl.E else 0  # the last one: a bad layer index
        with pytest.raises(coli.ColiError) as ei:
            Lt.forward_tiered(bad, layer, x)
        assert ei.value.status == -1
        bad.close()
    Lt.forward(x)
    assert Lt.status() == -3
    assert Lt.status() == 0
    Lt.close()
