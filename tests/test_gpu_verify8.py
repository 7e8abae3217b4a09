"""GPU parity of batches of 5 to 8 tokens, which the decode kernels take in one union pass (each
distinct expert of the batch read once): every stage against the CPU oracle, the production
kernel instances against the oracle's fp32 output, batch invariance, and longer batches in
chunks of 8.  Speculative verify ("colibrì 架构概述" §3.3: the main model checks the drafts of
the MTP head in one batched forward; README "如實呈現推測式解碼": draft and verify compute the
same function) is the use: 1 token + up to 7 drafts.  All calls go through the C ABI."""
import numpy as np
import pytest
import torch

from gen import workloads as W
from int4_routed_expert_quantize_gb300 import synthetic
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


@pytest.fixture(scope="module")
def tiny16():
    wl = W.WORKLOADS["tiny_t1"]
    L = synthetic.build_layer(wl, max_tokens=16)
    yield wl, L, O.Layer(wl)
    L.close()


@pytest.mark.parametrize("T,token0", [(5, 3), (6, 60), (7, 300), (8, 17)])
def test_tiny_five_to_eight_tokens_all_stages(tiny16, T, token0):
    wl, L, OL = tiny16
    assert L.launches(T) == 3  # router, gate/up, down: one union pass
    _compare_layer(L, OL, W.x_host(wl, T, token0), want_A=True)


def test_tiny_ragged_batch_in_chunks_of_eight(tiny16):
    """13 tokens: a chunk of 8 and a ragged chunk of 5, production instances"""
    wl, L, OL = tiny16
    assert L.launches(13) == 6
    x = W.x_host(wl, 13, token0=900)
    y = to_np(L.forward(torch.from_numpy(x).cuda()))
    o = OL.forward(x)
    assert np.array_equal(y, o["y"])
    assert normwise_rel(y, o["y64"]) <= TOL


@pytest.fixture(scope="module")
def glm8():
    wl = W.WORKLOADS["glm_verify_t8"]
    L = synthetic.build_layer(wl, max_tokens=8)
    yield wl, L, O.Layer(wl)
    L.close()


def test_glm_verify_t8_all_stages_one_union(glm8):
    """1 token + 7 drafts with the shared selection bias: every stage bit-exact, and the batch
    reads each distinct expert once (the union of all 8 tokens' picks plus the shared one)"""
    wl, L, OL = glm8
    x = W.x_host(wl, 8, 0)
    g, o = _compare_layer(L, OL, x, want_A=False)
    ids = to_np(g["ids"])
    nu = int(to_np(g["n_union"])[0])
    assert nu == len(set(ids.ravel().tolist())) + 1
    assert nu - 1 < 8 * wl.K
    assert L.launches(8) == 3


@pytest.mark.parametrize("T,token0", [(4, 0), (4, 40), (8, 8), (6, 77)])
def test_glm_verify_production_instances(glm8, T, token0):
    """the production (non-debug) kernels against the oracle's fp32 output"""
    wl, L, OL = glm8
    x = W.x_host(wl, T, token0)
    y = to_np(L.forward(torch.from_numpy(x).cuda()))
    o = OL.forward(x, want_dump=False)
    assert np.array_equal(y, o["y"])
    assert normwise_rel(y, o["y64"]) <= TOL


def test_glm_verify_t8_batch_invariance(glm8):
    """a token's output does not depend on its batch: forward(8)[t] == forward(1, x_t)"""
    wl, L, OL = glm8
    x = synthetic.x_tokens(wl, 8, token0=123)
    yb = to_np(L.forward(x))
    for t in range(8):
        assert np.array_equal(yb[t], to_np(L.forward(x[t:t + 1].contiguous()))[0])
