"""The synthetic workloads of the int4 routed-expert MoE layer.

Shapes follow the GLM-5.2-style layer the source pages describe (256 routed experts, top-8
sigmoid routing, one always-on shared expert, int4 experts of about 19 MB) and a tiny layer
for fast checks.  Every tensor is drawn from the counter-based generator with seed 0:
  weights  W ~ N(0, 0.02) (router kept fp32, expert matrices later quantised to int4)
  inputs   x ~ N(0, 1)
  gamma    0.9 + 0.2 * U[0,1)            (RMSNorm gain of the 16-layer stack)
  bias     selection-only router bias: "overlap" puts +1.0 on a seeded set of 4 experts so
           every token of a 4-token verify batch shares them (~50% overlap); "zipf" gives the
           expert of seeded rank i the bias c * i^-1.1 with c = 0.38, which skews 512 prefill
           tokens so the busiest expert gets about 200 of them.
Nothing here computes any part of the layer.
"""
from dataclasses import dataclass

import numpy as np

from . import gen

ZIPF_S = 1.1
ZIPF_C = 0.38
OVERLAP_SET = 4
OVERLAP_BIAS = 1.0


@dataclass(frozen=True)
class Workload:
    name: str
    d: int
    f: int
    E: int
    K: int
    n_shared: int
    T: int
    layers: int = 1
    has_norm: bool = False
    rms_eps: float = 1e-6
    bias: str = "none"
    seed: int = 0
    w_sigma: float = 0.02
    router_sigma: float = 0.02
    x_sigma: float = 1.0
    wbits: int = 4  # bits per expert weight: 4, or 8 / 2 for int8 / int2 experts

    @property
    def expert_bytes(self):
        """packed codes + f32 row scales of one expert (gate, up, down)"""
        return 3 * self.d * self.f * self.wbits // 8 + 4 * (2 * self.f + self.d)

    @property
    def n_slots(self):
        return self.E + self.n_shared


WORKLOADS = {
    "tiny_t1": Workload("tiny_t1", d=512, f=256, E=32, K=4, n_shared=1, T=1),
    "glm_decode_t1": Workload("glm_decode_t1", d=6144, f=2048, E=256, K=8, n_shared=1, T=1),
    "glm_verify_t4": Workload("glm_verify_t4", d=6144, f=2048, E=256, K=8, n_shared=1, T=4,
                              bias="overlap"),
    # speculative verify with 7 drafts: 1 + 7 tokens in one batch, the same overlap bias
    "glm_verify_t8": Workload("glm_verify_t8", d=6144, f=2048, E=256, K=8, n_shared=1, T=8,
                              bias="overlap"),
    "glm_stack16_t1": Workload("glm_stack16_t1", d=6144, f=2048, E=256, K=8, n_shared=1, T=1,
                               layers=16, has_norm=True),
    "glm_prefill_t512": Workload("glm_prefill_t512", d=6144, f=2048, E=256, K=8, n_shared=1,
                                 T=512, bias="zipf"),
    # int8 experts ("colibrì 架构概述" §3.1: int8 rows for the dense part and the MTP head) and
    # int2 experts (int2 packed, experimental) on the same layers
    "tiny_i8_t1": Workload("tiny_i8_t1", d=512, f=256, E=32, K=4, n_shared=1, T=1, wbits=8),
    "tiny_i2_t1": Workload("tiny_i2_t1", d=512, f=256, E=32, K=4, n_shared=1, T=1, wbits=2),
    "glm_i8_decode_t1": Workload("glm_i8_decode_t1", d=6144, f=2048, E=256, K=8, n_shared=1, T=1,
                                 wbits=8),
    "glm_i2_decode_t1": Workload("glm_i2_decode_t1", d=6144, f=2048, E=256, K=8, n_shared=1, T=1,
                                 wbits=2),
    # the GLM layer's shapes with 32 routed experts: the same kernels and per-step bytes
    # (9 experts, 170 MB, more than L2) with 0.6 GB resident, for counter captures
    "glm_e32_decode_t1": Workload("glm_e32_decode_t1", d=6144, f=2048, E=32, K=8, n_shared=1, T=1),
    "glm_e32_stack2_t1": Workload("glm_e32_stack2_t1", d=6144, f=2048, E=32, K=8, n_shared=1, T=1,
                                  layers=2, has_norm=True),
    "glm_e32_i8_decode_t1": Workload("glm_e32_i8_decode_t1", d=6144, f=2048, E=32, K=8, n_shared=1,
                                     T=1, wbits=8),
    "glm_e32_i2_decode_t1": Workload("glm_e32_i2_decode_t1", d=6144, f=2048, E=32, K=8, n_shared=1,
                                     T=1, wbits=2),
    "glm_e32_verify_t4": Workload("glm_e32_verify_t4", d=6144, f=2048, E=32, K=8, n_shared=1, T=4,
                                  bias="overlap"),
    # 256 tokens (the batched tensor-core path), zipf selection: ~33 union experts, 0.4 GB of
    # weights per forward
    "glm_e32_prefill_t256": Workload("glm_e32_prefill_t256", d=6144, f=2048, E=32, K=8, n_shared=1,
                                     T=256, bias="zipf"),
}


def expert_float_host(wl, layer, expert):
    """float32 gate [f,d], up [f,d], down [d,f] of expert `expert` (E = the shared expert)"""
    g = gen.normal_host((wl.f, wl.d), wl.seed, layer, gen.T_GATE, expert, sigma=wl.w_sigma)
    u = gen.normal_host((wl.f, wl.d), wl.seed, layer, gen.T_UP, expert, sigma=wl.w_sigma)
    dn = gen.normal_host((wl.d, wl.f), wl.seed, layer, gen.T_DOWN, expert, sigma=wl.w_sigma)
    return g, u, dn


def router_host(wl, layer):
    return gen.normal_host((wl.E, wl.d), wl.seed, layer, gen.T_ROUTER, 0, sigma=wl.router_sigma)


def gamma_host(wl, layer):
    return gen.uniform_affine_host((wl.d,), wl.seed, layer, gen.T_GAMMA, 0, 0.9, 0.2)


def x_host(wl, T, token0=0):
    """tokens token0 .. token0+T-1 of the input pool, [T, d]"""
    return gen.normal_host((T, wl.d), wl.seed, 0, gen.T_X, 0, idx0=token0 * wl.d, sigma=wl.x_sigma)


def bias_host(wl, layer):
    """float32 [E] selection bias, or None"""
    if wl.bias == "none":
        return None
    if wl.bias == "overlap":
        b = np.zeros(wl.E, dtype=np.float32)
        draws = gen.draws_host(64, wl.seed, layer, gen.T_PICK, 0)
        picked = []
        for z in draws:
            e = int(z % np.uint64(wl.E))
            if e not in picked:
                picked.append(e)
            if len(picked) == OVERLAP_SET:
                break
        b[picked] = OVERLAP_BIAS
        return b
    if wl.bias == "zipf":
        perm = np.arange(wl.E)
        draws = gen.draws_host(wl.E, wl.seed, layer, gen.T_PERM, 0)
        for i in range(wl.E - 1, 0, -1):  # Fisher-Yates
            j = int(draws[i] % np.uint64(i + 1))
            perm[i], perm[j] = perm[j], perm[i]
        b = np.zeros(wl.E, dtype=np.float32)
        b[perm] = (ZIPF_C * np.arange(1, wl.E + 1, dtype=np.float64) ** -ZIPF_S).astype(np.float32)
        return b
    raise ValueError(wl.bias)


# ---------------- device-side fills (torch CUDA tensors) ----------------

def expert_float_dev(wl, layer, expert, gate, up, down, stream=0):
    gen.normal_dev(gate, wl.seed, layer, gen.T_GATE, expert, sigma=wl.w_sigma, stream=stream)
    gen.normal_dev(up, wl.seed, layer, gen.T_UP, expert, sigma=wl.w_sigma, stream=stream)
    gen.normal_dev(down, wl.seed, layer, gen.T_DOWN, expert, sigma=wl.w_sigma, stream=stream)


def router_dev(wl, layer, out, stream=0):
    return gen.normal_dev(out, wl.seed, layer, gen.T_ROUTER, 0, sigma=wl.router_sigma, stream=stream)


def x_dev(wl, out, token0=0, stream=0):
    return gen.normal_dev(out, wl.seed, 0, gen.T_X, 0, idx0=token0 * wl.d, sigma=wl.x_sigma,
                          stream=stream)
