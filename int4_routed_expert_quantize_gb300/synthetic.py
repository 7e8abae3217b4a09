"""Resident layers filled from the seeded generator (gen/): the float weights are drawn on
the device, packed by the library's own int4 packer and loaded into the expert store.
Used by the benchmark, the smoke check and the tests; nothing here computes the layer."""
import torch

from gen import workloads

from . import coli


def build_layer(wl, layer=0, max_tokens=None, batch=8, stream=None):
    dev = torch.device("cuda")
    L = coli.MoeLayer.for_workload(wl, max_tokens)
    d, f, E = wl.d, wl.f, wl.E
    Wr = torch.empty((E, d), dtype=torch.float32, device=dev)
    workloads.router_dev(wl, layer, Wr)
    bias = workloads.bias_host(wl, layer)
    gamma = workloads.gamma_host(wl, layer) if wl.has_norm else None
    torch.cuda.synchronize()
    L.load_router(Wr, bias, gamma, stream=stream)
    del Wr
    gate = torch.empty((f, d), dtype=torch.float32, device=dev)
    up = torch.empty((f, d), dtype=torch.float32, device=dev)
    down = torch.empty((d, f), dtype=torch.float32, device=dev)
    rb = 3 * d * f // 2
    rec = torch.empty((batch, rb), dtype=torch.uint8, device=dev)
    sc = torch.empty((batch, 2 * f + d), dtype=torch.float32, device=dev)
    n = E + wl.n_shared
    for first in range(0, n, batch):
        count = min(batch, n - first)
        for j in range(count):
            workloads.expert_float_dev(wl, layer, first + j, gate, up, down)
            coli.quantize_i4_rows(gate, rec[j, : f * d // 2].view(f, d // 2), sc[j, :f])
            coli.quantize_i4_rows(up, rec[j, f * d // 2: f * d].view(f, d // 2), sc[j, f: 2 * f])
            coli.quantize_i4_rows(down, rec[j, f * d:].view(d, f // 2), sc[j, 2 * f:])
        torch.cuda.synchronize()
        L.load_experts(first, count, rec, sc, stream=stream)
    del gate, up, down, rec, sc
    torch.cuda.synchronize()
    return L


def x_tokens(wl, T, token0=0):
    x = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
    workloads.x_dev(wl, x, token0)
    return x
