"""Resident layers filled from the seeded generator (gen/): the float weights are drawn on
the device, packed by the library's own row packer of the layer's width (int4, int8 or int2)
and loaded into the expert store.
Used by the benchmark, the smoke check and the tests; nothing here computes the layer."""
import torch

from gen import workloads

from . import coli


def build_layer(wl, layer=0, max_tokens=None, batch=8, stream=None, hbm_slots=0):
    dev = torch.device("cuda")
    L = coli.MoeLayer.for_workload(wl, max_tokens, hbm_slots)
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
    wb = wl.wbits
    mat = f * d * wb // 8  # bytes of the gate, the up or the down codes
    rec = torch.empty((batch, 3 * mat), dtype=torch.uint8, device=dev)
    sc = torch.empty((batch, 2 * f + d), dtype=torch.float32, device=dev)
    n = E + wl.n_shared
    for first in range(0, n, batch):
        count = min(batch, n - first)
        for j in range(count):
            workloads.expert_float_dev(wl, layer, first + j, gate, up, down)
            coli.quantize_rows(gate, wb, rec[j, :mat].view(f, d * wb // 8), sc[j, :f])
            coli.quantize_rows(up, wb, rec[j, mat: 2 * mat].view(f, d * wb // 8), sc[j, f: 2 * f])
            coli.quantize_rows(down, wb, rec[j, 2 * mat:].view(d, f * wb // 8), sc[j, 2 * f:])
        torch.cuda.synchronize()
        L.load_experts(first, count, rec, sc, stream=stream)
    del gate, up, down, rec, sc
    torch.cuda.synchronize()
    return L


def x_tokens(wl, T, token0=0):
    x = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
    workloads.x_dev(wl, x, token0)
    return x
