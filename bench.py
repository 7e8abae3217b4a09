#!/usr/bin/env python
"""Benchmark of the int4 routed-expert MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl coli|reference]

A step is one pass of the whole layer (prep + router/top-K/union + gate/up SwiGLU + down/combine)
over one batch of synthetic tokens that already sit in HBM; the token changes every step (a pool
of 4096 seeded tokens), and L2 is flushed between steps by writing a 256 MB buffer, so expert
weights always come from HBM.  Each step is timed with CUDA events on the stream the kernels run
on; the per-kernel events give the roofline of the dominant kernel (gate/up).  With --gpus N under
torchrun every rank runs its own replica on its own tokens (weak scaling, no collective on the
data path) and the slowest rank's time is used.  Prints one JSON line.

--impl reference times the plain CPU oracle (oracle/) on the host cores instead, on the same
workload and metric; each of its steps is one token with the expert rows sampled so the whole
run stays within a few minutes.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gen import workloads as W  # noqa: E402

METRIC = "MoE-layer tokens/s and int4 expert-weight GB/s as % of GB300 HBM peak"
POOL = 4096
FLUSH_BYTES = 256 << 20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM = 6800.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--workload", default="glm_decode_t1", choices=sorted(W.WORKLOADS))
    p.add_argument("--impl", default="coli", choices=["coli", "reference"])
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--pool", type=int, default=POOL, help="distinct token batches cycled")
    p.add_argument("--no-graph", action="store_true",
                   help="launch each step's kernels from Python instead of replaying a CUDA graph")
    p.add_argument("--reference-budget", type=float, default=150.0,
                   help="seconds the reference arm may spend on its timed steps")
    return p.parse_args(argv)


# ------------------------------------------------------------------ bytes and peaks --------

def expert_bytes(wl, n_union_total):
    """nibbles + f32 row scales read per forward (union experts incl. the shared one)"""
    return n_union_total * wl.expert_bytes


def gateup_bytes(wl, n_union_total):
    return n_union_total * (wl.f * wl.d + 8 * wl.f)


def hbm_peak():
    try:
        with open(PEAKS_FILE) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM, "fallback"


def recorded_traffic(kernel, workload):
    """per-launch DRAM bytes from the committed ncu summary of this kernel, if it is current"""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(f"{kernel}:{workload}")
    except Exception:
        return None
    if not rec:
        return None
    return rec["bytes_per_launch"] if source_digest(rec["sources"]) == rec["sources_sha256_16"] else None


def source_digest(names):
    """digest of the kernel's source files (csrc/), so a recorded traffic figure is used only
    while the code it was measured on is unchanged"""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "int4_routed_expert_quantize_gb300", "csrc", n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ distributed ------------

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value, world):
    """slowest rank's value (host-side timing collective only)"""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks -----------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for ln in fh:
                parts = [p.strip() for p in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle -------------

def oracle_layer(wl, layer=0):
    from oracle import oracle as O
    return O.Layer(wl, layer)


def oracle_sample_step(OL, x_tok, phi):
    """One token through the oracle with a fraction phi of every expert's rows: full router,
    top-K and union; gate/up on the first phi*f rows (the rest of h is zero), h re-quantised,
    down on the first phi*d rows; combine in rank order.  phi = 1 is the whole layer."""
    import numpy as np

    from oracle import oracle as O
    wl = OL.wl
    if phi >= 1.0:
        return OL.forward(x_tok, want_dump=False, want_y64=False)["y"]
    d, f = wl.d, wl.f
    xn, ids, w = O.route_only(wl, x_tok, OL.Wr, OL.bias, OL.gamma)
    fr = max(32, int(round(phi * f / 32)) * 32)
    dr = max(1, int(round(phi * d)))
    y = np.zeros((x_tok.shape[0], dr), dtype=np.float32)
    for t in range(x_tok.shape[0]):
        qx, dx = O.quantize_q8(xn[t])
        experts = ([(wl.E, 1.0)] if wl.n_shared else []) + list(zip(ids[t], w[t]))
        for k, (ex, wk) in enumerate(experts):
            rec, sc = OL.recs[int(ex)]
            Wg = rec[: f * d // 2].reshape(f, d // 2)
            Wu = rec[f * d // 2: f * d].reshape(f, d // 2)
            Wd = rec[f * d:].reshape(d, f // 2)
            g, _ = O.i4_matvec(np.ascontiguousarray(Wg[:fr]), np.ascontiguousarray(sc[:fr]), d, qx, dx)
            u, _ = O.i4_matvec(np.ascontiguousarray(Wu[:fr]), np.ascontiguousarray(sc[f:f + fr]), d, qx, dx)
            h = np.zeros(f, dtype=np.float32)
            h[:fr] = [O.lib().orc_silu_mul(float(a), float(b)) for a, b in zip(g, u)]
            qh, dh = O.quantize_q8(h)
            e, _ = O.i4_matvec(np.ascontiguousarray(Wd[:dr]), np.ascontiguousarray(sc[2 * f:2 * f + dr]),
                               f, qh, dh)
            y[t] = e if k == 0 else (np.float32(wk) * e + y[t])
    return y


def cpu_baseline(wl, seconds):
    """the oracle as it stands, whole layer per token, on a bounded sample of tokens"""
    from oracle import oracle as O
    OL = oracle_layer(wl)
    ntok = 2
    x = W.x_host(wl, 64 * wl.T)
    # generate the experts of the candidate sample outside the timing
    _, ids, _ = O.route_only(wl, x[: 16 * wl.T], OL.Wr, OL.bias, OL.gamma)
    OL.ensure(sorted(set(ids.ravel().tolist()) | ({wl.E} if wl.n_shared else set())))
    # the 16 batches' experts are generated once; the timed loop cycles over those batches until
    # the time budget is spent (each token streams all its experts' bytes, far more than the
    # host's caches hold, so repeating a batch does not make it cheaper)
    t0 = time.perf_counter()
    done = 0
    while True:
        j = done % 16
        OL.forward(x[j * wl.T:(j + 1) * wl.T], want_dump=False, want_y64=False)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds and done >= ntok:
            break
    return {"value": done * wl.T / el, "unit": "tokens/s", "cores": O.lib().orc_num_threads(),
            "kind": "oracle",
            "sample": f"{done} batches of T={wl.T} token(s) of {wl.name} (16 distinct batches, "
                      f"cycled) through the full layer (experts pre-generated), {el:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return None
    from oracle import oracle as O
    wl = W.WORKLOADS[args.workload]
    if wl.layers > 1:
        wl = W.WORKLOADS["glm_decode_t1"] if wl.d == 6144 else wl
    OL = oracle_layer(wl)
    x = W.x_host(wl, 64 * wl.T)
    _, ids, _ = O.route_only(wl, x, OL.Wr, OL.bias, OL.gamma)
    OL.ensure(sorted(set(ids.ravel().tolist()) | ({wl.E} if wl.n_shared else set())))
    # size the per-step sample: a full token if it fits the budget, else a row fraction
    t0 = time.perf_counter()
    oracle_sample_step(OL, x[: wl.T], 1.0)
    full = time.perf_counter() - t0
    phi = min(1.0, args.reference_budget / max(1, args.steps + args.warmup) / max(full, 1e-6))
    phi = max(phi, 1.0 / 64)
    for i in range(args.warmup):
        j = i % 64
        oracle_sample_step(OL, x[j * wl.T:(j + 1) * wl.T], phi)
    t0 = time.perf_counter()
    for i in range(args.steps):
        j = i % 64
        oracle_sample_step(OL, x[j * wl.T:(j + 1) * wl.T], phi)
    el = time.perf_counter() - t0
    value = args.steps * wl.T * phi / el
    cores = O.lib().orc_num_threads()
    sample = (f"one batch of T={wl.T} of {wl.name} per step with {phi:.4f} of every expert's rows "
              f"(full router and union); tokens/s scaled by that fraction")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "i4xi8->i32,f32", "data": "synthetic",
            "config": {"workload": wl.name, "d": wl.d, "f": wl.f, "E": wl.E, "K": wl.K,
                       "n_shared": wl.n_shared, "T": wl.T, "layers": 1},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ GPU arm ----------------

def run_coli(args):
    import torch

    from int4_routed_expert_quantize_gb300 import coli, synthetic
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev_index = torch.cuda.current_device()
    wl = W.WORKLOADS[args.workload]
    T = wl.T
    layers = [synthetic.build_layer(wl, layer=l, max_tokens=T) for l in range(wl.layers)]
    stacked = wl.layers > 1
    npool = max(1, args.pool)
    pool = synthetic.x_tokens(wl, npool * T, token0=rank * npool * T).view(npool, T, wl.d)
    y = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
    xs = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")  # stack works in place
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush_l2(i):
        # write more than L2 holds: no line of the previous step's working set survives
        flush.fill_(float(i & 1023))
    stream = torch.cuda.current_stream()

    # one step's forward, optionally captured once into a CUDA graph (input copied into a static
    # buffer before the timed events, so the graph replays the same pointers every step)
    xin = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")

    def fwd():
        if stacked:
            coli.stack_forward(layers, xs)
        else:
            layers[0].forward(xin, y)

    graph = None
    if not args.no_graph:
        xin.copy_(pool[0])
        xs.copy_(pool[0])
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fwd()  # warm-up outside capture
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fwd()
        torch.cuda.synchronize()

    def step(i, evs):
        flush_l2(i)
        if stacked:
            xs.copy_(pool[i % npool])
        else:
            xin.copy_(pool[i % npool])
        evs[0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            fwd()
        evs[1].record(stream)

    for i in range(args.warmup):
        step(i, [torch.cuda.Event(enable_timing=True) for _ in range(2)])
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(dev_index) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("bench_timed")
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i, events[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    torch.cuda.nvtx.range_pop()
    barrier(world)
    clk = clocks.stop() if clocks else None
    for L in layers:
        st = L.status()
        if st != 0:
            raise RuntimeError(f"device status {st}")
    fwd_ms = [ev[0].elapsed_time(ev[1]) for ev in events]
    mean_fwd_ms = statistics.fmean(fwd_ms)
    total_fwd_s = reduce_max(sum(fwd_ms) / 1000.0, world)
    tokens = world * args.steps * T
    value = tokens / total_fwd_s
    # per-kernel durations: a second timed pass through the profiled entry point (events
    # between the three launches; no programmatic overlap there)
    kern = None
    if not stacked and T <= 4:
        n_prof = min(args.steps, 4000)
        pev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_prof)]
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("bench_profiled")
        for i in range(n_prof):
            flush_l2(i)
            layers[0].forward_profiled(pool[i % npool], y, pev[i])
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        kern = {"route": statistics.fmean(e[0].elapsed_time(e[1]) for e in pev),
                "gateup": statistics.fmean(e[1].elapsed_time(e[2]) for e in pev),
                "down": statistics.fmean(e[2].elapsed_time(e[3]) for e in pev),
                "steps": n_prof}
    n_launch = layers[0].launches(T)  # kernels one forward of one layer launches
    # union size of each step (T=1: always K+1); averaged over the pool for T>1
    if T == 1:
        n_union = wl.K + wl.n_shared
    else:
        sizes = []
        for i in range(min(args.steps, 256)):
            dmp = layers[0].forward_debug(pool[i % npool])
            sizes.append(int(dmp["n_union"].item()))
        n_union = statistics.fmean(sizes)
    ebytes = expert_bytes(wl, n_union) * wl.layers
    peak, peak_kind = hbm_peak()
    mean_s = total_fwd_s / (args.steps)
    expert_gbs = ebytes / mean_s / 1e9
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_fwd_ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "i4xi8->i32,f32", "data": "synthetic",
           "config": {"workload": wl.name, "d": wl.d, "f": wl.f, "E": wl.E, "K": wl.K,
                      "n_shared": wl.n_shared, "T": T, "layers": wl.layers,
                      "resident_expert_gb": round(wl.layers * (wl.E + wl.n_shared) * wl.expert_bytes / 1e9, 2),
                      "l2": "flushed between steps (256 MB write, outside the timed events)",
                      "tokens": f"pool of {npool} seeded batches, one per step",
                      "launch": "CUDA graph replay" if graph is not None else "direct launches"},
           "expert_bytes_per_step": ebytes, "mean_union_experts": n_union,
           "expert_gbs": expert_gbs, "expert_hbm_frac": expert_gbs / peak,
           "wall_s": wall, "gpu_launches": n_launch * wl.layers * args.steps}
    if kern:
        # the dominant kernel: the fused expert kernel when the forward runs as two launches
        # (all union expert bytes), else the gate/up kernel (its two thirds of them)
        if n_launch == 2:
            name, gb, t_ms = "expert_fused_kernel", expert_bytes(wl, n_union), kern["gateup"]
            kern = {"route": kern["route"], "experts": kern["gateup"], "steps": kern["steps"]}
        else:
            name, gb, t_ms = "gateup_decode_kernel", gateup_bytes(wl, n_union), kern["gateup"]
            db = n_union * (wl.d * wl.f // 2 + 4 * wl.d)
            out["down_gbs"] = db / (kern["down"] / 1000.0) / 1e9
        ach = gb / (t_ms / 1000.0) / 1e9
        out["roofline"] = {"kernel": name, "bound": "hbm", "achieved": ach,
                           "peak": peak, "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                           "unit": "GB/s", "frac": ach / peak, "algorithmic_bytes": gb,
                           "traffic": recorded_traffic(name, wl.name),
                           "timing": "CUDA events around the launch, profiled pass"}
        out["kernel_ms"] = kern
        out["gpu_launches"] += n_launch * kern["steps"]
    if clk:
        out["clocks"] = clk
    # end to end through the host-buffer entry point (pinned buffers, copies in the region)
    if not args.no_e2e and not stacked:
        xh = pool[:64].cpu().pin_memory()
        yh = torch.empty((T, wl.d), dtype=torch.float32).pin_memory()
        n_e2e = min(args.steps, 2000)
        for i in range(min(20, max(3, args.warmup))):
            layers[0].forward_host(xh[i % len(xh)], yh)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(n_e2e):
            layers[0].forward_host(xh[i % len(xh)], yh)
        el = reduce_max(time.perf_counter() - t0, world)
        out["e2e"] = {"value": world * n_e2e * T / el, "unit": "tokens/s",
                      "h2d_bytes_per_step": T * wl.d * 4, "d2h_bytes_per_step": T * wl.d * 4,
                      "steps": n_e2e, "note": "coli_moe_forward_host: H2D x, forward, D2H y, sync"}
    elif not args.no_e2e and stacked:
        xh = pool[:64].cpu().pin_memory()
        n_e2e = min(args.steps, 500)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(n_e2e):
            xs.copy_(xh[i % len(xh)], non_blocking=True)
            coli.stack_forward(layers, xs)
            yh = xs.to("cpu")
        el = reduce_max(time.perf_counter() - t0, world)
        out["e2e"] = {"value": world * n_e2e * T / el, "unit": "tokens/s",
                      "h2d_bytes_per_step": T * wl.d * 4, "d2h_bytes_per_step": T * wl.d * 4,
                      "steps": n_e2e}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl if not stacked else W.WORKLOADS["glm_decode_t1"],
                                           args.cpu_seconds)
        if stacked:
            out["cpu_baseline"]["value"] /= wl.layers
            out["cpu_baseline"]["sample"] += f"; divided by {wl.layers} layers per token"
    for L in layers:
        L.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return out if rank == 0 else None


def main(argv=None):
    args = parse_args(argv)
    out = run_reference(args) if args.impl == "reference" else run_coli(args)
    if out is not None:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
