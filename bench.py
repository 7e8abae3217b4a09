#!/usr/bin/env python
"""Benchmark of the int4 routed-expert MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl coli|reference]
                    [--configs all|none|name,name,...]

A step is one pass of the whole layer (prep + router/top-K/union + gate/up SwiGLU + down/combine)
over one batch of synthetic tokens that already sit in HBM; the batch changes every step (a pool
of seeded batches), and L2 is flushed between steps by writing a 256 MB buffer outside the timed
events, so expert weights always come from HBM.  Each step is timed with CUDA events on the
stream the kernels run on.  A second, profiled pass records events between the launches and
gives the roofline of the dominant kernel: the fused expert kernel for one token, the gate/up
kernel for 2-4 tokens, the two tensor-core GEMMs for a prefill batch.

The JSON line's top level is the headline workload (--workload, default glm_decode_t1: one
GLM-5.2-shaped layer, one token).  `configs` holds a shorter timed run of each of the other
layer configurations (tiny layer, 4-token verify batch, 16-layer stack, 512-token prefill), each
with its own roofline and clock record, and `spec_verify`: speculative verify forwards of
1 + G tokens (G = 0..7 drafts) with simulated draft acceptance.

With --gpus N under torchrun every rank runs its own replica on its own tokens (weak scaling, no
collective on the data path) and the slowest rank's time is used.

--impl reference times the plain CPU oracle (oracle/) on the host cores instead, on the same
workload and metric; each of its steps runs whole tokens of one batch through the oracle's
layer (as many of the batch's tokens as the time budget allows).
"""
import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
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
FALLBACK_BF16 = 1900.0
# the layer configurations the JSON line's `configs` object times besides the headline
CONFIGS = ["tiny_t1", "glm_decode_t1", "glm_verify_t4", "glm_stack16_t1", "glm_prefill_t512",
           "spec_verify", "glm_i8_decode_t1", "glm_i2_decode_t1", "tiered"]
# steps of a `configs` entry are capped so the whole default run stays within a few minutes
CONFIG_STEP_CAP = {"glm_prefill_t512": 60, "glm_stack16_t1": 300}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default="glm_decode_t1", choices=sorted(W.WORKLOADS))
    p.add_argument("--impl", default="coli", choices=["coli", "reference"])
    p.add_argument("--configs", default="all",
                   help="'all', 'none', or a comma list of workloads to time besides the headline")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample (all cores)")
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
    """gate and up codes + their row scales of the union experts"""
    return n_union_total * (2 * wl.f * wl.d * wl.wbits // 8 + 8 * wl.f)


def down_bytes(wl, n_union_total):
    return n_union_total * (wl.d * wl.f * wl.wbits // 8 + 4 * wl.d)


def expert_ops(wl, T):
    """integer multiply-adds of one forward, counted as 2 ops each: every (token, expert) pair
    and the shared expert's T rows run gate, up and down (3 d f MACs)"""
    pairs = T * wl.K + (T if wl.n_shared else 0)
    return 2 * pairs * 3 * wl.d * wl.f


def peaks():
    """(hbm GB/s, bf16 TFLOP/s burst, bf16 sustained, source)"""
    try:
        with open(PEAKS_FILE) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained",
                                                                            p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM, FALLBACK_BF16, 1700.0, "fallback"


def recorded_traffic(kernel, workload, n_union=None, pairs=None):
    """per-launch DRAM bytes from the committed ncu summary of this kernel, if it is current.
    A record taken on a smaller case of the same kernel and layer shapes carries a linear model
    (bytes per union expert, bytes per token-expert pair) measured there; the figure for this
    workload is that model at its own union size and pair count."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(f"{kernel}:{workload}")
    except Exception:
        return None
    if not rec or source_digest(rec["sources"]) != rec["sources_sha256_16"]:
        return None
    if "bytes_per_launch" in rec:
        return rec["bytes_per_launch"]
    if n_union is None:
        return None
    return rec["bytes_per_union_expert"] * n_union + rec.get("bytes_per_pair", 0.0) * (pairs or 0)


def source_digest(names):
    """digest of the kernel's source files (csrc/), so a recorded traffic figure is used only
    while the code it was measured on is unchanged"""
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "int4_routed_expert_quantize_gb300", "csrc", n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith(("model name", "cpu model")):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


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


def oracle_run(OL, x, seconds, min_batches=2):
    """whole batches of x (cycled) through the oracle's layer until `seconds` have passed;
    -> (batches, tokens, elapsed s)"""
    T = OL.wl.T
    nb = x.shape[0] // T
    t0 = time.perf_counter()
    done = 0
    while True:
        j = done % nb
        OL.forward(x[j * T:(j + 1) * T], want_dump=False, want_y64=False)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds and done >= min_batches:
            return done, done * T, el


def cpu_baseline(wl, seconds):
    """the oracle as it stands, whole layer per token, on a bounded sample of tokens: all host
    cores, then one core"""
    from oracle import oracle as O
    OL = oracle_layer(wl)
    x = W.x_host(wl, 16 * wl.T)
    # generate the experts of the sample outside the timing
    _, ids, _ = O.route_only(wl, x, OL.Wr, OL.bias, OL.gamma)
    OL.ensure(sorted(set(ids.ravel().tolist()) | ({wl.E} if wl.n_shared else set())))
    lib = O.lib()
    cores = lib.orc_num_threads()
    nb, ntok, el = oracle_run(OL, x, seconds)
    lib.orc_set_num_threads(1)
    try:
        nb1, ntok1, el1 = oracle_run(OL, x, seconds / 2, min_batches=1)
    finally:
        lib.orc_set_num_threads(cores)
    return {"value": ntok / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "value_1core": ntok1 / el1,
            "sample": f"{nb} batches of T={wl.T} token(s) of {wl.name} (16 distinct batches, "
                      f"cycled) through the full layer (experts pre-generated), {el:.1f} s on "
                      f"{cores} threads; then {nb1} batches on 1 thread, {el1:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_info()
    if rank != 0:
        return None
    from oracle import oracle as O
    wl = W.WORKLOADS[args.workload]
    layers = wl.layers
    if layers > 1:  # one layer of the stack per token, rate divided by the layer count
        wl = W.WORKLOADS["glm_decode_t1"] if wl.d == 6144 else wl
    OL = oracle_layer(wl)
    nbatch = 8
    x = W.x_host(wl, nbatch * wl.T)
    _, ids, _ = O.route_only(wl, x, OL.Wr, OL.bias, OL.gamma)
    OL.ensure(sorted(set(ids.ravel().tolist()) | ({wl.E} if wl.n_shared else set())))
    # tokens per step: the whole batch if the budget allows, else its first `m` tokens (each
    # token through the full layer); the rate is tokens processed over time
    t0 = time.perf_counter()
    OL.forward(x[:1], want_dump=False, want_y64=False)
    per_token = time.perf_counter() - t0
    m = int(max(1, min(wl.T, args.reference_budget / max(1, args.steps + args.warmup) / max(per_token, 1e-6))))

    def step(i):
        j = i % nbatch
        OL.forward(x[j * wl.T: j * wl.T + m], want_dump=False, want_y64=False)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    value = args.steps * m / el / layers
    cores = O.lib().orc_num_threads()
    sample = (f"{m} of the {wl.T} token(s) of one {wl.name} batch per step, each through the full "
              f"layer (router, union, every selected expert's rows)"
              + (f"; rate divided by {layers} layers per token" if layers > 1 else ""))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "i4xi8->i32,f32", "data": "synthetic",
            "config": {"workload": args.workload, "d": wl.d, "f": wl.f, "E": wl.E, "K": wl.K,
                       "n_shared": wl.n_shared, "T": wl.T, "layers": layers},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ GPU arm ----------------

class Bench:
    """state shared by the timed runs of one process: rank, stream, flush buffer"""

    def __init__(self, args):
        import torch
        self.args = args
        self.world, self.rank, local = dist_info()
        if self.world > 1:
            import torch.distributed as dist
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            torch.cuda.set_device(0)
        self.dev_index = torch.cuda.current_device()
        self.flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.hbm, self.bf16, self.bf16_sus, self.peak_kind = peaks()

    def flush_l2(self, i):
        # write more than L2 holds: no line of the previous step's working set survives
        self.flush.fill_(float(i & 1023))

    def close(self):
        if self.world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


def measure(B, wl, steps, warmup, want_e2e, pool):
    """Timed run of one workload: `steps` forwards (graph replay unless --no-graph), each on a new
    batch, L2 flushed before each; then a profiled pass for the per-kernel times.  -> dict"""
    import torch

    from int4_routed_expert_quantize_gb300 import coli, synthetic
    args, world, rank = B.args, B.world, B.rank
    T = wl.T
    layers = [synthetic.build_layer(wl, layer=l, max_tokens=T) for l in range(wl.layers)]
    stacked = wl.layers > 1
    npool = max(1, min(pool, (1 << 28) // (T * wl.d * 4)))  # at most 256 MB of tokens
    xpool = synthetic.x_tokens(wl, npool * T, token0=rank * npool * T).view(npool, T, wl.d)
    y = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
    xs = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")  # the stack works in place
    xin = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def fwd():
        if stacked:
            coli.stack_forward(layers, xs)
        else:
            layers[0].forward(xin, y)

    graph = None
    if not args.no_graph:
        xin.copy_(xpool[0])
        xs.copy_(xpool[0])
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
        B.flush_l2(i)
        (xs if stacked else xin).copy_(xpool[i % npool])
        evs[0].record(stream)
        if graph is not None:
            graph.replay()
        else:
            fwd()
        evs[1].record(stream)

    for i in range(warmup):
        step(i, [torch.cuda.Event(enable_timing=True) for _ in range(2)])
    torch.cuda.synchronize()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    clocks = ClockSampler(B.dev_index) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        step(warmup + i, events[i])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    clk = clocks.stop() if clocks else None
    for L in layers:
        st = L.status()
        if st != 0:
            raise RuntimeError(f"device status {st}")
    fwd_ms = [ev[0].elapsed_time(ev[1]) for ev in events]
    total_fwd_s = reduce_max(sum(fwd_ms) / 1000.0, world)
    value = world * steps * T / total_fwd_s
    n_launch = sum(L.launches(T) for L in layers)

    # per-kernel durations: a profiled pass (events between the launches, no programmatic
    # overlap), every layer of the stack in turn
    n_prof = min(steps, 400)
    pev = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in layers] for _ in range(n_prof)]
    torch.cuda.synchronize()
    for i in range(n_prof):
        B.flush_l2(i)
        if stacked:
            xs.copy_(xpool[i % npool])
            for L, ev in zip(layers, pev[i]):
                L.forward_profiled(xs, xs, ev)
        else:
            layers[0].forward_profiled(xpool[i % npool], y, pev[i][0])
    torch.cuda.synchronize()

    def mean_ms(a, b):
        return statistics.fmean(sum(e[a].elapsed_time(e[b]) for e in evl) for evl in pev)

    kern = {"route": mean_ms(0, 1), "gateup": mean_ms(1, 2), "down": mean_ms(2, 3), "steps": n_prof}
    # union size of each step (one token: always K + shared); averaged over sampled batches
    if T == 1:
        n_union = wl.K + wl.n_shared
    else:
        sizes = []
        for i in range(min(steps, 64 if T <= 8 else 4)):
            dmp = layers[0].forward_debug(xpool[i % npool])
            sizes.append(int(dmp["n_union"].item()))
            del dmp
        n_union = statistics.fmean(sizes)
    ebytes = expert_bytes(wl, n_union) * wl.layers
    mean_s = total_fwd_s / steps
    expert_gbs = ebytes / mean_s / 1e9
    out = {"value": value, "unit": "tokens/s", "ms_per_step": 1000.0 * mean_s,
           "config": {"workload": wl.name, "d": wl.d, "f": wl.f, "E": wl.E, "K": wl.K,
                      "n_shared": wl.n_shared, "T": T, "layers": wl.layers, "bias": wl.bias,
                      "weight_bits": wl.wbits,
                      "resident_expert_gb": round(wl.layers * (wl.E + wl.n_shared) * wl.expert_bytes / 1e9, 2),
                      "l2": "flushed between steps (256 MB write, outside the timed events)",
                      "tokens": f"pool of {npool} seeded batches, one per step",
                      "launch": "CUDA graph replay" if graph is not None else "direct launches"},
           "steps": steps, "warmup": warmup,
           "expert_bytes_per_step": ebytes, "mean_union_experts": n_union,
           "expert_gbs": expert_gbs, "expert_hbm_frac": expert_gbs / B.hbm,
           "wall_s": wall, "gpu_launches": n_launch * steps + n_launch * n_prof, "kernel_ms": kern}
    hbm_src = f"{B.peak_kind} hbm_gbs (copy, burst)"
    if n_launch == 8 * wl.layers:
        # tensor-core path: the two GEMM launches (gate/up, then down + the combine)
        t_ms = kern["gateup"] + kern["down"]
        ach = expert_bytes(wl, n_union) / (t_ms / 1000.0) / 1e9
        flops = expert_ops(wl, T)
        tf = flops / (t_ms / 1000.0) / 1e12
        out["roofline"] = {"kernel": "expert_gemm_kernel (gate/up, down) + combine_kernel",
                           "bound": "hbm", "achieved": ach, "peak": B.hbm, "peak_source": hbm_src,
                           "unit": "GB/s", "frac": ach / B.hbm,
                           "algorithmic_bytes": expert_bytes(wl, n_union),
                           "traffic": recorded_traffic("expert_gemm_kernel", wl.name, n_union,
                                                       T * (wl.K + wl.n_shared)),
                           "tensor": {"achieved": tf, "peak": B.bf16, "unit": "TFLOP/s",
                                      "frac": tf / B.bf16, "algorithmic_flops": flops,
                                      "peak_source": f"{B.peak_kind} bf16_tflops (burst); the MMAs "
                                                     "run kind::f16 on bf16 copies of the int8/int4 codes"},
                           "timing": "CUDA events around the launches, profiled pass"}
    elif n_launch == 2 * wl.layers:
        # the fused expert kernel reads every union expert's bytes
        t_ms = kern["gateup"] / wl.layers
        gb = expert_bytes(wl, n_union)
        ach = gb / (t_ms / 1000.0) / 1e9
        out["roofline"] = {"kernel": "expert_fused_kernel", "bound": "hbm", "achieved": ach,
                           "peak": B.hbm, "peak_source": hbm_src, "unit": "GB/s",
                           "frac": ach / B.hbm, "algorithmic_bytes": gb,
                           "traffic": recorded_traffic("expert_fused_kernel", wl.name),
                           "timing": "CUDA events around the launch, profiled pass"
                                     + (" (mean over the layers)" if stacked else "")}
        if wl.name == "tiny_t1":
            out["roofline"]["bound"] = "latency"
            out["roofline"]["note"] = "1 MB per step: launch- and latency-bound, %HBM not meaningful"
    else:
        gb = gateup_bytes(wl, n_union)
        t_ms = kern["gateup"] / wl.layers
        ach = gb / (t_ms / 1000.0) / 1e9
        out["roofline"] = {"kernel": "gateup_decode_kernel", "bound": "hbm", "achieved": ach,
                           "peak": B.hbm, "peak_source": hbm_src, "unit": "GB/s",
                           "frac": ach / B.hbm, "algorithmic_bytes": gb,
                           "traffic": recorded_traffic("gateup_decode_kernel", wl.name, n_union),
                           "timing": "CUDA events around the launch, profiled pass"}
        out["down_gbs"] = down_bytes(wl, n_union) / (kern["down"] / 1000.0) / 1e9
    if clk:
        out["clocks"] = clk
    # end to end through the host-buffer entry point (copies inside the timed region)
    if want_e2e:
        xh = xpool[:64].cpu().pin_memory()
        n_e2e = max(300, min(steps, 2000))  # enough calls for a stable host-side figure
        if not stacked:
            yh = torch.empty((T, wl.d), dtype=torch.float32).pin_memory()
            for i in range(min(20, max(3, warmup))):
                layers[0].forward_host(xh[i % len(xh)], yh)
            barrier(world)
            t0 = time.perf_counter()
            for i in range(n_e2e):
                layers[0].forward_host(xh[i % len(xh)], yh)
            el = reduce_max(time.perf_counter() - t0, world)
            note = ("coli_moe_forward_host: x into the handle's mapped pinned staging, one graph "
                    "launch (the GPU reads x from host memory, forward, the GPU writes y back), sync")
        else:
            barrier(world)
            t0 = time.perf_counter()
            for i in range(n_e2e):
                xs.copy_(xh[i % len(xh)], non_blocking=True)
                coli.stack_forward(layers, xs)
                yh = xs.to("cpu")
            el = reduce_max(time.perf_counter() - t0, world)
            note = "pinned H2D x, coli_moe_stack_forward (16 layers), D2H y"
        out["e2e"] = {"value": world * n_e2e * T / el, "unit": "tokens/s",
                      "h2d_bytes_per_step": T * wl.d * 4, "d2h_bytes_per_step": T * wl.d * 4,
                      "steps": n_e2e, "note": note}
    for L in layers:
        L.close()
    del layers, xpool
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# per-draft acceptance of the simulated speculative decode: with 3 drafts it gives 2.5 tokens per
# forward (1 + 0.7 + 0.49 + 0.343), inside the 2.2-2.8 the pages report for the int8 MTP head
SPEC_ACCEPT = 0.7


def emitted_tokens(accepted):
    """tokens one verify forward yields: the verified token plus the drafts accepted before the
    first rejected one.  accepted: bool [steps, G] (draft g accepted in isolation)"""
    import numpy as np
    accepted = np.asarray(accepted, dtype=bool)
    if accepted.shape[1] == 0:
        return np.ones(accepted.shape[0])
    return 1 + np.cumprod(accepted, axis=1).sum(axis=1)


def measure_spec(B, steps, warmup, max_drafts=7, seed=0):
    """Speculative verify on the GLM layer with the overlap bias: for G = 0..max_drafts drafts a
    forward of 1 + G tokens (one union pass), timed like measure(); acceptance is simulated per
    step (each draft accepted with probability SPEC_ACCEPT while all before it were, from a
    seeded generator), so a forward yields 1 + (accepted prefix) tokens.  -> dict"""
    import numpy as np
    import torch

    from int4_routed_expert_quantize_gb300 import synthetic
    wl = W.WORKLOADS["glm_verify_t8"]
    L = synthetic.build_layer(wl, max_tokens=1 + max_drafts)
    stream = torch.cuda.current_stream()
    rng = np.random.default_rng(seed)
    sweep = {}
    for G in range(0, max_drafts + 1):
        T = 1 + G
        npool = 256
        xpool = synthetic.x_tokens(wl, npool * T, token0=B.rank * npool * 8).view(npool, T, wl.d)
        xin = xpool[0].clone()
        y = torch.empty_like(xin)
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
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for i in range(warmup + steps):
            B.flush_l2(i)
            xin.copy_(xpool[i % npool])
            if i >= warmup:
                evs[i - warmup][0].record(stream)
            graph.replay()
            if i >= warmup:
                evs[i - warmup][1].record(stream)
        torch.cuda.synchronize()
        if L.status() != 0:
            raise RuntimeError("device status")
        t_ms = [e[0].elapsed_time(e[1]) for e in evs]
        emitted = emitted_tokens(rng.random((steps, G)) < SPEC_ACCEPT)
        nus = [int(L.forward_debug(xpool[i])["n_union"].item()) for i in range(16)]
        n_union = statistics.fmean(nus)
        mean_s = reduce_max(sum(t_ms) / 1000.0, B.world) / steps
        gbs = expert_bytes(wl, n_union) / mean_s / 1e9
        sweep[f"G{G}"] = {"tokens_per_forward_batch": T, "ms_per_forward": 1000.0 * mean_s,
                          "mean_union_experts": n_union, "expert_gbs": gbs,
                          "expert_hbm_frac": gbs / B.hbm,
                          "mean_emitted_per_forward": float(emitted.mean()),
                          "accepted_tokens_per_s": B.world * float(emitted.sum()) / (mean_s * steps),
                          "verified_tokens_per_s": B.world * T / mean_s, "launches": L.launches(T)}
        del graph, xpool
    L.close()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    best = max(sweep, key=lambda k: sweep[k]["accepted_tokens_per_s"])
    return {"workload": "glm_verify_t8 layer, 1 + G tokens per forward (G = 0..%d drafts)" % max_drafts,
            "acceptance": {"per_draft": SPEC_ACCEPT, "model": "a draft counts only if every draft before "
                           "it was accepted; seeded draws; tokens per forward = 1 + accepted prefix"},
            "steps": steps, "warmup": warmup, "sweep": sweep, "best": best,
            "best_accepted_tokens_per_s": sweep[best]["accepted_tokens_per_s"],
            "l2": "flushed between steps (256 MB write, outside the timed events)"}


def measure_tiered(B, steps, warmup, hbm_slots=64, n_pin=16):
    """The GLM layer with the prefill workload's Zipf selection bias, one token per forward, with
    only hbm_slots of its 256 routed experts in HBM: each forward routes on the GPU, lets the tier
    manager place its union (pinned, LRU, load) and copies the misses from pinned host memory
    over the host link before the expert kernels run.  Timed on the host clock (the call
    synchronises once to read the union).  Also times plain copies of expert records from pinned
    host memory into HBM (the host link's rate).  -> dict"""
    import torch

    from int4_routed_expert_quantize_gb300 import coli, synthetic
    wl = W.Workload("glm_zipf_t1", d=6144, f=2048, E=256, K=8, n_shared=1, T=1, bias="zipf")
    L = synthetic.build_layer(wl, max_tokens=1, hbm_slots=hbm_slots)
    tier = coli.Tier(1, wl.E, n_pin, hbm_slots - n_pin)
    xs = synthetic.x_tokens(wl, warmup + steps, token0=B.rank * (warmup + steps))
    y = torch.empty((1, wl.d), dtype=torch.float32, device="cuda")
    for i in range(warmup):
        L.forward_tiered(tier, 0, xs[i:i + 1], y)
    L.repin_tiered(tier, 0)  # pin the experts the warm-up found hottest
    torch.cuda.synchronize()
    st0, (r0, b0) = tier.stats(), L.tier_copies()
    t0 = time.perf_counter()
    for i in range(warmup, warmup + steps):
        L.forward_tiered(tier, 0, xs[i:i + 1], y)
    torch.cuda.synchronize()
    el = reduce_max(time.perf_counter() - t0, B.world)
    st1, (r1, b1) = tier.stats(), L.tier_copies()
    if L.status() != 0:
        raise RuntimeError("device status")
    # the host link: copies of whole records from pinned host memory into HBM, CUDA events
    nrec = 16
    src = torch.empty(nrec * wl.expert_bytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nrec * wl.expert_bytes, dtype=torch.uint8, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dst.copy_(src, non_blocking=True)
    e0.record()
    for k in range(nrec):
        dst[k * wl.expert_bytes:(k + 1) * wl.expert_bytes].copy_(
            src[k * wl.expert_bytes:(k + 1) * wl.expert_bytes], non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    link_gbs = nrec * wl.expert_bytes / (e0.elapsed_time(e1) / 1000.0) / 1e9
    L.close()
    tier.close()
    del xs, src, dst
    torch.cuda.empty_cache()
    calls = steps
    used = (st1["pin_hits"] - st0["pin_hits"]) + (st1["lru_hits"] - st0["lru_hits"]) + (st1["misses"] - st0["misses"])
    return {"workload": "glm layer (d=6144, f=2048, E=256, K=8), prefill's Zipf(1.1) selection bias, T=1",
            "hbm_slots": hbm_slots, "n_pin": n_pin, "n_lru": hbm_slots - n_pin,
            "resident_fraction": hbm_slots / wl.E, "steps": steps, "warmup": warmup,
            "ms_per_forward_wall": 1000.0 * el / calls,
            "tokens_per_s": B.world * calls / el,
            "miss_rate": (st1["misses"] - st0["misses"]) / max(1, used),
            "records_copied_per_forward": (r1 - r0) / calls,
            "host_link_bytes_per_forward": (b1 - b0) / calls,
            "host_link_gbs_records": link_gbs,
            "host_link_ms_per_forward_est": (b1 - b0) / calls / (link_gbs * 1e9) * 1000.0,
            "timing": "host clock around coli_moe_forward_tiered (one union read-back per call)"}


def run_coli(args):
    B = Bench(args)
    wl = W.WORKLOADS[args.workload]
    head = measure(B, wl, args.steps, args.warmup, not args.no_e2e, args.pool)
    out = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": B.world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": f"i{wl.wbits}xi8->i32,f32", "data": "synthetic"}
    out.update({k: v for k, v in head.items() if k not in ("value", "unit", "ms_per_step", "steps", "warmup")})
    if args.configs != "none":
        names = CONFIGS if args.configs == "all" else [n for n in args.configs.split(",") if n]
        cfgs = {}
        for name in names:
            if name == wl.name:
                continue
            if name == "tiered":
                steps = max(1, min(args.steps, 300))
                cfgs[name] = {f"slots{n}": measure_tiered(B, steps, 100, hbm_slots=n, n_pin=n // 4)
                              for n in (64, 128, 192)}
                continue
            if name == "spec_verify":
                steps = max(1, min(args.steps, 300))
                cfgs[name] = measure_spec(B, steps, max(3, min(args.warmup, 10)))
                out["gpu_launches"] += sum(v["launches"] * (steps + max(3, min(args.warmup, 10)))
                                           for v in cfgs[name]["sweep"].values())
                continue
            cwl = W.WORKLOADS[name]
            steps = max(1, min(args.steps, CONFIG_STEP_CAP.get(name, args.steps)))
            warm = max(3, min(args.warmup, 10))
            cfgs[name] = measure(B, cwl, steps, warm, False, args.pool)
            out["gpu_launches"] += cfgs[name]["gpu_launches"]
        out["configs"] = cfgs
    if B.rank == 0 and B.world == 1 and not args.no_cpu_baseline:
        base = wl if wl.layers == 1 else W.WORKLOADS["glm_decode_t1"]
        out["cpu_baseline"] = cpu_baseline(base, args.cpu_seconds)
        if wl.layers > 1:
            out["cpu_baseline"]["value"] /= wl.layers
            out["cpu_baseline"]["value_1core"] /= wl.layers
            out["cpu_baseline"]["sample"] += f"; divided by {wl.layers} layers per token"
    B.close()
    return out if B.rank == 0 else None


def main(argv=None):
    args = parse_args(argv)
    out = run_reference(args) if args.impl == "reference" else run_coli(args)
    if out is not None:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
