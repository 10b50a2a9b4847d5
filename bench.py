"""Benchmark of the latent-MoE layer hot path on B300 (one JSON line on rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole layer (D, router, top-k + softmax, permutation,
routed and shared NVFP4 SwiGLU experts, combine, U) over one batch of seeded
synthetic tokens.  Inputs are resident in HBM before timing; L2 (126 MB) is
defeated by rotating over independent layer instances whose bytes exceed it.
Time is taken with CUDA events on the launching stream (the steps are replayed
from a captured CUDA graph, so host launch cost is not measured), max over
ranks.  ``e2e`` repeats the measurement through the same C-ABI call with the
step's input copied from pinned host memory and its output read back.
``--impl reference`` times the CPU oracle (fp64 numpy) on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: latent, T, seed, layers per step, zipf pattern, instances rotated
    "layer145b_t1": dict(kind="decode", latent=1792, T=1, seed=0, layers=1, zipf=(0.0,), instances=16,
                         desc="one Edge0-145B latent-MoE layer, decode T=1"),
    "layer120b_t4": dict(kind="decode", latent=1280, T=4, seed=1, layers=1, zipf=(0.0,), instances=16,
                         desc="one Edge0-120B latent-MoE layer, speculative-verify batch T=4"),
    "stack48_145b_t1": dict(kind="decode", latent=1792, T=1, seed=2, layers=48, zipf=(0.0,), instances=1,
                            desc="48 Edge0-145B layers (all 48x512 experts resident), decode T=1"),
    "layer145b_t4096_zipf": dict(kind="prefill", latent=1792, T=4096, seed=3, layers=1, zipf=(1.1,),
                                 instances=2,
                                 desc="one Edge0-145B layer, prefill T=4096, Zipf(1.1) router bias"),
    # one layer at the widest verify window: a size for profiling captures of the decode kernel
    "layer145b_t16": dict(kind="decode", latent=1792, T=16, seed=0, layers=1, zipf=(0.0,), instances=16,
                          desc="one Edge0-145B layer, decode verify window T=16 (profiling size)"),
    # one layer of the 16K workload (its uniform-routing first layer): a size for profiling captures
    "layer145b_t16384": dict(kind="prefill", latent=1792, T=16384, seed=4, layers=1, zipf=(0.0,), instances=1,
                             desc="one Edge0-145B layer, prefill T=16384, uniform routing (profiling size)"),
    "prefill4x145b_t16384": dict(kind="prefill", latent=1792, T=16384, seed=4, layers=4,
                                 zipf=(0.0, 1.1, 0.0, 1.1), instances=1,
                                 desc="4 Edge0-145B layers, prefill T=16384, uniform/Zipf(1.1) alternating"),
    # the grouped layer of the default line's grouped object at its prefill size (profiling size)
    "grouped145b_g8_t4096": dict(kind="prefill", latent=1792, T=4096, seed=6, layers=1, zipf=(0.0,), instances=1,
                                 groups=8, shared_group=0,
                                 desc="one Edge0-145B layer with 8 D/U pairs (64 experts per group), prefill T=4096"),
}
DEFAULT_WORKLOAD = "prefill4x145b_t16384"
# reported with the default workload, each as an object of the same line
OTHER_CONFIGS = ("layer145b_t1", "layer120b_t4", "stack48_145b_t1", "layer145b_t4096_zipf")
SWEEP_T = tuple(range(1, 17))          # verify-window sizes of the T = 1..16 decode sweep
REF_SAMPLE_T = {"prefill": 4}          # tokens per reference-arm step (prefill workloads)
HIDDEN, E, K, F = 2560, 512, 10, 640
METRIC = "latent-MoE layer tok/s at T=1 and T=16K; % of HBM / bf16 tensor roofline"
MIN_TIMED_S = 2.0
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant kernel, from one
# ncu capture of the current kernels: the gate/up grouped GEMM on the uniform-routing
# layer of the 16K workload (profiles/ncu_grouped_nvfp4_layer145b_t16384.md), the decode
# kernel on one layer at T=1 (profiles/ncu_moe_decode_layer145b_t1_t16.md)
TRAFFIC = {("prefill4x145b_t16384", "gate_up_grouped"): 1524064000,
           ("layer145b_t1", "moe_decode_kernel"): 45092608}


def flops_per_token_layer(latent, groups=1):
    """Algorithmic FLOPs of one token through one layer: D (every group), router, k
    routed and the shared SwiGLU expert, U (every group) (2 per multiply-add)."""
    return (2 * HIDDEN * groups * latent + 2 * latent * E + (K + 1) * 3 * 2 * latent * F
            + 2 * groups * latent * HIDDEN)


def stage_flops(latent, T, groups=1):
    """Algorithmic FLOPs per launch of the prefill stages that are contractions."""
    TK = T * K
    return {"xz_gemm": 2 * T * HIDDEN * groups * latent + 2 * T * latent * E,
            "gate_up_grouped": 2 * (TK + T) * latent * 2 * F,
            "down_grouped": 2 * (TK + T) * F * latent,
            "u_gemm": 2 * T * groups * latent * HIDDEN}


def record_bytes(latent):
    return 3 * F * latent // 2 + 3 * F * latent // 16 + 12


def decode_algorithmic_bytes(latent, T, distinct_experts):
    """HBM bytes one decode forward must move: D, U, router, every distinct
    routed record once, the shared record, x and y."""
    dense = 2 * latent * HIDDEN * 2 + E * latent * 2
    return dense + (distinct_experts + 1) * record_bytes(latent) + 2 * T * HIDDEN * 2


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling during the timed region (clocks and throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ dist helpers
def dist_setup(n_gpus):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6400.0), d.get("bf16_tflops", 1800.0), d.get("bf16_tflops_sustained", 1400.0), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


# ------------------------------------------------------------------ oracle legs
# The bench runs the oracle (test infrastructure) in three places only, all outside
# the timed regions: the CPU baseline, the reference arm (--impl reference) and the
# parity report on a token sample of the timed inputs.
def _cores():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        return os.cpu_count() or 1


def _oracle_layer(seed, layer, latent, zipf, groups=1, shared_group=0):
    import synth
    from oracle import moe
    spec = synth.LayerSpec(seed=seed, layer=layer, latent=latent, zipf=zipf, groups=groups,
                           shared_group=shared_group)
    inp = synth.make_layer(spec)
    if groups > 1:
        return moe.GroupedLayer(inp.D, inp.U, inp.R, inp.bias, inp.expert, inp.shared, spec.latent, spec.ffn,
                                spec.top_k, inp.labels, shared_group), inp
    return moe.Layer(inp.D, inp.U, inp.R, inp.bias, inp.expert, inp.shared, spec.latent, spec.ffn,
                     spec.top_k), inp


def _pool_init():
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(1)
    except Exception:
        pass


def oracle_task(task):
    """One parity task (run in a spawned worker): ("layer", seed, layer, latent, zipf,
    x, y, idx) -> per-layer metrics on the GPU's input and routing (a grouped layer:
    ("glayer", seed, layer, latent, zipf, groups, shared_group, x, y, idx)); ("chain",
    seed, n_layers, latent, zipfs, x, idx per layer, y) -> end-to-end error of the
    oracle stack forced to the GPU's routing."""
    from oracle import compare, moe
    import numpy as np
    if task[0] in ("layer", "glayer"):
        if task[0] == "layer":
            _, seed, layer, latent, zipf, x, y, idx = task
            lay, _ = _oracle_layer(seed, layer, latent, zipf)
        else:
            _, seed, layer, latent, zipf, groups, sg, x, y, idx = task
            lay, _ = _oracle_layer(seed, layer, latent, zipf, groups, sg)
        rel, mx, flips, bad = compare.layer_check_metrics(lay, x, y, idx)
        return {"kind": "layer", "rel_l2": rel, "max_abs_over_rms": mx, "flips": flips, "bad": len(bad),
                "tokens": int(x.shape[0])}
    _, seed, n_layers, latent, zipfs, x, idx_layers, y = task
    lays = [_oracle_layer(seed, l, latent, zipfs[l % len(zipfs)])[0] for l in range(n_layers)]
    xf, flips, bad = compare.stack_chain(lays, x, idx_layers)
    got, ref = moe.bf16_to_f64(y), moe.bf16_to_f64(xf)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    return {"kind": "chain", "rel_l2": rel, "flips": flips, "bad": len(bad), "tokens": int(x.shape[0]),
            "bound": compare.stack_rel_l2(n_layers)}


def parity_summary(results):
    """Aggregate a config's oracle tasks: worst per-layer errors, flips, end to end."""
    from oracle import compare
    lay = [r for r in results if r["kind"] == "layer"]
    ch = [r for r in results if r["kind"] == "chain"]
    out = {"tokens": max([r["tokens"] for r in results] or [0]), "layers_checked": len(lay),
           "rel_l2_max": round(max([r["rel_l2"] for r in lay] or [0.0]), 6),
           "max_abs_over_rms_max": round(max([r["max_abs_over_rms"] for r in lay] or [0.0]), 6),
           "near_tie_flips": int(sum(r["flips"] for r in lay)),
           "flips_beyond_gap": int(sum(r["bad"] for r in lay)),
           "tolerance": {"rel_l2": compare.REL_L2, "max_abs_over_rms": compare.MAX_ABS, "gap": compare.GAP},
           "teacher_forced": "each layer on the GPU's input; where the GPU's experts differ at a near-tie, "
                             "the oracle is re-run on the GPU's experts"}
    if ch:
        # end to end against the oracle stack forced to the GPU's routing; that chain runs
        # on its own inputs, whose rounding drifts from the GPU's, so its own top-k may
        # differ from the forced choice (counted, not a GPU routing error)
        out["end_to_end_rel_l2"] = round(max(r["rel_l2"] for r in ch), 6)
        out["end_to_end_quadrature_bound"] = round(ch[0]["bound"], 6)
        out["oracle_chain_topk_differs"] = int(sum(r["flips"] + r["bad"] for r in ch))
    out["pass"] = (out["rel_l2_max"] <= compare.REL_L2 and out["max_abs_over_rms_max"] <= compare.MAX_ABS and
                   out["flips_beyond_gap"] == 0)
    return out


def cpu_baseline(wl, T_sample=1024):
    """The oracle as it stands, on host cores, for a bounded sample of the workload:
    one forward of the workload's first layer at T_sample tokens (prefill), or
    forwards of the workload's T tokens until ~10 s have passed (decode)."""
    import synth
    from oracle import moe
    lay, inp = _oracle_layer(wl["seed"], 0, wl["latent"], wl["zipf"][0])
    if wl["kind"] == "prefill":
        T = min(T_sample, wl["T"])
        x = synth.tokens_bf16(1000, T, HIDDEN)
        for e in range(E + 1):               # input bytes generated before the timed region
            inp.expert(e)
        t0 = time.perf_counter()
        moe.layer_forward(lay, x)
        el = time.perf_counter() - t0
        v = T / el / wl["layers"]
        sample = (f"one oracle forward of the workload's layer 0 at T={T} (each expert it uses dequantised "
                  f"once, fp64 matmuls), {el:.1f} s; tokens/s through the {wl['layers']}-layer step = "
                  f"per-layer rate / {wl['layers']} (every layer has the same shapes)")
    else:
        T = wl["T"]
        done, it, t0 = 0, 0, time.perf_counter()
        while True:
            moe.layer_forward(lay, synth.tokens_bf16(1000 + it, T, HIDDEN))
            done += T
            it += 1
            el = time.perf_counter() - t0
            if el > 10.0 or it >= 64:
                break
        v = done / el / wl["layers"]
        sample = f"{it} oracle forward(s) of the workload's layer 0 at T={T}, {el:.1f} s"
    return {"value": round(v, 4), "unit": "tok/s", "cores": _cores(), "kind": "oracle", "sample": sample}


def reference_arm(args, wl, config):
    """--impl reference: the oracle timed on the host, each step one bounded sample
    of the workload (tokens through every layer of the step), W untimed + K timed."""
    import synth
    from oracle import moe
    lays = [_oracle_layer(wl["seed"], l, wl["latent"], wl["zipf"][l % len(wl["zipf"])])[0]
            for l in range(wl["layers"])]
    T_s = REF_SAMPLE_T.get(wl["kind"], 1) if wl["kind"] == "prefill" else wl["T"]
    times = []
    for s in range(args.warmup + args.steps):
        x = synth.tokens_bf16(2000 + s, T_s, HIDDEN)
        t0 = time.perf_counter()
        if wl["layers"] > 1:
            moe.stack_forward(lays, x)
        else:
            moe.layer_forward(lays[0], x)
        el = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(el)
    step_s = statistics.median(times)
    v = T_s / step_s
    sample = (f"{T_s} token(s) of the workload through all {wl['layers']} layer(s) per step "
              f"(oracle, fp64; each step dequantises the experts its tokens use)")
    cfg = dict(config, sample=sample, sample_tokens_per_step=T_s)
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tok/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": cfg,
            "cpu_baseline": {"value": round(v, 4), "unit": "tok/s", "cores": _cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------ our implementation
def build_instances(wl, n_inst, max_tokens):
    import torch
    import synth
    from synth import device
    insts = []
    for i in range(n_inst):
        spec = synth.LayerSpec(seed=wl["seed"], layer=i, latent=wl["latent"],
                               zipf=wl["zipf"][i % len(wl["zipf"])])
        insts.append(device.DeviceLayer(synth.make_layer(spec), max_tokens=max_tokens))
    torch.cuda.synchronize()
    return insts


def timed_region(step, args, stream, world, local, min_s=MIN_TIMED_S, steps=None):
    """Warm-up, capture of the K timed steps in a CUDA graph, and the replay of that
    graph enough times (>= min_s) between events on the launching stream."""
    import torch
    steps = steps or args.steps
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, stream)
    stream.synchronize()
    # per-step estimate from a few direct steps (sets the replay count)
    t0 = time.perf_counter()
    n_est = 2
    with torch.cuda.stream(stream):
        for i in range(n_est):
            step(i, stream)
    stream.synchronize()
    est = (time.perf_counter() - t0) / n_est
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(steps):
                step(args.warmup + i, stream)
        stream.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()                  # one untimed replay (the graph's first launch)
        stream.synchronize()
    except Exception as e:                  # graph capture unavailable: launch directly
        print(f"# graph capture failed ({e}); timing direct launches", file=sys.stderr)
        graph = None
        torch.cuda.synchronize()
    reps = args.repeat if args.repeat else max(1, int(math.ceil(min_s / max(est * steps, 1e-6))))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for r in range(reps):
                if graph is not None:
                    graph.replay()
                else:
                    for i in range(steps):
                        step(args.warmup + i, stream)
            ev1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    el_ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    del graph
    return el_ms, steps * reps, reps, clk.summary()


def e2e_graphs(stream, calls):
    """One CUDA graph per call: H2D copy of its input from pinned host memory, the
    library call, D2H copy of its output to pinned host memory."""
    import torch
    graphs = []
    for c in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            c(stream)
        graphs.append(g)
    stream.synchronize()
    return graphs


def serial_e2e(stream, graphs, n_steps, world):
    """Steps one after another, the host reading each step's result before the next
    (autoregressive decode); CUDA events around the loop on the launching stream."""
    import torch
    # a graph replays on the current stream: every replay is made on the launching stream
    with torch.cuda.stream(stream):
        for g in graphs:
            g.replay()
    stream.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(n_steps):
            graphs[i % len(graphs)].replay()
            stream.synchronize()              # the host reads the step's result
        e1.record(stream)
    stream.synchronize()
    return max_over_ranks(e0.elapsed_time(e1), world) / n_steps


def decode_bytes_of(insts, xs, ys, T, L, stream):
    """Algorithmic bytes of one forward per instance (distinct routed experts read once)."""
    import numpy as np
    import latent_sparse_moe_router_b300 as ext
    out, distinct = [], []
    for j, d in enumerate(insts):
        ext.edge0_moe_forward(d.handle, xs[j], ys[j], T, stream)
        stream.synchronize()
        u = len(np.unique(d.routing(T)["idx"]))
        distinct.append(u)
        out.append(decode_algorithmic_bytes(L, T, u))
    return float(np.mean(out)), float(np.mean(distinct))


def decode_phases(insts, step, stream, n_layers, first, n=8):
    """Mean per-phase microseconds (averaged over layers and n profiled launches)."""
    import numpy as np
    import latent_sparse_moe_router_b300 as ext
    h0 = insts[0].handle
    for d in insts:
        ext.edge0_moe_profile_decode(d.handle, True)
    acc, cnt = None, 0
    for i in range(n):
        j = (first + i) % len(insts) if n_layers == 1 else 0
        step(j, stream)
        stream.synchronize()
        h = insts[j].handle if n_layers == 1 else h0
        for layer in ext.edge0_moe_decode_phase_times(h, n_layers):
            v = np.array([layer[k] for k in ext.DECODE_PHASE_NAMES])
            acc = v if acc is None else acc + v
            cnt += 1
    for d in insts:
        ext.edge0_moe_profile_decode(d.handle, False)
    return {k: round(float(v / cnt), 3) for k, v in zip(ext.DECODE_PHASE_NAMES, acc)}


def run_decode(args, wl, rank, world, local, sweep=None, parity_tokens=2):
    """Decode workloads: one layer at T <= 16 over rotated instances, or the 48-layer stack."""
    import numpy as np
    import torch
    import synth
    import latent_sparse_moe_router_b300 as ext
    from synth import device

    torch.cuda.set_device(local)
    T, L, n_layers = wl["T"], wl["latent"], wl["layers"]
    hbm, bf16, bf16_s, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    jobs = []
    sweep_out = None
    if n_layers == 1:
        insts = build_instances(wl, wl["instances"], max_tokens=16)
        n_inst = len(insts)
        xs = [device.bf16_tensor(synth.tokens_bf16(wl["seed"] * 1000 + rank * 100 + i, T, HIDDEN))
              for i in range(n_inst)]
        ys = [torch.empty_like(x) for x in xs]

        def step(i, s):
            j = i % n_inst
            ext.edge0_moe_forward(insts[j].handle, xs[j], ys[j], T, s)
        bytes_per_step, mean_u = decode_bytes_of(insts, xs, ys, T, L, stream)
        work_note = f"mean distinct routed experts {mean_u:.2f} over {n_inst} rotated instances"
        # parity sample: the timed inputs of the first instances
        for j in range(min(parity_tokens, n_inst)):
            ext.edge0_moe_forward(insts[j].handle, xs[j], ys[j], T, stream)
            stream.synchronize()
            jobs.append(("layer", wl["seed"], j, L, wl["zipf"][j % len(wl["zipf"])],
                         device.bf16_bits(xs[j]), device.bf16_bits(ys[j]), insts[j].routing(T)["idx"]))
        # e2e: pinned host buffers, H2D x, forward, D2H y per step, host waits per step
        hx = [torch.empty((T, HIDDEN), dtype=torch.bfloat16, pin_memory=True) for _ in range(n_inst)]
        hy = [torch.empty((T, HIDDEN), dtype=torch.bfloat16, pin_memory=True) for _ in range(n_inst)]
        for j in range(n_inst):
            hx[j].copy_(xs[j].cpu())

        def e2e_call(j):
            def c(s):
                xs[j].copy_(hx[j], non_blocking=True)
                ext.edge0_moe_forward(insts[j].handle, xs[j], ys[j], T, s)
                hy[j].copy_(ys[j], non_blocking=True)
            return c
        e2e_bytes = T * HIDDEN * 2
    else:
        # the 48-layer stack: all 48 x 512 records resident in one allocation
        stride = ext.edge0_expert_record_stride(L, F)
        big = torch.empty(n_layers * E * stride, dtype=torch.uint8, device="cuda")
        insts = []
        for l in range(n_layers):
            spec = synth.LayerSpec(seed=wl["seed"], layer=l, latent=L)
            rec = big[l * E * stride:(l + 1) * E * stride]
            insts.append(device.DeviceLayer(synth.make_layer(spec), max_tokens=16, records=rec))
        torch.cuda.synchronize()
        handles = [d.handle for d in insts]
        n_tok = 256
        x_bits_all = synth.tokens_bf16(wl["seed"], n_tok, HIDDEN)
        xs_all = device.bf16_tensor(x_bits_all)
        ys_all = torch.empty_like(xs_all)

        def step(i, s):
            j = i % n_tok
            ext.edge0_moe_stack_forward(handles, xs_all[j:j + 1], ys_all[j:j + 1], 1, 1e-6, s)
        bytes_per_step = n_layers * decode_algorithmic_bytes(L, 1, K)
        work_note = "48 layers x (D + U + router + 10 routed + 1 shared record) per token"
        # parity sample: tokens of the timed sequence, every layer traced
        for j in range(parity_tokens):
            tx = torch.empty((n_layers, 1, HIDDEN), dtype=torch.bfloat16, device="cuda")
            ty = torch.empty_like(tx)
            ti = torch.empty((n_layers, 1, K), dtype=torch.int32, device="cuda")
            yj = torch.empty((1, HIDDEN), dtype=torch.bfloat16, device="cuda")
            ext.edge0_moe_stack_forward_trace(handles, xs_all[j:j + 1], yj, 1, 1e-6, tx, ty, ti, stream)
            stream.synchronize()
            txb, tyb, tib = device.bf16_bits(tx), device.bf16_bits(ty), ti.cpu().numpy()
            for l in range(n_layers):
                jobs.append(("layer", wl["seed"], l, L, 0.0, txb[l], tyb[l], tib[l]))
            jobs.append(("chain", wl["seed"], n_layers, L, (0.0,), x_bits_all[j:j + 1], tib, device.bf16_bits(yj)))
        hx = torch.empty((1, HIDDEN), dtype=torch.bfloat16, pin_memory=True)
        hy = torch.empty((1, HIDDEN), dtype=torch.bfloat16, pin_memory=True)
        hx.copy_(xs_all[:1].cpu())
        xd = torch.empty((1, HIDDEN), dtype=torch.bfloat16, device="cuda")
        yd = torch.empty_like(xd)
        n_inst = 1

        def e2e_call(j):
            def c(s):
                xd.copy_(hx, non_blocking=True)
                ext.edge0_moe_stack_forward(handles, xd, yd, 1, 1e-6, s)
                hy.copy_(yd, non_blocking=True)
            return c
        e2e_bytes = HIDDEN * 2

    el_ms, steps_done, reps, clocks = timed_region(step, args, stream, world, local)
    ms_per_step = el_ms / steps_done
    value = T * world / (ms_per_step / 1e3)
    # the step is one kernel launch: its duration is the step time
    achieved_gbs = bytes_per_step / (ms_per_step / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved_gbs / hbm, 4), "traffic": TRAFFIC.get((wl["name"], "moe_decode_kernel")),
            "peak_kind": f"{peak_kind} HBM copy bandwidth",
            "kernel": "moe_decode_kernel", "bytes_per_launch": bytes_per_step, "note": work_note}
    # phase breakdown: a few profiled launches after the timed region (globaltimer stamps)
    phases = decode_phases(insts, step, stream, n_layers, args.warmup)
    graphs = e2e_graphs(stream, [e2e_call(j) for j in range(n_inst)])
    e_ms = serial_e2e(stream, graphs, max(args.steps, 32) if n_layers == 1 else 16, world)
    del graphs
    e2e = {"value": round(T * world / (e_ms / 1e3), 2), "unit": "tok/s", "h2d_bytes_per_step": e2e_bytes,
           "d2h_bytes_per_step": e2e_bytes, "pipelined": False,
           "note": "each step a CUDA graph of [H2D x from pinned host, forward, D2H y to pinned host]; "
                   "the host waits for every step's result before the next"}

    if sweep:
        # verify-window sweep: T tokens per forward over the same rotated instances
        sweep_out = []
        for Ts in sweep:
            xs_s = [device.bf16_tensor(synth.tokens_bf16(7000 + Ts * 100 + i, Ts, HIDDEN)) for i in range(n_inst)]
            ys_s = [torch.empty_like(x) for x in xs_s]
            b, mu = decode_bytes_of(insts, xs_s, ys_s, Ts, L, stream)

            def step_s(i, s, xs_s=xs_s, ys_s=ys_s, Ts=Ts):
                j = i % n_inst
                ext.edge0_moe_forward(insts[j].handle, xs_s[j], ys_s[j], Ts, s)
            el, nd, _, ck = timed_region(step_s, args, stream, world, local, min_s=0.4)
            ms = el / nd
            gbs = b / (ms / 1e3) / 1e9
            sweep_out.append({"T": Ts, "tok_s": round(Ts * world / (ms / 1e3), 1), "us_per_forward": round(ms * 1e3, 2),
                              "distinct_experts": round(mu, 2), "bytes_per_forward": round(b),
                              "achieved_gbs": round(gbs, 1), "frac": round(gbs / hbm, 4),
                              "sm_mhz": ck["sm_mhz"]})
    errs = [ext.edge0_moe_get_error(d.handle) for d in insts]
    assert all(e == ext.EDGE0_OK for e in errs), f"device wait ran out: {errs}"
    for d in insts:
        d.close()
    return dict(value=value, ms_per_step=ms_per_step, roofline=roof, e2e=e2e,
                gpu_launches=1 * steps_done, clocks=clocks, steps_done=steps_done, jobs=jobs, sweep=sweep_out,
                phases=phases)


def run_prefill(args, wl, rank, world, local, parity_tokens=8):
    import numpy as np
    import torch
    import synth
    import latent_sparse_moe_router_b300 as ext
    from synth import device

    torch.cuda.set_device(local)
    T, L, n_layers = wl["T"], wl["latent"], wl["layers"]
    G, sg = wl.get("groups", 1), wl.get("shared_group", 0)
    hbm, bf16, bf16_s, peak_kind = measured_peaks()
    stream = torch.cuda.Stream()
    n_inst = n_layers if n_layers > 1 else wl["instances"]
    insts = []
    for l in range(n_inst):
        spec = synth.LayerSpec(seed=wl["seed"], layer=l, latent=L, zipf=wl["zipf"][l % len(wl["zipf"])], groups=G,
                               shared_group=sg)
        insts.append(device.DeviceLayer(synth.make_layer(spec), max_tokens=T))
    torch.cuda.synchronize()
    handles = [d.handle for d in insts]
    n_x = 1 if n_layers > 1 else n_inst
    x_bits = [synth.tokens_bf16(wl["seed"] * 1000 + rank * 100 + i, T, HIDDEN) for i in range(n_x)]
    xs = [device.bf16_tensor(b) for b in x_bits]
    ys = [torch.empty_like(x) for x in xs]
    per_fwd = ext.PREFILL_KERNELS_PER_FORWARD + (T <= ext.U_SPLIT_MAX_TOKENS)
    if n_layers > 1:
        def step(i, s):
            ext.edge0_moe_stack_forward(handles, xs[0], ys[0], T, 1e-6, s)
        # per layer: the prefill kernels plus the residual norm
        launches_per_step = n_layers * (per_fwd + 1)
    else:
        def step(i, s):
            j = i % n_inst
            ext.edge0_moe_forward(handles[j], xs[j], ys[j], T, s)
        launches_per_step = per_fwd

    el_ms, steps_done, reps, clocks = timed_region(step, args, stream, world, local)
    ms_per_step = el_ms / steps_done
    value = T * world / (ms_per_step / 1e3)          # tokens through the whole step per second
    step_flops = T * n_layers * flops_per_token_layer(L, G)
    step_tflops = step_flops / (ms_per_step / 1e3) / 1e12

    # per-kernel durations: the library's stage events on the launching stream,
    # over a few direct steps after the timed region
    for h in handles:
        ext.edge0_moe_profile_stages(h, True)
    n_prof = max(3, min(args.steps, 8))
    sums = np.zeros(ext.EDGE0_PREFILL_STAGES)
    n_launch = 0
    with torch.cuda.stream(stream):
        for i in range(n_prof):
            if n_layers > 1:
                for l, h in enumerate(handles):
                    # every layer on the step's input x (per-layer stage times, read back per call)
                    ext.edge0_moe_forward(h, xs[0], ys[0], T, stream)
                    sums += np.array(ext.edge0_moe_stage_times(h))
                    n_launch += 1
            else:
                j = i % n_inst
                ext.edge0_moe_forward(handles[j], xs[j], ys[j], T, stream)
                sums += np.array(ext.edge0_moe_stage_times(handles[j]))
                n_launch += 1
    for h in handles:
        ext.edge0_moe_profile_stages(h, False)
    stage_ms = sums / n_launch
    names = ext.PREFILL_STAGE_NAMES
    top = int(np.argmax(stage_ms))
    sflops = stage_flops(L, T, G)
    tname = names[top]
    if tname in sflops:
        ach = sflops[tname] / (stage_ms[top] / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": bf16, "unit": "TFLOP/s",
                "frac": round(ach / bf16, 4), "traffic": TRAFFIC.get((wl["name"], tname)), "kernel": tname,
                "flops_per_launch": sflops[tname],
                "peak_kind": f"{peak_kind} cuBLAS bf16 dense burst (kernel timed alone by stage events at "
                             f"median SM {clocks['sm_mhz']} MHz of max {clocks['sm_max_mhz']})",
                "frac_of_sustained": round(ach / bf16_s, 4),
                "sustained_peak": bf16_s}
    else:
        roof = {"bound": "hbm", "achieved": None, "peak": hbm, "unit": "GB/s", "frac": None, "traffic": None,
                "kernel": tname, "note": "dominant stage is not a contraction"}
    roof["step"] = {"tflops": round(step_tflops, 1), "frac_burst": round(step_tflops / bf16, 4),
                    "frac_sustained": round(step_tflops / bf16_s, 4), "flops_per_step": step_flops,
                    "flops_per_token_layer": flops_per_token_layer(L, G)}
    stages = {n: round(float(m), 4) for n, m in zip(names, stage_ms)}
    stages["timed_layer_ms_sum"] = round(float(stage_ms.sum()), 4)

    # parity sample: seeded token rows of the timed input, every layer on the GPU's
    # input to it (per-layer calls reproduce the stack's bits) and the stack end to end
    jobs = []
    sel = np.sort(np.random.default_rng(77).choice(T, parity_tokens, replace=False))
    cur = xs[0]
    idx_layers = []
    for l in range(n_layers):
        yl = torch.empty_like(cur)
        ext.edge0_moe_forward(handles[l], cur, yl, T, stream)
        stream.synchronize()
        idx = insts[l].routing(T)["idx"][sel]
        idx_layers.append(idx)
        if G > 1:
            jobs.append(("glayer", wl["seed"], l, L, wl["zipf"][l % len(wl["zipf"])], G, sg,
                         device.bf16_bits(cur)[sel], device.bf16_bits(yl)[sel], idx))
        else:
            jobs.append(("layer", wl["seed"], l, L, wl["zipf"][l % len(wl["zipf"])],
                         device.bf16_bits(cur)[sel], device.bf16_bits(yl)[sel], idx))
        if n_layers > 1:
            nx = torch.empty_like(cur)
            ext.edge0_residual_rmsnorm(cur, yl, nx, T, HIDDEN, 1e-6, stream)
            cur = nx
    if n_layers > 1:
        stream.synchronize()
        jobs.append(("chain", wl["seed"], n_layers, L, wl["zipf"], x_bits[0][sel], idx_layers,
                     device.bf16_bits(cur)[sel]))

    # e2e through the C ABI with pinned host buffers: every step copies its x in from pinned
    # host memory, runs the forward and copies its y out to pinned host memory, and the host
    # reads each step's result.  Prefill batches are independent, so the steps are
    # pipelined as a server would run them: step i+1's input copy and step i-1's output
    # copy (each on its own stream) overlap step i's kernels, two device buffers each way,
    # and the host waits for step i-1's result after launching step i.
    hx = torch.empty((T, HIDDEN), dtype=torch.bfloat16, pin_memory=True)
    hy = [torch.empty((T, HIDDEN), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    hx.copy_(xs[0].cpu())
    xb = [xs[0], torch.empty_like(xs[0])]
    yb = [ys[0], torch.empty_like(ys[0])]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    x_in = [torch.cuda.Event() for _ in range(2)]
    y_done = [torch.cuda.Event() for _ in range(2)]
    y_out = [torch.cuda.Event() for _ in range(2)]
    n_e2e = max(3, min(args.steps, 10))

    def fwd(x, y):
        if n_layers > 1:
            ext.edge0_moe_stack_forward(handles, x, y, T, 1e-6, stream)
        else:
            ext.edge0_moe_forward(handles[0], x, y, T, stream)

    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d.wait_event(e0)
    d2h.wait_event(e0)
    for i in range(n_e2e):
        b = i & 1
        if i >= 2:
            h2d.wait_event(y_done[b])           # the forward of step i-2 is done with xb[b]
        with torch.cuda.stream(h2d):
            xb[b].copy_(hx, non_blocking=True)
        x_in[b].record(h2d)
        stream.wait_event(x_in[b])
        if i >= 2:
            stream.wait_event(y_out[b])         # step i-2's y has been copied out of yb[b]
        fwd(xb[b], yb[b])
        y_done[b].record(stream)
        d2h.wait_event(y_done[b])
        with torch.cuda.stream(d2h):
            hy[b].copy_(yb[b], non_blocking=True)
        y_out[b].record(d2h)
        if i >= 1:
            y_out[(i - 1) & 1].synchronize()    # the host reads step i-1's result
    y_out[(n_e2e - 1) & 1].synchronize()        # and the last one
    stream.wait_event(y_out[(n_e2e - 1) & 1])
    e1.record(stream)
    e1.synchronize()
    e_ms = max_over_ranks(e0.elapsed_time(e1), world) / n_e2e
    e2e = {"value": round(T * world / (e_ms / 1e3), 1), "unit": "tok/s",
           "h2d_bytes_per_step": T * HIDDEN * 2, "d2h_bytes_per_step": T * HIDDEN * 2,
           "pipelined": True}
    errs = [ext.edge0_moe_get_error(h) for h in handles]
    assert all(e == ext.EDGE0_OK for e in errs), f"device wait ran out: {errs}"
    for d in insts:
        d.close()
    return dict(value=value, ms_per_step=ms_per_step, roofline=roof, e2e=e2e,
                gpu_launches=launches_per_step * steps_done, clocks=clocks, steps_done=steps_done,
                stages=stages, layer_tok_s=value * n_layers, jobs=jobs)


def run_tiered(args, rank, world, local, n_slots=128, n_warm=64, n_tok=256):
    """Expert residency tiering: one Edge0-145B layer with Zipf(1.1) routing, its 512
    records in pinned host memory and n_slots of them cached in device memory after a
    warm-up and a rebalance; T=1 forwards timed back to back against the handle that
    reads every record from device memory, and the host link's copy bandwidth."""
    import numpy as np
    import torch
    import synth
    import latent_sparse_moe_router_b300 as ext
    from synth import device
    torch.cuda.set_device(local)
    spec = synth.LayerSpec(seed=3, layer=0, latent=1792, zipf=1.1)
    dl = device.DeviceLayer(synth.make_layer(spec), max_tokens=16)
    host = torch.empty(dl.records.numel(), dtype=torch.uint8, pin_memory=True)
    host.copy_(dl.records.cpu())
    tl = ext.MoELayer(hidden=spec.hidden, latent=spec.latent, n_experts=spec.n_experts, top_k=spec.top_k,
                      ffn=spec.ffn, max_tokens=16, D=dl.D, U=dl.U, router=dl.R, router_bias=dl.bias,
                      experts=dl.records, expert_stride=dl.stride, shared_expert=dl.shared)
    stream = torch.cuda.Stream()
    ext.edge0_moe_tier_attach(tl.handle, host, n_slots, stream)
    xs = [device.bf16_tensor(synth.tokens_bf16(9000 + rank * 1000 + j, 1, HIDDEN)) for j in range(n_warm + n_tok)]
    ys = [torch.empty_like(x) for x in xs]
    for j in range(n_warm):
        ext.edge0_moe_forward(tl.handle, xs[j], ys[j], 1, stream)
    ext.edge0_moe_tier_rebalance(tl.handle, stream)
    st0 = ext.edge0_moe_tier_stats(tl.handle)

    def timed(handle):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        e0.record(stream)
        for j in range(n_warm, n_warm + n_tok):
            ext.edge0_moe_forward(handle, xs[j], ys[j], 1, stream)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3

    t_tier = timed(tl.handle)
    st1 = ext.edge0_moe_tier_stats(tl.handle)
    y_tier = [device.bf16_bits(ys[j]) for j in range(n_warm, n_warm + 8)]
    t_res = timed(dl.handle)
    same = all(np.array_equal(a, device.bf16_bits(ys[n_warm + i])) for i, a in enumerate(y_tier))
    # the host link: one 256 MB pinned -> device copy
    src = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    dst.copy_(src, non_blocking=True)
    e1.record()
    e1.synchronize()
    link_gbs = (256 << 20) / (e0.elapsed_time(e1) / 1e3) / 1e9
    misses = st1["misses"] - st0["misses"]
    hbytes = st1["host_bytes"] - st0["host_bytes"]
    out = {"workload": "layer145b_t1_zipf_tiered",
           "desc": "one Edge0-145B layer, Zipf(1.1) routing, records in pinned host memory, "
                   f"{n_slots} of 512 cached in device memory after {n_warm} warm-up tokens and a rebalance",
           "value": round(n_tok / t_tier, 1), "unit": "tok/s", "tokens": n_tok,
           "resident_value": round(n_tok / t_res, 1), "n_slots": n_slots, "resident_experts": st1["resident"],
           "misses_per_token": round(misses / n_tok, 3), "routed_per_token": spec.top_k,
           "host_bytes_per_token": round(hbytes / n_tok), "host_read_gbs": round(hbytes / t_tier / 1e9, 2),
           "host_link_copy_gbs": round(link_gbs, 1),
           "bitwise_equal_to_resident": bool(same),
           "note": "host_read_gbs = bytes copied from host memory over the whole timed interval; "
                   "host_link_copy_gbs = one pinned 256 MB host-to-device copy"}
    assert ext.edge0_moe_get_error(tl.handle) == ext.EDGE0_OK
    tl.close()
    dl.close()
    return out


def run_noalloc(args, rank, world, local, n=40):
    """The allocation-free decode entry against the handle forward on one Edge0-145B
    layer at T=1: the difference is what each of its calls adds (R D and the |z|
    bound recomputed into the library's static scratch)."""
    import numpy as np
    import torch
    import synth
    import latent_sparse_moe_router_b300 as ext
    from synth import device
    torch.cuda.set_device(local)
    spec = synth.LayerSpec(seed=0, layer=0, latent=1792)
    dl = device.DeviceLayer(synth.make_layer(spec), max_tokens=16)
    x = device.bf16_tensor(synth.tokens_bf16(5, 1, HIDDEN))
    y0, y1 = torch.empty_like(x), torch.empty_like(x)
    s = torch.cuda.Stream()

    def na():
        ext.edge0_moe_forward_noalloc(spec.hidden, spec.latent, spec.n_experts, spec.top_k, spec.ffn, dl.D, dl.U,
                                      dl.R, dl.bias, dl.records, dl.stride, dl.shared, x, y1, 1, None, s)

    def hf():
        ext.edge0_moe_forward(dl.handle, x, y0, 1, s)

    out = {}
    for name, f in (("noalloc_us", na), ("handle_us", hf)):
        for _ in range(5):
            f()
        s.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(n):
            f()
        e1.record(s)
        e1.synchronize()
        out[name] = round(e0.elapsed_time(e1) * 1e3 / n, 2)
    out["same_output"] = bool(np.array_equal(device.bf16_bits(y0), device.bf16_bits(y1)))
    out["note"] = ("one Edge0-145B layer at T=1, the same token and weights, calls back to back on one stream "
                   "(same L2 state for both); the difference is the per-call R D and |z|-bound recomputation")
    dl.close()
    return out


GROUPED = dict(latent=1792, groups=8, shared_group=0, seed=6, T=(1, 4096), inputs=16,
               desc="one Edge0-145B layer with grouped latent projections: 8 D/U pairs, 64 experts per group")


def run_grouped(args, rank, world, local, parity_tokens=4):
    """A grouped layer (8 D/U pairs, each expert labelled with its group) at a decode
    size and a prefill size.  Both run the prefill kernels.  T=1 is reported against
    the HBM roofline (every group's D and U, the router operand, the distinct records,
    x and y), T=4096 against the bf16 tensor roofline (the layer's FLOPs with all G
    groups in D and U)."""
    import numpy as np
    import torch
    import synth
    import latent_sparse_moe_router_b300 as ext
    from synth import device
    torch.cuda.set_device(local)
    g = GROUPED
    L, G = g["latent"], g["groups"]
    hbm, bf16, bf16_s, peak_kind = measured_peaks()
    spec = synth.LayerSpec(seed=g["seed"], layer=0, latent=L, groups=G, shared_group=g["shared_group"])
    d = device.DeviceLayer(synth.make_layer(spec), max_tokens=max(g["T"]))
    stream = torch.cuda.Stream()
    out = {"desc": g["desc"], "groups": G, "latent": L, "experts_per_group": E // G, "jobs": []}
    for T in g["T"]:
        n_in = g["inputs"] if T <= 16 else 2
        x_bits = [synth.tokens_bf16(g["seed"] * 1000 + rank * 100 + 10 * T + i, T, HIDDEN) for i in range(n_in)]
        xs = [device.bf16_tensor(b) for b in x_bits]
        ys = [torch.empty_like(x) for x in xs]

        def step(i, s):
            ext.edge0_moe_forward(d.handle, xs[i % n_in], ys[i % n_in], T, s)
        el_ms, steps_done, _, clocks = timed_region(step, args, stream, world, local)
        ms = el_ms / steps_done
        r = {"T": T, "value": round(T * world / (ms / 1e3), 1), "unit": "tok/s", "ms_per_step": round(ms, 6),
             "clocks": clocks,
             "gpu_launches": (ext.PREFILL_KERNELS_PER_FORWARD + (T <= ext.U_SPLIT_MAX_TOKENS)) * steps_done,
             "steps": steps_done}
        if T <= 16:
            distinct = []
            for i in range(n_in):
                ext.edge0_moe_forward(d.handle, xs[i], ys[i], T, stream)
                stream.synchronize()
                distinct.append(len(np.unique(d.routing(T)["idx"])))
            nbytes = (2 * G * L * HIDDEN * 2 + E * HIDDEN * 4 + (np.mean(distinct) + 1) * record_bytes(L)
                      + 2 * T * HIDDEN * 2)
            ach = nbytes / (ms / 1e3) / 1e9
            r["roofline"] = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                             "frac": round(ach / hbm, 4), "traffic": None, "kernel": "whole forward",
                             "bytes_per_forward": int(nbytes),
                             "bytes": "all G D_g and U_g (bf16), the router operand R D (fp32), the "
                                      "distinct routed records and the shared one, x and y",
                             "peak_kind": f"{peak_kind} HBM copy bandwidth"}
        else:
            fl = T * (2 * HIDDEN * G * L + 2 * L * E + (K + 1) * 3 * 2 * L * F + 2 * G * L * HIDDEN)
            tf = fl / (ms / 1e3) / 1e12
            r["roofline"] = {"bound": "tensor", "achieved": round(tf, 1), "peak": bf16, "unit": "TFLOP/s",
                             "frac": round(tf / bf16, 4), "traffic": None, "kernel": "whole forward",
                             "flops_per_forward": fl, "frac_of_sustained": round(tf / bf16_s, 4),
                             "peak_kind": f"{peak_kind} cuBLAS bf16 dense burst"}
        # parity sample: seeded tokens of the timed input, oracle on the GPU's routing
        ext.edge0_moe_forward(d.handle, xs[0], ys[0], T, stream)
        stream.synchronize()
        sel = np.sort(np.random.default_rng(78).choice(T, min(T, parity_tokens), replace=False))
        idx = d.routing(T)["idx"][sel]
        out["jobs"].append(("glayer", g["seed"], 0, L, 0.0, G, g["shared_group"], x_bits[0][sel],
                            device.bf16_bits(ys[0])[sel], idx))
        out[f"t{T}"] = r
    assert ext.edge0_moe_get_error(d.handle) == ext.EDGE0_OK
    d.close()
    return out


def config_of(name, wl, world):
    if wl["kind"] == "prefill":
        l2 = (f"inputs larger than L2: x {wl['T'] * HIDDEN * 2 / 1e6:.0f} MB per layer input, "
              f"expert records ~1 GB per layer, activations ~{wl['T'] * K * (wl['latent'] * 4 + F * 2) * 2 / 1e9:.1f} GB")
    elif wl["layers"] == 1:
        l2 = (f"rotating {wl['instances']} independent layer instances "
              f"(~{wl['instances'] * decode_algorithmic_bytes(wl['latent'], wl['T'], K * wl['T']) / 1e6:.0f} MB touched) > 126 MB L2")
    else:
        l2 = "48-layer stack, 47.6 GB of records > 126 MB L2"
    out = {"workload": name, "desc": wl["desc"], "hidden": HIDDEN, "latent": wl["latent"],
           "experts": E, "top_k": K, "ffn": F, "T": wl["T"], "layers_per_step": wl["layers"],
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU", "l2": l2}
    if wl.get("groups", 1) > 1:
        out["latent_groups"] = wl["groups"]
    return out


def sub_line(name, r, world):
    """The other configurations' objects in the default line."""
    wl = WORKLOADS[name]
    out = {"workload": name, "desc": wl["desc"], "value": round(r["value"], 2), "unit": "tok/s",
           "ms_per_step": round(r["ms_per_step"], 6), "roofline": r["roofline"], "e2e": r["e2e"],
           "clocks": r["clocks"], "gpu_launches": r["gpu_launches"], "steps": r["steps_done"],
           "config": config_of(name, dict(wl, name=name), world)}
    if wl["kind"] == "prefill":
        out["stages_ms_per_layer"] = r["stages"]
    else:
        out["phases_us_per_layer"] = r["phases"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--repeat", type=int, default=0,
                    help="graph replays inside the timed region (0: enough for >= 2 s)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true",
                    help="report the default workload alone (skip the other configurations and the sweep)")
    ap.add_argument("--no-parity", action="store_true", help="skip the oracle parity report")
    ap.add_argument("--only", default="",
                    help="comma list of the other configurations to report with the default workload")
    ap.add_argument("--instances", type=int, default=0,
                    help="override the number of rotated layer instances (profiling runs)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    wl = dict(WORKLOADS[args.workload], name=args.workload)
    if args.instances:
        wl["instances"] = args.instances
    rank, world, local = dist_setup(args.gpus)
    config = config_of(args.workload, wl, world)

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(reference_arm(args, wl, config)), flush=True)
        return

    # the oracle's parity workers are spawned before any CUDA work of this process
    pool = None
    if not args.no_parity and rank == 0:
        import multiprocessing as mp
        pool = mp.get_context("spawn").Pool(max(1, min(32, os.cpu_count() or 1)), initializer=_pool_init)

    run = run_prefill if wl["kind"] == "prefill" else run_decode
    kw = {"sweep": SWEEP_T} if (wl["name"] == "layer145b_t1" and not args.no_decode) else {}
    r = run(args, wl, rank, world, local, **kw)
    extra, jobs = {}, {args.workload: r["jobs"]}
    if wl["kind"] == "prefill":
        extra["stages_ms_per_layer"] = r["stages"]
        extra["layer_tok_s"] = round(r["layer_tok_s"], 1)
    if r.get("sweep"):
        extra["verify_sweep"] = r["sweep"]
    if r.get("phases"):
        extra["phases_us_per_layer"] = r["phases"]
    # the other configurations (and the T = 2..16 verify-window sweep) on the same run
    if args.workload == DEFAULT_WORKLOAD and not args.no_decode:
        import torch
        others = [n for n in OTHER_CONFIGS if not args.only or n in args.only.split(",")]
        for name in others:
            torch.cuda.empty_cache()
            owl = dict(WORKLOADS[name], name=name)
            if owl["kind"] == "decode":
                o = run_decode(args, owl, rank, world, local, sweep=SWEEP_T if name == "layer145b_t1" else None)
            else:
                o = run_prefill(args, owl, rank, world, local)
            jobs[name] = o["jobs"]
            key = "decode_t1" if name == "layer145b_t1" else name
            extra[key] = sub_line(name, o, world)
            if o.get("sweep"):
                extra["verify_sweep"] = {"workload": name, "layer": "Edge0-145B", "points": o["sweep"]}
        if not args.only or "tiered" in args.only.split(","):
            torch.cuda.empty_cache()
            extra["tiered_decode"] = run_tiered(args, rank, world, local)
        if not args.only or "noalloc" in args.only.split(","):
            extra["noalloc_decode"] = run_noalloc(args, rank, world, local)
        if not args.only or "grouped" in args.only.split(","):
            torch.cuda.empty_cache()
            gr = run_grouped(args, rank, world, local)
            jobs["grouped_145b_g8"] = gr.pop("jobs")
            extra["grouped_145b_g8"] = gr
    if rank != 0:
        return
    if pool is not None:
        parity = {}
        for name, js in jobs.items():
            res = pool.map(oracle_task, js) if js else []
            parity[name] = parity_summary(res)
        pool.close()
        pool.join()
        extra["parity"] = parity
    cb = None if args.no_cpu_baseline else cpu_baseline(wl)
    line = {"metric": METRIC, "value": round(r["value"], 1), "unit": "tok/s", "n_gpus": world,
            "steps": r["steps_done"], "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "nvfp4 weights; bf16 operands on the tensor cores (f16 in the decode GEMV); fp32 accumulate",
            "data": "synthetic (seeded; random NVFP4 experts and N(0,1/fan_in) bf16 projections)",
            "config": config, "roofline": r["roofline"], "cpu_baseline": cb, "e2e": r["e2e"],
            "gpu_launches": r["gpu_launches"], "clocks": r["clocks"]}
    line.update(extra)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
