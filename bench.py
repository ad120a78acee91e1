"""Benchmark of the MXFP4 routed-expert MoE layer on one GB300 (or N ranks).

Headline workload: one MoE layer, batch-1 decode -- 896 experts of
d=7168, f=1536 resident in HBM (15.7 GB), router W_r bf16 [896 x 7168],
x fp32, top-16, softmax combine over the selected logits.  A step is one
token through the whole layer (router + top-k + 16 experts + combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` is tokens/s of the whole job (every
rank runs independent tokens: weak scaling, no collective on the data path).
Every timed region is exactly K steps between two events on the launching
stream (a barrier and a device synchronisation on both sides); the region
is repeated (at least 20 times, and for about a second in all) and the
median is reported with its minimum and maximum.  The same line carries the
other resident-pool configurations under "configs" (same pool, same rules):
the single-expert GEMV, batched decode of 64 tokens and prefill of 4096.

One configuration alone, one JSON line each:
  --workload expert       one expert GEMV (gate/up + SwiGLU + down), 1 token
  --workload decode64     batched decode, 64 tokens, grouped by expert
  --workload prefill4096  4096 bf16 tokens, selection bias ~N(0,1)
  --workload prefill4096_mxq  the same with the activations quantised to
                          MXFP4 (block-scaled E2M1 x E2M1 products)
  --workload shared       the two bf16 shared experts of a layer, batch 1
  --workload stream       4 layers x 896 experts in pinned host memory behind
                          an 8 GB HBM LRU cache, 256 tokens, RMSNorm +
                          residual, Zipf(1.1) selection bias; the recorded
                          trace is replayed offline (LRU, Belady, sizes);
                          --pin-hot N pins the N most requested experts of
                          256 untimed history tokens first
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

D, F, E, K = 7168, 1536, 896, 16
EXPERT_BYTES = 17547264
ROUTER_BYTES = E * D * 2
GATEUP_BYTES = K * 2 * (F * D // 2 + F * D // 32)   # 187,170,816
DOWN_BYTES = K * (D * F // 2 + D * F // 32)          # 93,585,408
LAYER_BYTES = K * EXPERT_BYTES + ROUTER_BYTES        # 293,601,280
N_ROUTER_COPIES = 16
# DRAM read + write bytes of one launch of the fused batch-1 kernel at the
# 896-expert workload, from a one-pass ncu capture of this bench (median of
# three launches); the algorithmic bytes are LAYER_BYTES = 293,601,280.
# None whenever the kernel changed since the capture; the last capture is
# kept beside it, labelled.
FUSED_TRAFFIC = None
FUSED_TRAFFIC_LAST = 294038272
# The same for the block-scaled batch-1 kernel (k3_mx_layer<float>): median
# of five launches (read 297,508,864 B + write 3,815,936 B), this build.
MX_TRAFFIC = 301324800
MX_TRAFFIC_LAST = 301324800
TRAFFIC_LAST_NOTE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch at this workload "
                     "(median of 3 launches), taken before the router rule became selectable; the "
                     "kernel has changed since, its memory accesses have not")
N_TOKENS = 1024
# Kernels of the secondary configurations (names for the roofline lines and
# launches per step).  One expert: gate/up + SwiGLU, then down.
EXPERT_GEMV_KERNEL = "k3_rows_pipe + k3_down_t1 (one expert: gate/up + SwiGLU, down)"
EXPERT_GEMV_LAUNCHES = 2
# Multi-token forwards: router GEMM + top-k, grouping, tile plan, token
# scales, token gather, gate/up, h pieces, down + combine.
GROUPED_GATEUP_KERNEL = "k3_tc_expert<0,1> (tcgen05 kind::f8f6f4)"
GROUPED_LAUNCHES = 9
# With MXFP4 activations (K3MOE_OPT_MXQ): router GEMM + top-k, grouping,
# tile plan, pair slots, token tiles, gate/up, down + combine.
MXQ_GATEUP_KERNEL = "k3_mxq_expert<0> (tcgen05 kind::mxf4, E2M1 x E2M1, block-scaled)"
MXQ_LAUNCHES = 8
FP4_PER_BF16 = 6.0  # nominal dense FP4 : bf16 tensor throughput (13.5 : 2.25 PFLOP/s)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------ ranks
# N > 1: every rank runs the same workload on its own GPU over its own
# tokens (weak scaling, no collective on the data path).  The only
# cross-rank steps are a barrier around the timed region and the maximum of
# the ranks' times, which sets the whole job's rate.

def max_over_ranks(v, world, device=None):
    """Largest value of `v` over all ranks (v itself when world == 1)."""
    if world <= 1:
        return v
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rank_first_token(rank, n_per_rank):
    """Index of the first synthetic token of this rank's disjoint shard."""
    return rank * n_per_rank


def job_rate(units_per_rank, world, ms_max):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    return units_per_rank * world / (ms_max * 1e-3)


def measured_bf16_tflops():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- setup

def build_pool(dev, pool_id=1, layer=0):
    """896 packed experts in one device tensor (generated on the host by the
    seeded generator, copied through a pinned staging buffer)."""
    import torch
    import synth
    from mxfp4_routed_expert_select_gb300 import k3moe as k
    eb = k.expert_bytes(D, F)
    blobs = torch.empty((E, eb), dtype=torch.uint8, device=dev)
    stage = [torch.empty(eb, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    evs = [torch.cuda.Event() for _ in range(2)]
    t0 = time.time()
    for e in range(E):
        b = e % 2
        evs[b].synchronize()
        views = k.host_plane_views(stage[b].data_ptr(), D, F)
        ex = synth.expert(pool_id, layer, e, D, F)
        for name, arr in views.items():
            arr[...] = ex[name]
        blobs[e].copy_(stage[b], non_blocking=True)
        evs[b].record()
    torch.cuda.synchronize()
    log("pool: %d experts (%.2f GB) in %.1f s" % (E, E * eb / 1e9, time.time() - t0))
    return blobs, [k.expert_view(blobs[e].data_ptr(), D, F) for e in range(E)]


def cpu_baseline_sample(budget_s=12.0, pool_id=1):
    """The oracle as it stands on the host cores: whole layer for as many
    tokens as fit in ~budget_s (at least one)."""
    import oracle
    import synth
    Wr_bits = synth.router_bf16(pool_id, 0, E, D)
    done, t_oracle = 0, 0.0
    while True:
        x = synth.token_f32(pool_id, done, D).astype(np.float64)[None]
        lg = oracle.router_logits(x, Wr_bits)
        ids, w, _ = oracle.topk(lg, K)
        ex = {int(e): synth.expert(pool_id, 0, int(e), D, F) for e in ids[0]}
        t0 = time.perf_counter()
        lg = oracle.router_logits(x, Wr_bits)
        ids, w, _ = oracle.topk(lg, K)
        oracle.combine(x, ids, w, ex, E)
        t_oracle += time.perf_counter() - t0
        done += 1
        if t_oracle >= budget_s or done >= 64:
            break
    return done, t_oracle, oracle.max_threads()


# ---------------------------------------------------------------- timing

MIN_REPEATS = 20      # timed regions per measurement, at least
REGION_SECONDS = 1.0  # ... and about this long in all


def max_over_ranks_list(vals, world, device=None):
    """Element-wise maximum over all ranks of a list of floats."""
    if world <= 1:
        return list(vals)
    import torch
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def graph_plan(steps, n_inputs, chunk_max=32):
    """How a timed region of exactly `steps` steps is replayed from CUDA
    graphs: `full` replays of graphs holding `chunk` consecutive steps, then
    one graph of the `rem` remaining steps (full * chunk + rem == steps).
    `variants` graphs of `chunk` steps start at input offsets chunk * v, so
    that successive replays walk up to `n_inputs` distinct inputs."""
    steps = max(1, int(steps))
    chunk = max(1, min(steps, chunk_max))
    full, rem = divmod(steps, chunk)
    variants = max(1, min(n_inputs // chunk, 64)) if full else 0
    return {"chunk": chunk, "full": full, "rem": rem, "variants": variants}


def spread(ms, steps):
    """Median, minimum and maximum per-step time (ms) over the repeats."""
    return {"repeats": len(ms), "ms_per_step_median": round(statistics.median(ms) / steps, 6),
            "ms_per_step_min": round(min(ms) / steps, 6), "ms_per_step_max": round(max(ms) / steps, 6)}


def timed_region(step, steps, warmup, dev_index, world, use_graph=True, n_inputs=1, chunk_max=32,
                 min_repeats=None, seconds=None):
    """Warm-up, then the timed region -- exactly `steps` steps between two
    events on the current stream, a barrier (N > 1) and a device
    synchronisation before it and a synchronisation after it -- repeated at
    least `min_repeats` times and for about `seconds` in all, with the
    clocks sampled meanwhile.  step(i) enqueues step i (its input i mod
    n_inputs).  Returns (ms of each repeat, max over ranks; clocks; plan)."""
    import torch
    min_repeats = MIN_REPEATS if min_repeats is None else min_repeats
    seconds = REGION_SECONDS if seconds is None else seconds
    s = torch.cuda.current_stream()
    dev = torch.device("cuda", dev_index)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if use_graph:
        plan = graph_plan(steps, n_inputs, chunk_max)
        graphs = []
        for v in range(plan["variants"]):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for j in range(plan["chunk"]):
                    step(v * plan["chunk"] + j)
            graphs.append(g)
        g_rem = None
        if plan["rem"]:
            g_rem = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_rem):
                for j in range(plan["rem"]):
                    step(j)
        for g in graphs + ([g_rem] if g_rem is not None else []):  # untimed first replays
            g.replay()
        torch.cuda.synchronize()
        ctr = [0]

        def region():
            for _ in range(plan["full"]):
                graphs[ctr[0] % len(graphs)].replay()
                ctr[0] += 1
            if g_rem is not None:
                g_rem.replay()
    else:
        plan = {"graph": None}
        base = [warmup]

        def region():
            for i in range(steps):
                step(base[0] + i)
            base[0] += steps
    t0 = time.perf_counter()  # one untimed region sizes the repeats
    region()
    torch.cuda.synchronize()
    one = max_over_ranks(max(time.perf_counter() - t0, 1e-6), world, dev)
    repeats = max(min_repeats, min(5000, int(seconds / one)))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(repeats)]
    clock = ClockSampler(dev_index)
    clock.start()
    time.sleep(0.3)
    for r in range(repeats):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev[r][0].record(s)
        region()
        ev[r][1].record(s)
        torch.cuda.synchronize()
    clocks = clock.stop()
    ms = max_over_ranks_list([a.elapsed_time(b) for a, b in ev], world, dev)
    return ms, clocks, plan


def _kernel_events(layer, step, n):
    """Per-phase durations (ms) of `n` eager forwards, from the layer's four
    events recorded on its stream: [route, route->gate/up, gate/up->end]."""
    import torch
    s = torch.cuda.current_stream()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for q in evs:  # torch creates the CUDA event at its first record
        for e in q:
            e.record(s)
    torch.cuda.synchronize()
    for i in range(n):
        layer.set_events(evs[i])
        step(i)
    layer.set_events(None)
    torch.cuda.synchronize()
    return ([q[0].elapsed_time(q[1]) for q in evs], [q[1].elapsed_time(q[2]) for q in evs],
            [q[2].elapsed_time(q[3]) for q in evs])


DATA = ("synthetic (seeded SplitMix64: uniform E2M1 codes, E8M0 in [120,130], x ~ N(0,1), "
        "W_r ~ N(0,0.02) bf16)")


def _roofline(name, nbytes, k_ms, bound="hbm", traffic=None, traffic_src=None):
    peak, src = measured_peaks()
    ach = nbytes / (k_ms * 1e-3) / 1e9
    return {"kernel": name, "bound": bound, "achieved": round(ach, 1), "peak": peak,
            "peak_source": src, "unit": "GB/s", "frac": round(ach / peak, 4), "traffic": traffic,
            "traffic_source": traffic_src, "algorithmic_bytes": int(nbytes)}


def _e2e(step_host, steps, warmup, world, dev_index, h2d, d2h, units_per_step, unit):
    """The metric end to end: every step copies its inputs from pinned host
    memory and reads its result back (eager launches), same timing rules."""
    ms, _, _ = timed_region(step_host, steps, warmup, dev_index, world, use_graph=False,
                            seconds=REGION_SECONDS / 2)
    med = statistics.median(ms)
    return {"value": round(job_rate(steps * units_per_step, world, med), 2), "unit": unit,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "repeats": len(ms)}


class Ctx:
    """What every resident-pool configuration shares: the device, the 896
    packed experts in HBM and the router weights."""

    def __init__(self, dev_index):
        import torch
        import synth
        self.dev_index = dev_index
        self.dev = torch.device("cuda", dev_index)
        torch.cuda.set_device(self.dev)
        self.blobs, self.views = build_pool(self.dev)
        self.Wr_bits = synth.router_bf16(1, 0, E, D)
        self.Wr0 = torch.from_numpy(self.Wr_bits.view(np.int16)).to(self.dev)


# ------------------------------------------------------------------ arms

def run_decode1(args, ctx, rank, world):
    """The headline: batch-1 decode through the whole layer, one token per
    step, 1024 distinct tokens and 16 router copies walked by the replays."""
    import torch
    import synth
    from mxfp4_routed_expert_select_gb300 import k3moe as k
    dev = ctx.dev
    routers = [ctx.Wr0] + [ctx.Wr0.clone() for _ in range(N_ROUTER_COPIES - 1)]
    layers = [k.Layer(E, K, D, F, r, ctx.views, max_tokens=1) for r in routers]
    X = torch.from_numpy(np.stack([synth.token_f32(1, rank_first_token(rank, N_TOKENS) + t, D)
                                   for t in range(N_TOKENS)])).to(dev)
    out = torch.empty(D, dtype=torch.float32, device=dev)

    def step(i):
        layers[i % N_ROUTER_COPIES].forward(X[i % N_TOKENS], 1, out)

    ms, clocks, plan = timed_region(step, args.steps, args.warmup, ctx.dev_index, world,
                                    use_graph=not args.no_graph, n_inputs=N_TOKENS)
    per = statistics.median(ms) / args.steps
    # each layer kernel's own duration, eager, events on its stream around it
    n_ev = min(args.steps, 200)
    r_ms, gu_ms, dn_ms = _kernel_events(layers[0], lambda i: layers[0].forward(X[i % N_TOKENS], 1, out), n_ev)
    eager_ms = statistics.mean([a + b + c for a, b, c in zip(r_ms, gu_ms, dn_ms)])

    # e2e through the C ABI with host buffers: H2D of the token, the layer,
    # D2H of the output, every step
    xh = torch.empty((N_TOKENS, D), dtype=torch.float32, pin_memory=True)
    xh.copy_(X.cpu())
    oh = torch.empty(D, dtype=torch.float32, pin_memory=True)
    xd = torch.empty(D, dtype=torch.float32, device=dev)

    def step_host(i):
        xd.copy_(xh[i % N_TOKENS], non_blocking=True)
        layers[i % N_ROUTER_COPIES].forward(xd, 1, out)
        oh.copy_(out, non_blocking=True)

    e2e = _e2e(step_host, args.steps, args.warmup, world, ctx.dev_index, D * 4, D * 4, 1, "tokens/s")

    mx, fused = layers[0].mx_t1(), layers[0].fused_t1()
    if mx:
        k_name = "k3_mx_layer<float> (router + top-k + 16 experts on tcgen05 kind::mxf4 + combine)"
        traffic, traffic_last = (MX_TRAFFIC, None) if E == 896 and MX_TRAFFIC else \
            (None, {"bytes": MX_TRAFFIC_LAST, "source": TRAFFIC_LAST_NOTE} if E == 896 else None)
    elif fused:
        k_name = "k3_moe_t1_fused (router + top-k + 16 experts + combine)"
        traffic, traffic_last = (FUSED_TRAFFIC, None) if E == 896 and FUSED_TRAFFIC else \
            (None, {"bytes": FUSED_TRAFFIC_LAST, "source": TRAFFIC_LAST_NOTE} if E == 896 else None)
    else:
        k_name, traffic, traffic_last = "k3_router_t1 + k3_rows_t1 + k3_down_t1", None, None
    # one kernel per step (default path): its average duration over the timed
    # region, replay gaps included, is at most the step time
    k_ms = per if (mx or fused) and not args.no_graph else eager_ms
    roof = _roofline(k_name, LAYER_BYTES, k_ms, traffic=traffic,
                     traffic_src=("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch at this "
                                  "workload (median of the captured launches)") if traffic else None)
    if traffic_last:
        roof["traffic_last_capture"] = traffic_last
    peak = roof["peak"]
    layer_gbs = LAYER_BYTES / (per * 1e-3) / 1e9
    result = {
        "metric": "MoE-layer decode tokens/s (batch 1, 896 experts, top-16, MXFP4)",
        "value": round(job_rate(args.steps, world, statistics.median(ms)), 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4 weights (e2m1 + e8m0), fp32 activations and accumulation",
        "data": DATA,
        "config": {"workload": "moe_layer_decode_b1: %d experts d=7168 f=1536 resident (%.1f GB), "
                               "router bf16 [%dx7168], top-16, softmax combine" % (E, E * EXPERT_BYTES / 1e9, E),
                   "global_batch": world, "seq_len": 1, "parallelism": "replicas" if world > 1 else "single",
                   "launch": ("cuda graphs of %d steps (%d offsets) + %d, replayed" %
                              (plan["chunk"], plan["variants"], plan["rem"])) if plan.get("chunk")
                   else "host launch per step",
                   "l2": "inputs larger than L2: every step reads 16 experts (281 MB) and a router "
                         "copy (12.8 MB); %d router copies and %d distinct tokens walked by the "
                         "replays" % (N_ROUTER_COPIES, min(N_TOKENS, max(plan.get("variants", 1), 1) *
                                                                 plan.get("chunk", args.steps)))},
        "timing": spread(ms, args.steps),
        "layer_hbm": {"bytes_per_token": LAYER_BYTES, "gbs": round(layer_gbs, 1),
                      "frac_of_peak": round(layer_gbs / peak, 4), "frac_of_8tbs": round(layer_gbs / 8000, 4)},
        "kernels_ms": {"layer_kernel": round(k_ms, 6), "layer_kernel_eager_events": round(eager_ms, 6),
                       "eager_launches_sampled": n_ev},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": (1 if (fused or mx) else 3) * args.steps,
        "clocks": clocks,
    }
    for l in layers:
        l.close()
    return result


def run_reference(args):
    """The oracle (plain fp64 C on the host cores) on the same workload; each
    step is one token through router + top-k + 16 experts + combine, or a
    fixed fraction of a token when K + W steps would not fit in ~3 minutes."""
    import oracle
    import synth
    Wr_bits = synth.router_bf16(1, 0, E, D)
    # probe one token to size the per-step sample
    x = synth.token_f32(1, 0, D).astype(np.float64)[None]
    lg = oracle.router_logits(x, Wr_bits)
    ids, w, _ = oracle.topk(lg, K)
    ex = {int(e): synth.expert(1, 0, int(e), D, F) for e in ids[0]}
    t0 = time.perf_counter()
    oracle.combine(x, ids, w, ex, E)
    per_token = time.perf_counter() - t0
    budget = 180.0
    frac_experts = K
    while frac_experts > 1 and per_token * frac_experts / K * (args.steps + args.warmup) > budget:
        frac_experts //= 2
    times = []
    for i in range(args.warmup + args.steps):
        x = synth.token_f32(1, i, D).astype(np.float64)[None]
        ids_full = oracle.topk(oracle.router_logits(x, Wr_bits), K)[0]
        sub = ids_full[:, :frac_experts]
        ex = {int(e): synth.expert(1, 0, int(e), D, F) for e in sub[0]}
        t0 = time.perf_counter()
        lg = oracle.router_logits(x, Wr_bits)
        ids, w, _ = oracle.topk(lg, K)
        oracle.combine(x, ids[:, :frac_experts], w[:, :frac_experts], ex, E)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    tok = len(times) * frac_experts / K
    value = tok / sum(times)
    sample = ("%d steps, each one token through the oracle's router + top-16 + %d of its 16 "
              "experts + combine (value counts %d/16 token per step)" % (len(times), frac_experts, frac_experts))
    return {
        "impl": "reference",
        "metric": "MoE-layer decode tokens/s (batch 1, 896 experts, top-16, MXFP4)",
        "value": round(value, 4), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (same seeded inputs)",
        "config": {"workload": "moe_layer_decode_b1: 896 experts d=7168 f=1536, router bf16, top-16"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------ other workloads

def _base_line(metric, value, unit, world, args, ms_step, dtype, config, clocks):
    return {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype, "data": DATA,
            "config": config, "clocks": clocks}


def cfg_steps(args, cap):
    """Steps of one timed region of a secondary configuration: --steps, at
    most `cap` (so that the default line stays within about a minute)."""
    return max(1, min(args.steps, cap))


def run_expert(args, ctx, rank, world):
    """One expert GEMV per step, rotating over the 896 resident experts and
    1024 tokens (17.5 MB per expert: every step reads HBM, not L2)."""
    import torch
    import synth
    from mxfp4_routed_expert_select_gb300 import k3moe as k
    dev = ctx.dev
    steps = cfg_steps(args, 1024)
    X = torch.from_numpy(np.stack([synth.token_f32(1, rank * N_TOKENS + t, D)
                                   for t in range(N_TOKENS)])).to(dev)
    y = torch.empty(D, dtype=torch.float32, device=dev)
    ws = torch.zeros(k.expert_gemv_workspace(D, F) // 4 + 4, dtype=torch.float32, device=dev)
    perm = synth.permutation(E, synth.tag(synth.K_MISC, 1, 0, 7))

    def step(i):
        k.expert_gemv(y, X[i % N_TOKENS], ctx.views[int(perm[i % E])], D, F, ws)

    ms, clocks, plan = timed_region(step, steps, args.warmup, ctx.dev_index, world, True, n_inputs=E)
    per = statistics.median(ms) / steps
    nbytes = EXPERT_BYTES + 2 * D * 4
    xh = torch.empty((N_TOKENS, D), dtype=torch.float32, pin_memory=True)
    xh.copy_(X.cpu())
    yh = torch.empty(D, dtype=torch.float32, pin_memory=True)
    xd = torch.empty(D, dtype=torch.float32, device=dev)

    def step_host(i):
        xd.copy_(xh[i % N_TOKENS], non_blocking=True)
        k.expert_gemv(y, xd, ctx.views[int(perm[i % E])], D, F, ws)
        yh.copy_(y, non_blocking=True)

    e2e = _e2e(step_host, steps, args.warmup, world, ctx.dev_index, D * 4, D * 4, 1, "expert GEMVs/s")
    return {
        "metric": "single MXFP4 expert GEMV (1 token, d=7168, f=1536) per second",
        "value": round(job_rate(steps, world, statistics.median(ms)), 2), "unit": "expert GEMVs/s",
        "steps": steps, "ms_per_step": round(per, 6), "higher_is_better": True,
        "config": {"workload": "expert_gemv_b1: one expert d=7168 f=1536 (17,547,264 B), x fp32 [7168], "
                               "y fp32 [7168]",
                   "launch": "cuda graphs of %d steps (%d offsets) + %d, replayed" %
                             (plan["chunk"], plan["variants"], plan["rem"]),
                   "l2": "inputs larger than L2: 896 distinct experts (15.7 GB) rotated"},
        "timing": spread(ms, steps),
        "roofline": _roofline(EXPERT_GEMV_KERNEL, nbytes, per),
        "tflops": round(2 * 3 * D * F / (per * 1e-3) / 1e12, 3),
        "e2e": e2e, "gpu_launches": EXPERT_GEMV_LAUNCHES * steps, "clocks": clocks,
        "expert_hbm": {"bytes_per_gemv": nbytes, "gbs": round(nbytes / (per * 1e-3) / 1e9, 1)}}


def run_shared(args, ctx, rank, world, n_layers=4, n_shared=2):
    """The two bf16 shared experts of a layer at batch 1 (132 MB per token
    at d = 7168, f = 1536), four layers' copies rotated so that every step
    reads HBM."""
    import torch
    import synth
    from mxfp4_routed_expert_select_gb300 import k3moe as k
    dev = ctx.dev
    steps = cfg_steps(args, 256)
    sb = k.shared_expert_bytes(D, F)
    blobs = torch.empty((n_layers * n_shared, sb), dtype=torch.uint8, device=dev)
    for l in range(n_layers):
        for s_ in range(n_shared):
            ex = synth.shared_expert(3, l, s_, D, F)
            raw = np.concatenate([ex["gate"].ravel(), ex["up"].ravel(), ex["down"].ravel()]).view(np.uint8)
            blobs[l * n_shared + s_].copy_(torch.from_numpy(raw))
    views = [[k.shared_expert_view(blobs[l * n_shared + s_].data_ptr(), D, F) for s_ in range(n_shared)]
             for l in range(n_layers)]
    X = torch.from_numpy(np.stack([synth.token_f32(3, rank * N_TOKENS + t, D) for t in range(N_TOKENS)])).to(dev)
    y = torch.empty(D, dtype=torch.float32, device=dev)
    ws = torch.empty(k.shared_workspace(n_shared, F) // 4, dtype=torch.float32, device=dev)

    def step(i):
        k.shared_forward(y, X[i % N_TOKENS], 1, views[i % n_layers], D, F, ws)

    ms, clocks, plan = timed_region(step, steps, args.warmup, ctx.dev_index, world, True, n_inputs=N_TOKENS)
    per = statistics.median(ms) / steps
    nbytes = n_shared * sb + 2 * D * 4
    return {
        "metric": "shared-expert tokens/s (the two bf16 shared experts of a layer, batch 1)",
        "value": round(job_rate(steps, world, statistics.median(ms)), 2), "unit": "tokens/s",
        "steps": steps, "ms_per_step": round(per, 6), "higher_is_better": True,
        "dtype": "bf16 weights, fp32 activations and accumulation",
        "config": {"workload": "shared_experts_b1: 2 bf16 SwiGLU experts d=7168 f=1536 (%d B), x fp32 [7168]"
                               % (n_shared * sb),
                   "launch": "cuda graphs of %d steps (%d offsets) + %d, replayed" %
                             (plan["chunk"], plan["variants"], plan["rem"]),
                   "l2": "inputs larger than L2: %d layers' shared experts (%.0f MB) rotated" %
                         (n_layers, n_layers * n_shared * sb / 1e6)},
        "timing": spread(ms, steps),
        "roofline": _roofline("k3_shared_gateup + k3_shared_down (bf16 rows, CUDA cores)", nbytes, per),
        "gpu_launches": 2 * steps, "clocks": clocks}


def run_batched(args, ctx, rank, world, T, bf16, use_bias, mxq=False):
    """The layer on T tokens per step: the grouped path (router, top-k,
    grouping by expert, grouped gate/up + SwiGLU, grouped down, combine);
    mxq: with MXFP4-quantised activations on block-scaled MMAs."""
    import torch
    import synth
    from mxfp4_routed_expert_select_gb300 import k3moe as k
    dev = ctx.dev
    if args.tokens:
        T = args.tokens  # smaller batches for profiler captures
    steps = cfg_steps(args, 64 if T <= 64 else 20)
    bias = None
    if use_bias:
        bias = torch.from_numpy(synth.bias_normal(1, 0, E).astype(np.float32)).to(dev)
    NB = max(2, min(16, (1 << 28) // (T * D * (2 if bf16 else 4))))
    n_r = 4 if T >= 1024 else 16
    routers = [ctx.Wr0] + [ctx.Wr0.clone() for _ in range(n_r - 1)]
    layers = [k.Layer(E, K, D, F, r, ctx.views, bias, max_tokens=T) for r in routers]
    if mxq:
        for l in layers:
            l.set_option(k.K3MOE_OPT_MXQ, 1)
        assert layers[0].mxq(), "the MXFP4-activation path does not apply to this layer"
    if bf16:
        Xs = [torch.from_numpy(synth.tokens_bf16(1, T, D, t0=rank * NB * T + b * T).view(np.int16))
              .to(dev).view(torch.bfloat16) for b in range(NB)]
    else:
        Xs = [torch.from_numpy(synth.tokens_f32(1, T, D, t0=rank * NB * T + b * T)).to(dev)
              for b in range(NB)]
    out = torch.empty((T, D), dtype=torch.float32, device=dev)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)

    def step(i):
        layers[i % n_r].forward(Xs[i % NB], T, out)

    # distinct experts per batch (the weight bytes a batch must read)
    U = []
    for b in range(NB):
        layers[0].forward(Xs[b], T, out, ids)
        torch.cuda.synchronize()
        U.append(len(np.unique(ids.cpu().numpy())))
    Umean = statistics.mean(U)
    use_graph = T <= 64
    ms, clocks, plan = timed_region(step, steps, args.warmup, ctx.dev_index, world, use_graph,
                                    n_inputs=NB, chunk_max=8)
    per = statistics.median(ms) / steps
    r_ms, gu_ms, dn_ms = _kernel_events(layers[0], lambda i: layers[0].forward(Xs[i % NB], T, out),
                                        64 if T <= 64 else 8)
    xb = T * D * (2 if bf16 else 4)
    w_bytes = Umean * EXPERT_BYTES
    step_bytes = w_bytes + ROUTER_BYTES + xb + T * D * 4
    gu_bytes = Umean * 2 * (F * D // 2 + F * D // 32) + xb
    flops = 2 * T * K * 3 * D * F + 2 * T * E * D
    xh = torch.empty(tuple(Xs[0].shape), dtype=Xs[0].dtype, pin_memory=True)
    xh.copy_(Xs[0].cpu())
    oh = torch.empty((T, D), dtype=torch.float32, pin_memory=True)
    xd = torch.empty_like(Xs[0])

    def step_host(i):
        xd.copy_(xh, non_blocking=True)
        layers[i % n_r].forward(xd, T, out)
        oh.copy_(out, non_blocking=True)

    e2e = _e2e(step_host, steps, args.warmup, world, ctx.dev_index, xb, T * D * 4, T, "tokens/s")
    name = ("decode%d" % T if T <= 64 else "prefill%d" % T) + ("_mxq" if mxq else "")
    desc = ("moe_layer_%s: %d experts d=7168 f=1536 resident (%.1f GB), router bf16 [%dx7168], "
            "top-16, X %s [%dx7168]%s, grouped by expert%s" %
            (name, E, E * EXPERT_BYTES / 1e9, E, "bf16" if bf16 else "fp32", T,
             ", selection bias ~N(0,1)" if use_bias else "",
             "; activations and h quantised to MXFP4 (OCP rule), E2M1 x E2M1 block-scaled MMAs" if mxq else ""))
    gu_kernel = MXQ_GATEUP_KERNEL if mxq else GROUPED_GATEUP_KERNEL
    line = {
        "metric": "MoE-layer tokens/s (%d tokens per step, 896 experts, top-16, MXFP4%s)" %
                  (T, " weights and activations" if mxq else ""),
        "value": round(job_rate(steps * T, world, statistics.median(ms)), 2), "unit": "tokens/s",
        "steps": steps, "ms_per_step": round(per, 6), "higher_is_better": True,
        "dtype": "mxfp4 weights (e2m1 + e8m0), %s activations, fp32 accumulation" % ("bf16" if bf16 else "fp32"),
        "config": {"workload": desc, "global_batch": T * world, "seq_len": 1,
                   "launch": ("cuda graphs of %d steps (%d offsets) + %d, replayed" %
                              (plan["chunk"], plan["variants"], plan["rem"])) if use_graph
                   else "host launch per step",
                   "l2": "inputs larger than L2: %d token batches, %d router copies, %.0f distinct "
                         "experts (%.2f GB) per batch" % (NB, n_r, Umean, w_bytes / 1e9)},
        "timing": spread(ms, steps),
        "roofline": _roofline(gu_kernel + " (gate/up + SwiGLU over the batch's experts; the timed span "
                              "also holds grouping, tile plan and token preparation)",
                              gu_bytes, statistics.mean(gu_ms)),
        "step_bytes": {"distinct_experts": Umean, "bytes": int(step_bytes),
                       "gbs": round(step_bytes / (per * 1e-3) / 1e9, 1),
                       "frac_of_peak": round(step_bytes / (per * 1e-3) / 1e9 / measured_peaks()[0], 4)},
        "tflops": round(flops / (per * 1e-3) / 1e12, 2),
        "kernels_ms": {"route_topk": round(statistics.mean(r_ms), 4),
                       "group_gate_up_swiglu": round(statistics.mean(gu_ms), 4),
                       "down_combine": round(statistics.mean(dn_ms), 4)},
        "e2e": e2e, "gpu_launches": (MXQ_LAUNCHES if mxq else GROUPED_LAUNCHES) * steps, "clocks": clocks}
    if mxq:
        # block-scaled FP4 products: the FP4 peak from the measured bf16 one
        # and the nominal ratio; at this batch the weights' bytes cap it
        bf, bsrc = measured_bf16_tflops()
        fp4 = bf * FP4_PER_BF16
        ach = flops / (per * 1e-3) / 1e12
        cap = (flops / step_bytes) * measured_peaks()[0] * 1e9 / 1e12  # TFLOP/s at the HBM roofline
        line["mxfp4"] = {"tflops": round(ach, 1), "peak_tflops": round(fp4, 1),
                         "peak_source": "%s bf16 burst x %.0f (nominal FP4:bf16)" % (bsrc, FP4_PER_BF16),
                         "frac_of_peak": round(ach / fp4, 4), "flop_per_byte": round(flops / step_bytes, 1),
                         "hbm_bound_cap_tflops": round(cap, 1), "hbm_bound_cap_frac": round(cap / fp4, 4),
                         "frac_of_cap": round(ach / cap, 4)}
    for l in layers:
        l.close()
    return line


def _mem_available():
    try:
        with open("/proc/meminfo") as fh:
            for ln in fh:
                if ln.startswith("MemAvailable:"):
                    return int(ln.split()[1]) * 1024
    except OSError:
        pass
    return 0


def stream_launches(hits):
    """Kernels k3moe_stream_decode launches for a hit trace [T, layers, k]:
    per token and layer RMSNorm and the router, one gate/up + down pair over
    the hits (when there are any) and one pair per miss."""
    hits = np.asarray(hits).astype(bool)
    nh = hits.sum(axis=-1)
    nm = hits.shape[-1] - nh
    return int((2 + 2 * (nh > 0) + 2 * nm).sum())


def _stream_policy(k, cache, slots, n_w, n_tok, n_layers, hits, plain_lru):
    """Offline replays of the recorded trace (warm-up + timed tokens): the
    live hit flags reproduced by the LRU replay (plain LRU runs only), LRU
    against Belady's optimum at this cache's size, and a sizing sweep."""
    keys, bl = cache.trace()
    timed = slice(keys.size - hits.size, keys.size)
    out = {"trace_keys": int(keys.size), "timed_keys": int(hits.size)}
    if plain_lru:
        _, flags = k.trace_replay(keys, bl, slots, "lru")
        out["lru_replay_reproduces_live"] = bool(np.array_equal(flags[timed], hits.reshape(-1)))
    _, bel = k.trace_replay(keys, bl, slots, "belady")
    out["belady_hit_rate_timed"] = round(float(bel[timed].mean()), 4)
    caps = [16 * n_layers, 128, 256, slots, 2 * slots, 4 * slots, E * n_layers]
    lru = k.trace_sweep(keys, bl, caps, "lru")
    best = k.trace_sweep(keys, bl, caps, "belady")
    out["sizing"] = {"slots": caps, "lru_hit_rate": [round(int(h) / keys.size, 4) for h in lru],
                     "belady_hit_rate": [round(int(h) / keys.size, 4) for h in best],
                     "note": "whole recorded trace from an empty cache"}
    # the pinned hot set sized offline: hot keys of the first half's
    # histogram, hit rate on the second half, per number pinned
    half = keys.size // 2
    hot = k.hot_set(np.bincount(keys[:half], minlength=E * n_layers).astype(np.uint32), slots)
    counts = [0, slots // 4, slots // 2, 3 * slots // 4, slots - 16]
    pin = k.trace_pin_sweep(keys, bl, slots, hot, counts, count_from=half)
    out["pin_sweep"] = {"pinned": counts,
                        "hit_rate_second_half": [round(int(h) / (keys.size - half), 4) if h >= 0 else None
                                                 for h in pin],
                        "note": "hot set from the first half's request histogram, LRU in the other slots"}
    return out


def run_stream(args, rank, world, dev_index, n_layers=4, cache_bytes=8_000_000_000, n_tok=256):
    """Host-streamed pool: n_layers x 896 experts in pinned host memory, an
    HBM LRU cache of `cache_bytes`, batch-1 tokens through all layers with
    RMSNorm + residual (k3moe_stream_decode)."""
    import torch
    import synth
    from mxfp4_routed_expert_select_gb300 import k3moe as k
    dev = torch.device("cuda", dev_index)
    torch.cuda.set_device(dev)
    eb = k.expert_bytes(D, F)
    need = n_layers * E * eb
    if _mem_available() < need + 32 * (1 << 30):
        raise SystemExit("stream workload needs %.1f GB of host memory (+32 GB headroom); %.1f GB "
                         "available" % (need / 1e9, _mem_available() / 1e9))
    t0 = time.time()
    host = torch.empty((n_layers * E, eb), dtype=torch.uint8, pin_memory=True)
    for l in range(n_layers):
        for e in range(E):
            views = k.host_plane_views(host[l * E + e].data_ptr(), D, F)
            ex = synth.expert(2, l, e, D, F)
            for nm, arr in views.items():
                arr[...] = ex[nm]
    log("host pool: %d x %d experts (%.2f GB) in %.1f s" % (n_layers, E, need / 1e9, time.time() - t0))
    layers = []
    for l in range(n_layers):
        Wr = torch.from_numpy(synth.router_bf16(2, l, E, D).view(np.int16)).to(dev)
        b = torch.from_numpy(synth.bias_zipf(2, l, E).astype(np.float32)).to(dev)
        layers.append(k.Layer(E, K, D, F, Wr, None, b, max_tokens=1))
        layers[-1]._hold = (Wr, b)
    base = host.data_ptr()
    cache = k.Cache(cache_bytes, eb, [base + q * eb for q in range(n_layers * E)], n_layers, E)
    n_w = max(args.warmup, 3)
    n_h = 256 if args.pin_hot > 0 else 0  # history tokens before the hot set is pinned
    X = torch.from_numpy(synth.tokens_f32(2, n_h + n_w + n_tok + 64, D, t0=rank * 100000)).to(dev)
    out = torch.empty_like(X)
    # the host link, measured in this run: pinned host -> HBM copies of one expert
    probe = torch.empty(eb, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream()
    # every blob of the pool crosses the host link once before timing (as a
    # serving process warms its pool): the first copy engine access to a host
    # page is much slower than the later ones on some boxes
    t_w = time.time()
    for q in range(n_layers * E):
        probe.copy_(host[q], non_blocking=True)
    torch.cuda.synchronize()
    log("host pool warmed in %.1f s" % (time.time() - t_w))
    rates = []
    for rep in range(3):  # the same 16 experts three times; the best pass counts
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        p0.record(s)
        for q in range(16):
            probe.copy_(host[(q * 37) % (n_layers * E)], non_blocking=True)
        p1.record(s)
        torch.cuda.synchronize()
        rates.append(16 * eb / (p0.elapsed_time(p1) * 1e-3) / 1e9)
    h2d_gbs = max(rates)
    del probe
    if n_h:
        k.stream_decode(layers, cache, X[:n_h], n_h, out[:n_h], 1e-6, want_trace=False)
        k.check(cache.pin_hot(args.pin_hot), "k3moe_cache_pin_hot")
        X, out = X[n_h:], out[n_h:]
    cache.record_trace(True)
    k.stream_decode(layers, cache, X[:n_w], n_w, out[:n_w], 1e-6, want_trace=False)
    st0 = cache.stats()
    clock = ClockSampler(dev_index)
    clock.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(s)
    ids, hits = k.stream_decode(layers, cache, X[n_w:n_w + n_tok], n_tok, out[n_w:n_w + n_tok], 1e-6)
    e1.record(s)
    torch.cuda.synchronize()
    wall = time.perf_counter() - w0
    clocks = clock.stop()
    ms = e0.elapsed_time(e1)
    st1 = cache.stats()
    policy = _stream_policy(k, cache, st1["slots"], n_w, n_tok, n_layers, hits, args.pin_hot == 0)
    look = st1["lookups"] - st0["lookups"]
    nh = st1["hits"] - st0["hits"]
    h2d = st1["h2d_bytes"] - st0["h2d_bytes"]
    hbm = st1["hbm_bytes"] - st0["hbm_bytes"]
    peak, src = measured_peaks()
    ideal_s = (look * eb) / (peak * 1e9) + h2d / (h2d_gbs * 1e9)
    # e2e: tokens from pinned host memory, the result read back, per token
    xh = torch.empty((64, D), dtype=torch.float32, pin_memory=True)
    xh.copy_(X[n_w + n_tok:].cpu())
    oh = torch.empty((64, D), dtype=torch.float32, pin_memory=True)
    xd = torch.empty(D, dtype=torch.float32, device=dev)
    od = torch.empty(D, dtype=torch.float32, device=dev)

    def step_host(i):
        xd.copy_(xh[i % 64], non_blocking=True)
        k.stream_decode(layers, cache, xd, 1, od, 1e-6, want_trace=False)
        oh[i % 64].copy_(od, non_blocking=True)

    e2e = _e2e(step_host, 32, 3, world, dev_index, D * 4, D * 4, 1, "tokens/s")
    args.steps = n_tok
    line = _base_line("host-streamed MoE decode tokens/s (4 layers x 896 experts in pinned host "
                      "memory, 8 GB HBM LRU cache)", round(n_tok * world / (ms * 1e-3), 3), "tokens/s",
                      world, args, ms / n_tok,
                      "mxfp4 weights (e2m1 + e8m0), fp32 activations and accumulation",
                      {"workload": "stream_decode_b1: %d layers x 896 experts d=7168 f=1536 (%.2f GB) "
                                   "in pinned host memory, HBM LRU cache %.1f GB (%d slots), %d tokens, "
                                   "RMSNorm + residual, Zipf(1.1) selection bias" %
                                   (n_layers, need / 1e9, cache_bytes / 1e9, st1["slots"], n_tok),
                       "global_batch": world, "seq_len": 1,
                       "launch": "host loop in the library (rmsnorm, route, ids to host, split cache "
                                 "acquire, hit experts while the misses copy, each miss "
                                 "as its copy lands, release)",
                       "l2": "inputs larger than L2 (expert slots 17.5 MB each, 64 per token)",
                       "host_pool": "every blob copied to HBM once before timing (pool warmed)",
                       "warmup_tokens": n_w,
                       "policy": ("LRU with the %d most requested experts of %d history tokens "
                                  "pinned" % (args.pin_hot, n_h)) if n_h else "LRU"}, clocks)
    line.update({
        "cache": {"lookups": look, "hits": nh, "hit_rate": round(nh / max(look, 1), 4),
                  "h2d_bytes": h2d, "hbm_expert_bytes": hbm,
                  "h2d_bytes_per_token": round(h2d / n_tok), "hbm_bytes_per_token": round(hbm / n_tok),
                  "slots": st1["slots"]},
        "host_link_gbs": round(h2d_gbs, 1), "host_link_probe_passes_gbs": [round(r, 1) for r in rates],
        "h2d_achieved_gbs": round(h2d / (ms * 1e-3) / 1e9, 1),
        "roofline": {"kernel": "whole step (expert bytes from HBM + misses over the host link)",
                     "bound": "hbm+host-link", "achieved": round(ideal_s / (ms * 1e-3), 4),
                     "peak": 1.0, "peak_source": "ideal time = hits and misses at %s HBM %.0f GB/s and "
                     "measured host link %.1f GB/s" % (src, peak, h2d_gbs), "unit": "ideal/measured",
                     "frac": round(ideal_s / (ms * 1e-3), 4), "traffic": None},
        "wall_s": round(wall, 3), "e2e": e2e, "gpu_launches": stream_launches(hits),
        "cache_policy": policy})
    cache.close()
    for l in layers:
        l.close()
    return line


POOL_WORKLOADS = {
    "expert": lambda a, c, r, w: run_expert(a, c, r, w),
    "decode64": lambda a, c, r, w: run_batched(a, c, r, w, 64, False, False),
    "prefill4096": lambda a, c, r, w: run_batched(a, c, r, w, 4096, True, True),
    "prefill4096_mxq": lambda a, c, r, w: run_batched(a, c, r, w, 4096, True, True, mxq=True),
    "shared": lambda a, c, r, w: run_shared(a, c, r, w),
}
WORKLOADS = dict(POOL_WORKLOADS, stream=None)


def _set_timing(min_repeats, seconds):
    global MIN_REPEATS, REGION_SECONDS
    MIN_REPEATS = max(1, int(min_repeats))
    REGION_SECONDS = max(0.0, float(seconds))


def as_line(sub, args, world):
    """A secondary configuration's object as a JSON line of its own."""
    line = {"metric": sub["metric"], "value": sub["value"], "unit": sub["unit"], "n_gpus": world,
            "steps": sub["steps"], "warmup": args.warmup, "ms_per_step": sub["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": sub.get("dtype", "mxfp4 weights (e2m1 + e8m0), fp32 activations and accumulation"),
            "data": DATA}
    line.update({k_: v for k_, v in sub.items() if k_ not in line})
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="headline only: leave out the secondary configurations")
    ap.add_argument("--no-graph", action="store_true", help="launch every step from the host")
    ap.add_argument("--workload", default="decode1", choices=["decode1"] + sorted(WORKLOADS))
    ap.add_argument("--pin-hot", type=int, default=0,
                    help="stream workload: run 256 untimed history tokens, then pin the N most "
                         "requested experts of the cache's histogram before timing")
    ap.add_argument("--min-repeats", type=int, default=MIN_REPEATS,
                    help="timed regions per measurement at least (profiler captures: 1)")
    ap.add_argument("--region-seconds", type=float, default=REGION_SECONDS,
                    help="about how long the repeats of one measurement last (profiler captures: 0)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens per step of the decode64 / prefill workloads (profiler captures)")
    ap.add_argument("--experts", type=int, default=896,
                    help="experts per layer (smaller pools for profiler captures; 896 is the workload)")
    args = ap.parse_args()
    global E, ROUTER_BYTES, LAYER_BYTES
    _set_timing(args.min_repeats, args.region_seconds)
    E = args.experts
    ROUTER_BYTES = E * D * 2
    LAYER_BYTES = K * EXPERT_BYTES + ROUTER_BYTES
    if args.warmup < 3:
        args.warmup = 3
    args.steps = max(1, args.steps)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    import torch
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
        __graft_entry__.build()
    if args.workload == "stream":
        res = run_stream(args, rank, world, local)
    else:
        ctx = Ctx(local)
        if args.workload != "decode1":
            res = as_line(POOL_WORKLOADS[args.workload](args, ctx, rank, world), args, world)
        else:
            res = run_decode1(args, ctx, rank, world)
            if not args.no_configs:
                res["configs"] = {name: fn(args, ctx, rank, world) for name, fn in POOL_WORKLOADS.items()}
            if rank == 0 and not args.no_cpu_baseline:
                n, t, cores = cpu_baseline_sample()
                res["cpu_baseline"] = {"value": round(n / t, 4), "unit": "tokens/s", "cores": cores,
                                       "kind": "oracle",
                                       "sample": "%d tokens of the same layer (router + top-16 + 16 experts + "
                                                 "combine, fp64, OpenMP over all host cores) in %.1f s" % (n, t)}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
