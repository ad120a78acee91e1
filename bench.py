"""Benchmark of the MXFP4 routed-expert MoE layer on one GB300 (or N ranks).

Default workload: one MoE layer, batch-1 decode -- 896 experts of
d=7168, f=1536 resident in HBM (15.7 GB), router W_r bf16 [896 x 7168],
x fp32, top-16, softmax combine over the selected logits.  A step is one
token through the whole layer (router + top-k + 16 experts + combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  `value` is tokens/s of the whole job (every
rank runs independent tokens: weak scaling, no collective on the data path).
Extra workloads for development: --workload expert|decode64|prefill4096.
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
N_TOKENS = 1024


def log(*a):
    print(*a, file=sys.stderr, flush=True)


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


# ------------------------------------------------------------------ arms

def run_ours(args, rank, world, dev_index):
    import torch
    import synth
    from mxfp4_routed_expert_select_gb300 import k3moe as k
    dev = torch.device("cuda", dev_index)
    torch.cuda.set_device(dev)
    blobs, views = build_pool(dev)
    Wr_bits = synth.router_bf16(1, 0, E, D)
    Wr0 = torch.from_numpy(Wr_bits.view(np.int16)).to(dev)
    routers = [Wr0] + [Wr0.clone() for _ in range(N_ROUTER_COPIES - 1)]
    layers = [k.Layer(E, K, D, F, r, views, max_tokens=1) for r in routers]
    X = torch.from_numpy(np.stack([synth.token_f32(1, rank * N_TOKENS + t, D)
                                   for t in range(N_TOKENS)])).to(dev)
    out = torch.empty(D, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream()

    def step(i):
        layers[i % N_ROUTER_COPIES].forward(X[i % N_TOKENS], 1, out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # The timed steps replay a CUDA graph holding G_STEPS consecutive layer
    # forwards (different tokens and router copies), as a decode loop would:
    # no host launch overhead inside the step.
    G_STEPS = 32
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(G_STEPS):
                step(i)
        graph.replay()
        torch.cuda.synchronize()

    # per-kernel events on the launching stream for the first steps of the
    # timed region
    n_ev = min(args.steps, 2000)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_ev)]
    for quad in evs:  # torch creates the CUDA event at its first record
        for e in quad:
            e.record(s)
    clock = ClockSampler(dev_index)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clock.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if graph is not None:
        s = torch.cuda.current_stream()
        n_rep = (args.steps + G_STEPS - 1) // G_STEPS
        args.steps = n_rep * G_STEPS
        t_start.record(s)
        for _ in range(n_rep):
            graph.replay()
        t_end.record(s)
    else:
        t_start.record(s)
        for i in range(args.steps):
            L = layers[i % N_ROUTER_COPIES]
            if i < n_ev:
                L.set_events(evs[i])
            elif i == n_ev:
                for l in layers:
                    l.set_events(None)
            step(i)
        t_end.record(s)
    torch.cuda.synchronize()
    clocks = clock.stop()
    for l in layers:
        l.set_events(None)
    if world > 1:
        torch.distributed.barrier()
    ms = t_start.elapsed_time(t_end)
    if world > 1:
        tt = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms = float(tt.item())
    if graph is not None:
        # the fused kernel's own duration, events on its stream around each launch
        for i in range(n_ev):
            L = layers[i % N_ROUTER_COPIES]
            L.set_events(evs[i])
            step(i)
        for l in layers:
            l.set_events(None)
        torch.cuda.synchronize()
    route_ms = [e[0].elapsed_time(e[1]) for e in evs]
    gu_ms = [e[1].elapsed_time(e[2]) for e in evs]
    dn_ms = [e[2].elapsed_time(e[3]) for e in evs]

    fused = layers[0].fused_t1()
    # the opt-in f16-activation mode, same workload, for the record
    act16 = None
    if fused:
        for l in layers:
            l.set_option(k.K3MOE_OPT_ACT_F16, 1)
        for i in range(args.warmup):
            step(i)
        torch.cuda.synchronize()
        g16 = None
        if not args.no_graph:
            g16 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g16):
                for i in range(G_STEPS):
                    step(i)
            g16.replay()
            torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(s)
        if g16 is not None:
            for _ in range(args.steps // G_STEPS):
                g16.replay()
        else:
            for i in range(args.steps):
                step(i)
        a1.record(s)
        torch.cuda.synchronize()
        ams = a0.elapsed_time(a1) / (args.steps if g16 is None else (args.steps // G_STEPS) * G_STEPS)
        for l in layers:
            l.set_option(k.K3MOE_OPT_ACT_F16, 0)
        act16 = {"value": round(world * 1e3 / ams, 2), "unit": "tokens/s", "ms_per_step": round(ams, 5),
                 "layer_gbs": round(LAYER_BYTES / (ams * 1e-3) / 1e9, 1),
                 "note": "K3MOE_OPT_ACT_F16: activations rounded to f16 (16-element power-of-two blocks), "
                         "fp32 accumulation; not the headline"}

    # e2e through the C ABI with host buffers: H2D of the token, the layer,
    # D2H of the output, every step
    n_e2e = min(args.steps, 5000)
    xh = torch.empty((N_TOKENS, D), dtype=torch.float32, pin_memory=True)
    xh.copy_(X.cpu())
    oh = torch.empty(D, dtype=torch.float32, pin_memory=True)
    xd = torch.empty(D, dtype=torch.float32, device=dev)
    for i in range(args.warmup):
        xd.copy_(xh[i % N_TOKENS], non_blocking=True)
        layers[i % N_ROUTER_COPIES].forward(xd, 1, out)
        oh.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    e0.record(s)
    for i in range(n_e2e):
        xd.copy_(xh[i % N_TOKENS], non_blocking=True)
        layers[i % N_ROUTER_COPIES].forward(xd, 1, out)
        oh.copy_(out, non_blocking=True)
    e1.record(s)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    if world > 1:
        tt = torch.tensor([e2e_ms], device=dev)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(tt.item())

    peak, peak_src = measured_peaks()
    gu_avg = statistics.mean(gu_ms)
    if fused:
        # one kernel per step: its average duration over the timed region is at
        # most the step time (graph replay gaps count against it)
        eager_ms = statistics.mean([a + b + c for a, b, c in zip(route_ms, gu_ms, dn_ms)])
        k_ms = ms / args.steps if graph is not None else eager_ms
        k_name, k_bytes = "k3_moe_t1_fused (router + top-k + 16 experts + combine)", LAYER_BYTES
    else:
        k_ms, k_name, k_bytes = gu_avg, "k3_rows_pipe (gate/up + SwiGLU, 16 experts)", GATEUP_BYTES
    achieved = k_bytes / (k_ms * 1e-3) / 1e9
    layer_gbs = LAYER_BYTES / (ms / args.steps * 1e-3) / 1e9
    result = {
        "metric": "MoE-layer decode tokens/s (batch 1, 896 experts, top-16, MXFP4)",
        "value": round(args.steps * world / (ms * 1e-3), 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4 weights (e2m1 + e8m0), fp32 activations and accumulation",
        "data": "synthetic (seeded SplitMix64: uniform E2M1 codes, E8M0 in [120,130], x ~ N(0,1), W_r ~ N(0,0.02) bf16)",
        "config": {"workload": "moe_layer_decode_b1: 896 experts d=7168 f=1536 resident (15.7 GB), "
                               "router bf16 [896x7168], top-16, softmax combine",
                   "global_batch": world, "seq_len": 1, "parallelism": "replicas" if world > 1 else "single",
                   "launch": "cuda graph of 32 steps, replayed" if graph is not None else "host launch per step",
                   "l2": "inputs larger than L2: %d rotated router copies (%.0f MB) + 896 experts "
                         "(16 random per token, 281 MB/token) + %d distinct tokens"
                         % (N_ROUTER_COPIES, N_ROUTER_COPIES * ROUTER_BYTES / 1e6, N_TOKENS)},
        "layer_hbm": {"bytes_per_token": LAYER_BYTES, "gbs": round(layer_gbs, 1),
                      "frac_of_peak": round(layer_gbs / peak, 4), "frac_of_8tbs": round(layer_gbs / 8000, 4)},
        "kernels_ms": ({"fused_layer": round(k_ms, 5), "fused_layer_eager_events": round(eager_ms, 5),
                        "steps_sampled": n_ev} if fused else
                       {"route_topk": round(statistics.mean(route_ms), 5),
                        "gate_up_swiglu": round(gu_avg, 5),
                        "down_combine": round(statistics.mean(dn_ms), 5), "steps_sampled": n_ev}),
        "roofline": {"kernel": k_name, "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "algorithmic_bytes": k_bytes},
        "e2e": {"value": round(n_e2e * world / (e2e_ms * 1e-3), 2), "unit": "tokens/s",
                "h2d_bytes_per_step": D * 4, "d2h_bytes_per_step": D * 4, "steps": n_e2e},
        "gpu_launches": (1 if fused else 3) * args.steps,
        "act_f16_mode": act16,
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch every step from the host")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
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
    res = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            n, t, cores = cpu_baseline_sample()
            res["cpu_baseline"] = {"value": round(n / t, 4), "unit": "tokens/s", "cores": cores,
                                   "kind": "oracle",
                                   "sample": "%d tokens of the same layer (router + top-16 + 16 experts + "
                                             "combine, fp64) in %.1f s" % (n, t)}
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
