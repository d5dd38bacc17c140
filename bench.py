#!/usr/bin/env python3
"""Benchmark of the exact width-k verify pass on GB300.

Workload: the synthetic 12-layer hybrid verify stack at hidden 2560 - every
layer a Gated DeltaNet mixer (16 QK / 48 V heads, head dim 128, per-row state
snapshots) followed by a MoE of 512 experts (top-10 routed + 1 sigmoid-gated
shared, intermediate 640), all projections affine Q4/group-64 with random
weights.  One step = one verify pass of k draft rows through all 12 layers
(every row of the hot path: dense Q4 products, routing, routed experts with
fused gate/up + SwiGLU + combine, GDN conv/norm/gates/delta rule/gated norm
with snapshots, layer norms and residual adds).  Accepting a prefix
(gdn_commit) is an O(1) host pointer swap without device work; it runs in
the end-to-end loop.

Metric: verified rows/s per layer = k * layers / step time, and the achieved
HBM bandwidth of the dominant call (the routed-expert call) against the
measured copy bandwidth.  The step's weight reads (~3 GB at k = 9) exceed the
129 MB L2 many times, so no flush is needed between steps.

Multi-GPU: the verify pass does not shard (see DESIGN); with --gpus N every
rank runs an independent replica and `value` sums the replicas.

--impl reference times the CPU oracle (test infrastructure) on one layer of
the same workload per step, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = ("12-layer hybrid verify stack, hidden 2560: GDN 16 QK/48 V heads d128 + MoE 512 experts "
            "top-10 + shared, I 640, affine Q4/g64 weights (synthetic, seed 0)")
EXPERT_BYTES = lambda H, I: int((2 * I * H + H * I) * 0.5625)  # noqa: E731


# DRAM traffic of the routed-expert kernel, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum) of both layers of a 2-layer
# stack at k = 9: 412.20 MB read and 6.01 MB written over two launches whose
# algorithmic bytes sum to 2 x 206226468.  Expert traffic grows with the
# distinct experts read, like the algorithmic bytes, so a full launch's
# traffic is this ratio times its bytes.  The figure holds only for the
# kernel sources it was taken on; any change to them reports null until the
# kernel is captured again.
MOE_TRAFFIC_RATIO = 418.21e6 / (2 * 206226468.0)
MOE_TRAFFIC_SOURCES = {
    "q4_kernels.cu": "a94468e049b2fbd81dd3166390c0df9f1db161b0dbc8452b3257527cd279805e",
    "common.cuh": "3152f57d8b02c0851d797f946658401567ffcc928311abd7bf76f26a90568479",
    "internal.h": "696848aff2ec6ff05f190ffe0d7e8dcbbeb1b1fc9cfeb8b2064a4bb5a8586494",
}


def moe_traffic(bytes_per_launch):
    """DRAM bytes per routed-expert launch, or None once the kernel changed."""
    import hashlib

    csrc = os.path.join(ROOT, "speculative_decode_verification_gb300", "csrc")
    for name, digest in MOE_TRAFFIC_SOURCES.items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != digest:
                return None
    return MOE_TRAFFIC_RATIO * bytes_per_launch


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device, self.proc, self.lines = device, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.device)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
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


# ------------------------------------------------------------------ oracle

def oracle_layer_step(cfg, k, seed=0, layer=0, weights=None):
    """One layer of the stack on the CPU oracle; returns (seconds, weights)."""
    from oracle import oracle as O
    from speculative_decode_verification_gb300 import synth as S
    from speculative_decode_verification_gb300.stack import shapes

    sh = shapes(cfg)
    if weights is None:
        weights = S.HostLayerWeights(seed, layer, sh["H"], sh["NP"], sh["Z"], sh["E"], sh["I"], cfg["n_qk_heads"],
                                     cfg["n_v_heads"], cfg["d"])
    S0, t0 = S.gdn_initial_state(seed, f"stack.L{layer}.gdn", cfg["n_qk_heads"], cfg["n_v_heads"], cfg["d"],
                                 s_std=0.02, tail_std=1.0)
    h0 = S.f32_normal(seed, f"bench.h{k}", (k, sh["H"])).astype(np.float64)
    # draw the experts this step routes to before the clock starts (input generation)
    t = time.perf_counter()
    O.stack_layer(weights, h0, S0.astype(np.float64), t0, k, cfg["n_qk_heads"], cfg["n_v_heads"], cfg["d"], sh["T"])
    return time.perf_counter() - t, weights


def host_cpu():
    """The host CPU's model and logical core count, read at run time."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    import platform

    return f"{model or platform.processor() or platform.machine()} ({os.cpu_count()} logical cores)"


def oracle_mode(threaded):
    """Selects the oracle build (OpenMP over all host cores, or the plain
    single-threaded one); returns the threads it uses (None: no OpenMP build)."""
    from oracle import oracle as O
    O.build()
    if threaded and O.build_threaded() is None:
        return None
    return O.use_threads(threaded)


def cpu_baseline(cfg, k, runs=5):
    """One full-shape layer at width k on the oracle, both modes: the median of
    `runs` timed runs after one warm-up (which also draws the layer's weights
    and routed experts, untimed)."""
    _, w = oracle_layer_step(cfg, k)
    out = {}
    for threaded in (False, True):
        n = oracle_mode(threaded)
        if n is None:
            continue
        oracle_layer_step(cfg, k, weights=w)
        ts = [oracle_layer_step(cfg, k, weights=w)[0] for _ in range(runs)]
        out[threaded] = (n, float(np.median(ts)))
    oracle_mode(False)
    n1, t1 = out[False]
    single = {"value": k / t1, "unit": "verified rows/s per layer", "cores": 1, "ms_per_layer": t1 * 1e3}
    nt, tt = out.get(True, out[False])
    return {"value": k / tt, "unit": "verified rows/s per layer", "cores": nt, "kind": "oracle",
            "sample": f"one of the {cfg['layers']} layers at k={k} (full shapes), float64 C oracle "
                      f"({'OpenMP over output rows, ' + str(nt) + ' threads' if True in out else 'single thread'}), "
                      f"median of {runs} runs after one warm-up, {tt * 1e3:.0f} ms per layer",
            "statistic": f"median of {runs}", "host": host_cpu(), "single_thread": single}


def run_reference(args, cfg):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    k = args.k
    _, w = oracle_layer_step(cfg, k)    # draws the weights and routed experts (untimed)
    nt = oracle_mode(True) or oracle_mode(False)
    for _ in range(args.warmup):
        oracle_layer_step(cfg, k, weights=w)
    ts = [oracle_layer_step(cfg, k, weights=w)[0] for _ in range(args.steps)]
    step = float(np.median(ts))
    value = k / step
    sample = (f"one full-shape layer at k={k} per step, float64 C oracle on {nt} host threads "
              f"(OpenMP over output rows), median of {args.steps} steps")
    line = {"metric": "verified rows/s per layer", "value": value, "unit": "verified rows/s per layer",
            "impl": "reference", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step * 1e3, "ms_per_step_mean": float(np.mean(ts)) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "k": k, "layers_per_step": 1,
                       "note": "CPU oracle, one layer per step (bounded sample)"},
            "cpu_baseline": {"value": value, "unit": "verified rows/s per layer", "cores": nt, "kind": "oracle",
                             "sample": sample, "host": host_cpu()},
            "e2e": {"value": value, "unit": "verified rows/s per layer", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ ours

def time_steps(graph, stream, steps):
    """Mean ms per replay of `graph` over `steps` back-to-back replays, from
    CUDA events recorded on the replay stream (synchronised on both sides)."""
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(steps):
            graph.replay()
        e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_ours(args, cfg):
    import torch

    from speculative_decode_verification_gb300 import binding as B
    from speculative_decode_verification_gb300 import synth as S
    from speculative_decode_verification_gb300.stack import DeviceStack, shapes

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (GB300)")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    vf = B.Verify(local)
    sh = shapes(cfg)
    L, H, T = cfg["layers"], sh["H"], sh["T"]
    ds = DeviceStack(vf, cfg, seed=0, n_slots=max(10, max(int(w) for w in args.widths.split(',') if w) + 1, args.k + 1),
                     vocab=S.FLASH_VOCAB)
    stream = torch.cuda.Stream()
    widths = sorted(set([int(w) for w in args.widths.split(",") if w] + [args.k]))
    hbm, peak_kind = peaks()
    per_k, head, timed = {}, None, {}
    for k in widths:  # set-up and untimed measurements per width; the timed trials follow
        h0 = torch.from_numpy(S.f32_normal(0, f"bench.h{k}", (k, H))).cuda()
        h = torch.empty_like(h0)
        idx_all = torch.zeros((L, k, T), dtype=torch.int32, device="cuda")
        idx = [idx_all[l] for l in range(L)]
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(L)]
        with torch.cuda.stream(stream):
            for row in ev:
                for e in row:
                    e.record()
        torch.cuda.synchronize()
        for st in ds.states:
            st.cur, st.pending_k = 0, 0
        def capture(events_for_layer):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                for st in ds.states:
                    st.cur, st.pending_k = 0, 0
                with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
                    h.copy_(h0)
                    if events_for_layer is None:  # the public one-call pass
                        vf.verify_stack_k(ds.layers, ds.states, h, k, idx_all, stream.cuda_stream)
                    else:
                        for l, (Ly, st) in enumerate(zip(ds.layers, ds.states)):
                            vf.set_layer_events(events_for_layer(l))
                            vf.verify_layer_k(Ly, st, h, k, idx[l], stream.cuda_stream)
                        vf.set_layer_events(None)
            return graph

        for st in ds.states:
            st.cur, st.pending_k = 0, 0
        with torch.cuda.stream(stream):
            h.copy_(h0)
            lc0 = vf.launch_count()
            ds.verify(h, k, idx, stream.cuda_stream)          # warm (first launches, first touch)
            n_launch = vf.launch_count() - lc0                # our kernels in one verify pass (eager)
            if k == args.k:
                launches_per_pass = n_launch
        torch.cuda.synchronize()
        # breakdown graph: every sub-step boundary of every layer (untimed)
        gb = capture(lambda l: ev[l])
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(3):
                gb.replay()
        torch.cuda.synchronize()
        names = ["norm1", "in_proj", "gdn", "out_proj", "norm2", "router", "experts"]
        sub = {n: float(np.mean([ev[l][i].elapsed_time(ev[l][i + 1]) * 1e3 for l in range(L)]))
               for i, n in enumerate(names)}
        del gb
        # timed graph: the verify step alone, one verify_stack_k call (an event
        # between two kernels stops the second from overlapping the first, so
        # the step carries none)
        g = capture(None)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                g.replay()
        torch.cuda.synchronize()
        timed[k] = g
        # per-step spread: an event after each of up to 200 replays (a graph
        # boundary already orders them)
        n_pct = max(3, min(args.steps, 200))
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_pct + 1)]
        with torch.cuda.stream(stream):
            evs[0].record()
            for i in range(n_pct):
                g.replay()
                evs[i + 1].record()
        torch.cuda.synchronize()
        step_ms = np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(n_pct)])
        # the routed-expert call's own duration: a second graph of the same step
        # with events around that call in every layer (durations averaged over
        # layers and replays)
        evm = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(L)]
        with torch.cuda.stream(stream):
            for row in evm:
                for e in row:
                    e.record()
        torch.cuda.synchronize()
        gm = capture(lambda l: [None] * 6 + evm[l])
        torch.cuda.synchronize()
        moe_samples = []
        for _ in range(max(3, min(args.steps // 10, 50))):
            with torch.cuda.stream(stream):
                gm.replay()
            stream.synchronize()
            moe_samples += [evm[l][0].elapsed_time(evm[l][1]) * 1e3 for l in range(L)]
        del gm
        moe_timed_us = float(np.mean(moe_samples))
        U = [len(np.unique(idx[l].cpu().numpy())) for l in range(L)]
        moe_bytes = [(u + 1) * EXPERT_BYTES(H, sh["I"]) + k * H * (2 + 8) + k * (sh["E"] + 1) * 4 for u in U]
        dense_bytes = int(0.5625 * (sh["NP"] * H + H * sh["Z"] + (sh["E"] + 1) * H))
        gdn_bytes = cfg["n_v_heads"] * cfg["d"] ** 2 * 4 * (1 + k) + 3 * sh["C"] * 2 * (1 + k)
        step_bytes = sum(moe_bytes) + L * (dense_bytes + gdn_bytes)
        per_k[k] = {"ms_per_step_p10_p50_p90": [round(float(np.percentile(step_ms, q)), 4) for q in (10, 50, 90)],
                    "layer_us": {n: round(v, 2) for n, v in sub.items()},
                    "distinct_experts_per_layer": float(np.mean(U)),
                    "step_bytes": step_bytes}
        per_k[k]["experts_us_timed"] = moe_timed_us
        if k == args.k:
            moe_us = moe_timed_us
            achieved = float(np.mean(moe_bytes)) / (moe_us * 1e-6) / 1e9
            head = dict(U=float(np.mean(U)), moe_us=moe_us, moe_bytes=float(np.mean(moe_bytes)), achieved=achieved)
    # The timed trials, back to back with the clock sampler running: the
    # widths ascending, descending, then ascending again (the pages' protocol
    # reverses the order on the second trial).  Each trial of a width is W
    # warm-up replays and exactly `steps` timed replays; the headline keeps
    # trial 1, and each width also reports its three trials and their median.
    sampler = ClockSampler(local)
    sampler.start()
    t_w = time.perf_counter()  # nvidia-smi needs a moment to start: keep the GPU busy meanwhile (untimed)
    with torch.cuda.stream(stream):
        while time.perf_counter() - t_w < 0.6:
            timed[widths[0]].replay()
            stream.synchronize()
    for order in (widths, widths[::-1], widths):
        for k in order:
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    timed[k].replay()
            torch.cuda.synchronize()
            barrier(world)
            per_k[k].setdefault("ms_per_step_trials", []).append(
                max_over_ranks(time_steps(timed[k], stream, args.steps), world))
    clocks = sampler.stop()
    for k in widths:
        tr = per_k[k]["ms_per_step_trials"]
        ms, ms3 = tr[0], float(np.median(tr))
        per_k[k].update({"rows_per_s_per_layer": k * L / (ms * 1e-3) * world, "ms_per_step": ms,
                         "step_GBs": per_k[k]["step_bytes"] / (ms * 1e-3) / 1e9, "ms_per_step_median3": ms3,
                         "rows_per_s_per_layer_median3": k * L / (ms3 * 1e-3) * world})
    head["ms"] = per_k[args.k]["ms_per_step"]
    head["clocks"] = clocks
    st, code = vf.device_status()
    if st != B.OK:
        raise SystemExit(f"device error {code} during the benchmark")
    del timed
    # ---- end to end through the public API: host buffers, copies inside the timed region
    k = args.k
    hh = torch.from_numpy(S.f32_normal(0, f"bench.h{k}", (k, H))).pin_memory()
    hout = torch.empty_like(hh).pin_memory()
    hd = torch.empty((k, H), dtype=torch.float32, device="cuda")
    for st in ds.states:
        st.cur, st.pending_k = 0, 0
    accepted = k // 2

    def e2e_step():
        with torch.cuda.stream(stream):
            hd.copy_(hh, non_blocking=True)
            ds.verify(hd, k, None, stream.cuda_stream)
            hout.copy_(hd, non_blocking=True)
        stream.synchronize()
        ds.commit(accepted)

    for _ in range(args.warmup):
        e2e_step()
    barrier(world)
    n_e2e = max(3, min(args.steps, 200))
    # each step timed on its own (host clock; the step ends with a stream
    # synchronize): the median is robust to a rare host stall, the mean is kept
    e2e_t = []
    for _ in range(n_e2e):
        t0 = time.perf_counter()
        e2e_step()
        e2e_t.append(time.perf_counter() - t0)
    launches_per_step = launches_per_pass  # the timed steps replay graphs of the same kernels
    e2e_s = max_over_ranks(float(np.median(e2e_t)), world)
    e2e_mean_s = max_over_ranks(float(np.mean(e2e_t)), world)
    loop = device_loop(args, ds, vf, stream, k, H, world)
    if rank != 0:
        return 0
    cpu = None if args.no_cpu_baseline else cpu_baseline(cfg, k)
    value = per_k[k]["rows_per_s_per_layer"]
    line = {
        "metric": "verified rows/s per layer", "value": value, "unit": "verified rows/s per layer",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "k": k, "layers": L, "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (weights read per step far above 129 MB); no flush",
                   "per_k": {str(kk): v for kk, v in per_k.items()}},
        "roofline": {"bound": "hbm", "achieved": head["achieved"], "peak": hbm, "unit": "GB/s",
                     "frac": head["achieved"] / hbm, "traffic": moe_traffic(head["moe_bytes"]),
                     "traffic_unit": "DRAM bytes per launch (ncu read + write of a 2-layer capture, scaled)",
                     "kernel": "q4_gather_experts_k (routing kernel, fused routed gate/up+SwiGLU and down kernel, combine kernel)",
                     "bytes_per_launch": head["moe_bytes"], "us_per_launch": head["moe_us"],
                     "distinct_experts": head["U"], "peak_kind": peak_kind},
        "clocks": head["clocks"],
        "e2e": {"value": k * L / e2e_s * world, "unit": "verified rows/s per layer",
                "h2d_bytes_per_step": k * H * 4, "d2h_bytes_per_step": k * H * 4,
                "ms_per_step": e2e_s * 1e3, "ms_per_step_mean": e2e_mean_s * 1e3, "steps": n_e2e,
                "statistic": "median of per-step host times",
                "path": "DeviceStack.verify (one CUDA graph replay of verify_stack_k per state configuration)"},
        "gpu_launches": launches_per_step * args.steps,
        "cpu_baseline": cpu,
        "device_loop": loop,
    }
    print(json.dumps(line), flush=True)
    return 0


def device_loop(args, ds, vf, stream, k, H, world):
    """Decode steps with acceptance and commit on the device: per step the
    host copies the k input rows in, one graph replay runs the verify pass and
    verify_accept_greedy (greedy choice over a 248,320-entry vocabulary,
    accepted prefix, commit of every layer's state), and the host reads back
    the result (accepted rows, next token, the k choices).  The target logits
    are synthetic and fixed: N(0, 1) with one planted winner per row (logit
    100 at a seeded token), and the drafts follow the winners up to row
    k // 2, so k // 2 + 1 rows stand every step and the next token is known by
    construction.  The LM head that would produce the logits is not part of
    the pass.  Reported beside the headline, not in it."""
    import torch

    from speculative_decode_verification_gb300 import synth as S

    V = S.FLASH_VOCAB
    x = S.vocab_logits(0, f"bench.loop.logits{k}", k, V, 0)
    t = (S.uniform_f32(S.tensor_seed(0, f"bench.loop.winners{k}"), k, 0.0, 1.0) * V).astype(np.int64) % V
    x[np.arange(k), t] = 100.0
    m = min(k // 2, k - 1)
    draft = t[: k - 1].astype(np.int32)
    if m < k - 1:
        draft[m] = (t[m] + 1) % V
    a_want, next_want = m + 1, int(t[m])
    logits = torch.from_numpy(x).cuda()
    dd = torch.from_numpy(np.concatenate([draft, [0]]).astype(np.int32)).cuda()
    res = torch.zeros(2 + k, dtype=torch.int32, device="cuda")
    hh = torch.from_numpy(S.f32_normal(0, f"bench.h{k}", (k, H))).pin_memory()
    rout = torch.empty(2 + k, dtype=torch.int32).pin_memory()
    hd = torch.empty((k, H), dtype=torch.float32, device="cuda")
    for st in ds.states:
        st.cur, st.pending_k = 0, 0
    ds.to_device()

    def step():
        with torch.cuda.stream(stream):
            hd.copy_(hh, non_blocking=True)
            ds.verify_accept(hd, k, logits, dd, res, stream.cuda_stream)
            rout.copy_(res, non_blocking=True)
        stream.synchronize()

    for _ in range(args.warmup):
        step()
    barrier(world)
    ts = []
    for _ in range(max(3, min(args.steps, 200))):
        t0 = time.perf_counter()
        step()
        ts.append(time.perf_counter() - t0)
        if int(rout[0]) != a_want or int(rout[1]) != next_want:
            raise SystemExit(f"device acceptance gave {rout[:2].tolist()}, expected {[a_want, next_want]}")
    # device-timed replays of the same graph (input rows refreshed on the device each step)
    h0 = hd.clone()
    n_dev = max(3, min(args.steps, 500))

    def device_ms(run):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record()
            for _ in range(n_dev):
                hd.copy_(h0)
                run()
            e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n_dev

    dev_ms = device_ms(lambda: ds.verify_accept(hd, k, logits, dd, res, stream.cuda_stream))
    # the same loop with the target head in the graph: final norm, the Q4 LM
    # head over the full vocabulary (357.6 MB of weights), acceptance, commit
    sel = None
    if ds.vocab:
        def step_sel():
            with torch.cuda.stream(stream):
                hd.copy_(hh, non_blocking=True)
                ds.verify_select_accept(hd, k, dd, res, stream.cuda_stream)
                rout.copy_(res, non_blocking=True)
            stream.synchronize()

        for _ in range(args.warmup):
            step_sel()
        ts_sel, acc = [], []
        for _ in range(max(3, min(args.steps, 200))):
            t0 = time.perf_counter()
            step_sel()
            ts_sel.append(time.perf_counter() - t0)
            acc.append(int(rout[0]))
        sel_dev = device_ms(lambda: ds.verify_select_accept(hd, k, dd, res, stream.cuda_stream))
        unf_dev = device_ms(lambda: ds.verify_select_accept(hd, k, dd, res, stream.cuda_stream, fused=False))
        sel_s = max_over_ranks(float(np.median(ts_sel)), world)
        sel = {"ms_per_step": sel_s * 1e3, "device_ms_per_step": max_over_ranks(sel_dev, world),
               "device_ms_per_step_unfused": max_over_ranks(unf_dev, world),
               "lm_head_bytes": int(0.5625 * V * H), "accepted_rows_mean": float(np.mean(acc)),
               "path": "DeviceStack.verify_select_accept: verify_stack_k + final norm + verify_lm_head_accept "
                       "(the LM head with its argmax epilogue, acceptance and commit) in one graph; unfused: "
                       "q4_qmv_k logits then verify_accept_greedy"}
    ds.to_host()
    st, code = vf.device_status()
    if st != 0:
        raise SystemExit(f"device error {code} in the device loop")
    host_s = max_over_ranks(float(np.median(ts)), world)
    dev_ms = max_over_ranks(dev_ms, world)
    L = ds.n_layers
    return {"k": k, "V": V, "accepted_rows": a_want, "steps": len(ts),
            "ms_per_step": host_s * 1e3, "verified_rows_per_s_per_layer": k * L / host_s * world,
            "device_ms_per_step": dev_ms,
            "h2d_bytes_per_step": k * H * 4, "d2h_bytes_per_step": (2 + k) * 4,
            "statistic": "median of per-step host times; device time from CUDA events over back-to-back replays",
            "path": "DeviceStack.verify_accept: one graph replay of verify_stack_k + verify_accept_greedy "
                    "(device-held commits)",
            "with_lm_head": sel}


def run_kernels(args):
    """Each hot-path kernel alone on its own configuration.  A timed batch is
    one replay of a CUDA graph of R back-to-back calls between two CUDA events
    on the launching stream, rotating over enough weight copies or input sets
    that a batch touches more than 3 x L2, so no call finds its inputs in L2;
    per-call time = batch time / R, median of --steps batches after --warmup.  One JSON line per
    (kernel, config, k), then a summary line.  Not the bench contract line: a
    per-kernel roofline table."""
    import torch
    from speculative_decode_verification_gb300 import binding as B
    from speculative_decode_verification_gb300 import synth as S

    vf = B.Verify(0)
    hbm, peak_kind = peaks()
    stream = torch.cuda.Stream()
    L2 = 129 << 20
    keep = []

    def q4(name, n_out, k_in, n_experts=None, gate_up=False, down=False):
        e = 1 if n_experts is None else n_experts
        shp = (e, n_out, k_in // 8) if n_experts else (n_out, k_in // 8)
        gshp = (e, n_out, k_in // 64) if n_experts else (n_out, k_in // 64)
        p = torch.empty(shp, dtype=torch.int32, device="cuda")
        sc = torch.empty(gshp, dtype=torch.int16, device="cuda")
        bi = torch.empty(gshp, dtype=torch.int16, device="cuda")
        vf.synth_q4(p, sc, bi, S.q4_seeds(0, name), S.SCALE_RANGE, S.BIAS_RANGE, centered=False)
        rows = B.q4_experts(p, sc, bi) if n_experts else B.q4_weight(p, sc, bi)
        t = vf.tile(rows, gate_up=gate_up, down=down)
        torch.cuda.synchronize()
        del p, sc, bi
        keep.append(t.buf)
        return t.struct

    def dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
        keep.append(t)
        return t

    def time_calls(calls, R=40):
        """calls: the rotation set (callables).  One CUDA graph holds R >= len(calls)
        back-to-back calls cycling through the set (no host work between the
        kernels); per-call time = replay time / R, median over replays."""
        R = max(R, len(calls))
        with torch.cuda.stream(stream):
            for c in calls:  # first launches outside the capture
                c()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(R):
                calls[i % len(calls)]()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for it in range(args.warmup + args.steps):
            with torch.cuda.stream(stream):
                e0.record()
                g.replay()
                e1.record()
            e1.synchronize()
            if it >= args.warmup:
                ts.append(e0.elapsed_time(e1) * 1e3 / R)
        del g
        return float(np.median(ts))

    lines = []

    def emit(kernel, config, k, us, nbytes, extra=None):
        d = {"kernel": kernel, "config": config, "k": k, "us": round(us, 3), "bytes": int(nbytes),
             "GBs": round(nbytes / us / 1e3, 1), "frac": round(nbytes / us / 1e3 / hbm, 4), "peak": hbm,
             "peak_kind": peak_kind}
        if extra:
            d.update(extra)
        lines.append(d)
        print(json.dumps(d), flush=True)

    widths = [int(w) for w in args.widths.split(",") if w]
    kmax = max(widths)
    only = set(args.only.split(",")) if args.only else None

    def want(name):
        return only is None or name in only

    # the tiny configuration: one 512 x 512 projection at k = 1..4 and a
    # 2/2-head, d = 32 GDN step at k = 2.  Its 147 KB of weights are rotated
    # over 8 copies and stay in L2: these rows measure latency, not bandwidth.
    if want("tiny"):
        N = K = 512
        Ws = [q4(f"kbench.tiny.c{c}", N, K) for c in range(8)]
        x = dev(S.bf16_normal(0, "kbench.tiny.x", (4, K)).view(np.int16))
        y = torch.empty((4, N), dtype=torch.float32, device="cuda")
        for k in (1, 2, 3, 4):
            us = time_calls([(lambda W=W, k=k: vf.q4_qmv_k(W, x, k, y, B.F32, stream.cuda_stream)) for W in Ws])
            emit("q4_qmv_k", f"tiny {N}x{K}", k, us, 0.5625 * N * K + 2 * k * K + 4 * k * N, {"l2_resident": True})
        Hk, Hv, d, k = 2, 2, 32, 2
        C = 2 * Hk * d + Hv * d
        gp = {key: dev(v) for key, v in S.gdn_params(0, "kbench.tiny.gdn", Hk, Hv, d).items()}
        params = B.gdn_params(Hk, Hv, d, gp["conv_w"], gp["A_log"], gp["dt_bias"], gp["norm_w"])
        calls = []
        for r in range(8):
            slots = [torch.zeros((Hv, d, d), dtype=torch.float32, device="cuda") for _ in range(k + 1)]
            tails = [torch.zeros((3, C), dtype=torch.int16, device="cuda") for _ in range(k + 1)]
            inp = {key: dev(v.view(np.int16) if v.dtype == np.uint16 else v)
                   for key, v in S.gdn_inputs(0, f"kbench.tiny.gdn.{r}", k, Hk, Hv, d).items()}
            o = torch.empty((k, Hv * d), dtype=torch.float32, device="cuda")
            keep.extend(slots + tails + [o])
            gi = B.gdn_inputs(inp["qkv"], inp["z"], inp["a"], inp["b"])
            calls.append(lambda slots=slots, tails=tails, gi=gi, o=o:
                         vf.gdn_verify_k(params, B.gdn_state(slots, tails, cur=0), gi, k, o, B.F32, stream.cuda_stream))
        us = time_calls(calls)
        emit("gdn_verify_k", f"tiny gdn Hk{Hk} Hv{Hv} d{d}", k, us,
             Hv * d * d * 4 * (1 + k) + 3 * C * 2 * (1 + k) + k * (C + Hv * d + 2 * Hv) * 2 + k * Hv * d * 4,
             {"l2_resident": True})
        del Ws
        keep.clear()
        torch.cuda.empty_cache()
    # a1: dense Q4 products, the dense configuration's shapes and the LM head; copies rotated
    for (N, K) in [sh for sh in S.DENSE_SHAPES if want("dense")] + ([S.LM_HEAD] if want("lm_head") else []):
        wbytes = 0.5625 * N * K
        n_copies = int(np.ceil(3 * L2 / wbytes)) + 1
        Ws = [q4(f"kbench.dense.{N}x{K}.c{c}", N, K) for c in range(n_copies)]
        x = dev(S.bf16_normal(0, f"kbench.x.{K}", (kmax, K)).view(np.int16))
        y = torch.empty((kmax, N), dtype=torch.float32, device="cuda")
        t1 = None
        for k in widths:
            us = time_calls([(lambda W=W, k=k: vf.q4_qmv_k(W, x, k, y, B.F32, stream.cuda_stream)) for W in Ws])
            t1 = us if k == 1 else t1
            emit("q4_qmv_k", f"dense {N}x{K}" + (" (LM head)" if (N, K) == S.LM_HEAD else ""), k, us,
                 wbytes + 2 * k * K + 4 * k * N,
                 {"t_over_t1": round(us / t1, 3) if t1 else None, "copies": n_copies})
        del Ws
        keep.clear()
        torch.cuda.empty_cache()
    # a2-a4: routed experts, the Ornith-shaped configuration (no shared expert);
    # the expert weights (453 MB) exceed 3 x L2; 8 input sets rotated
    m = S.ORNITH_MOE
    E, T, H, I = m["E"], m["T"], m["H"], m["I"]
    gu = q4("kbench.moe.gu", 2 * I, H, E, gate_up=True) if want("experts") else None
    dn = q4("kbench.moe.dn", H, I, E, down=True) if want("experts") else None
    for k in (widths if want("experts") else []):
        sets = []
        for r in range(8):
            logits = dev(S.f32_normal(0, f"kbench.moe.l{k}.{r}", (k, E)))
            x = dev(S.bf16_normal(0, f"kbench.moe.x{k}.{r}", (k, H)).view(np.int16))
            idx = torch.zeros((k, T), dtype=torch.int32, device="cuda")
            w = torch.zeros((k, T), dtype=torch.float32, device="cuda")
            y = torch.zeros((k, H), dtype=torch.float32, device="cuda")
            keep.extend([idx, w, y])
            sets.append((logits, x, idx, w, y))
        us = time_calls([(lambda st=st, k=k: vf.q4_gather_experts_k(gu, dn, st[0], E, T, st[1], k, st[2], st[3], st[4],
                                                                     B.F32, stream=stream.cuda_stream))
                         for st in sets])
        U = float(np.mean([np.unique(st[2].cpu().numpy()).size for st in sets]))
        emit("q4_gather_experts_k", f"experts E{E} T{T} H{H} I{I}", k, us,
             U * 3 * H * I * 0.5625 + k * H * (2 + 4) + k * E * 4, {"distinct_experts": U})
    del gu, dn
    keep.clear()
    torch.cuda.empty_cache()
    # a5-a7: the GDN verify step, the Flash-Next-shaped configuration; 8 state
    # rings and input sets rotated
    g = S.FLASH_GDN
    Hk, Hv, d = g["n_qk_heads"], g["n_v_heads"], g["d"]
    C = 2 * Hk * d + Hv * d
    gp = {key: dev(v) for key, v in S.gdn_params(0, "kbench.gdn", Hk, Hv, d).items()}
    params = B.gdn_params(Hk, Hv, d, gp["conv_w"], gp["A_log"], gp["dt_bias"], gp["norm_w"])
    S0, t0 = S.gdn_initial_state(0, "kbench.gdn", Hk, Hv, d, s_std=0.02, tail_std=1.0)
    rings = []
    for r in range(8 if want("gdn") else 0):
        slots = [dev(S0) if s == 0 else torch.zeros((Hv, d, d), dtype=torch.float32, device="cuda")
                 for s in range(kmax + 1)]
        tails = [dev(t0.view(np.int16)) if s == 0 else torch.zeros((3, C), dtype=torch.int16, device="cuda")
                 for s in range(kmax + 1)]
        keep.extend(slots + tails)
        rings.append((slots, tails))
    for k in (widths if want("gdn") else []):
        calls = []
        for r, (slots, tails) in enumerate(rings):
            inp = {key: dev(v.view(np.int16) if v.dtype == np.uint16 else v)
                   for key, v in S.gdn_inputs(0, f"kbench.gdn.{k}.{r}", k, Hk, Hv, d).items()}
            o = torch.empty((k, Hv * d), dtype=torch.float32, device="cuda")
            keep.append(o)
            gi = B.gdn_inputs(inp["qkv"], inp["z"], inp["a"], inp["b"])

            def call(slots=slots, tails=tails, gi=gi, o=o, k=k):
                vf.gdn_verify_k(params, B.gdn_state(slots, tails, cur=0), gi, k, o, B.F32, stream.cuda_stream)

            calls.append(call)
        us = time_calls(calls)
        nbytes = Hv * d * d * 4 * (1 + k) + 3 * C * 2 * (1 + k) + k * (C + Hv * d + 2 * Hv) * 2 + k * Hv * d * 4
        emit("gdn_verify_k", f"gdn Hk{Hk} Hv{Hv} d{d}", k, us, nbytes)
    del rings
    keep.clear()
    torch.cuda.empty_cache()
    # next row: greedy acceptance over the Flash-Next vocabulary (no states to
    # commit); logits sets rotated over > 3 x L2
    V = S.FLASH_VOCAB
    for k in (widths if want("accept") else []):
        n_sets = int(np.ceil(3 * L2 / (k * V * 4))) + 1
        base = torch.from_numpy(S.vocab_logits(0, f"kbench.accept.{k}", k, V, 0)).cuda()
        sets = []
        for r in range(n_sets):
            lg = base.roll(r, dims=1).contiguous()  # same values, other positions
            res = torch.zeros(2 + k, dtype=torch.int32, device="cuda")
            sets.append((lg, res))
        dft = torch.zeros(max(k - 1, 1), dtype=torch.int32, device="cuda")
        us = time_calls([(lambda st=st, k=k: vf.accept_greedy(st[0], k, dft, st[1], stream=stream.cuda_stream))
                         for st in sets])
        emit("verify_accept_greedy", f"accept V{V}", k, us, k * V * 4 + 4 * (k - 1) + 4 * (k + 2),
             {"sets": n_sets})
        del sets, base
        torch.cuda.empty_cache()
    # next row: width-k attention verify at the Flash-Next attention shape over
    # caches of 4,096 and 65,536 positions; caches rotated over > 3 x L2
    ac = S.FLASH_ATTN
    Hq, Hkv, D = ac["n_q_heads"], ac["n_kv_heads"], ac["d"]
    params = B.attn_params(Hq, Hkv, D, ac["rope_dim"], ac["theta"])
    gen = torch.Generator(device="cuda")
    gen.manual_seed(0)
    attn_ps = [int(x) for x in args.attn_p.split(",") if x]
    for P in (attn_ps if want("attn") else ()):
        cap = P + kmax
        cache_bytes = 2 * Hkv * cap * D * 2
        n_c = int(np.ceil(3 * L2 / cache_bytes)) + 1
        split = B.attn_default_split(cap)
        nb = B.attn_workspace_bytes(params, cap, split, kmax)
        caches = []
        for _ in range(n_c):
            Kc = torch.randn((Hkv, cap, D), generator=gen, device="cuda").half().view(torch.int16)
            Vc = torch.randn((Hkv, cap, D), generator=gen, device="cuda").half().view(torch.int16)
            wk = torch.empty(nb, dtype=torch.uint8, device="cuda")
            caches.append((Kc, Vc, wk))
        for k in widths:
            ins = {n: dev(S.bf16_normal(0, f"kbench.attn.{n}{k}", (k, (Hq if n in "qg" else Hkv) * D)).view(np.int16))
                   for n in ("q", "g", "k", "v")}
            ai = B.attn_inputs(ins["q"], ins["g"], ins["k"], ins["v"])
            o = torch.empty((k, Hq * D), dtype=torch.float32, device="cuda")
            calls = []
            for (Kc, Vc, wk) in caches:
                kc = B.kv_cache(Kc, Vc, wk, P, split)
                keep.append(kc)
                calls.append(lambda kc=kc, k=k: vf.attn_verify_k(params, kc, ai, k, o, B.F32, stream.cuda_stream))
            us = time_calls(calls)
            flops = sum(4.0 * Hq * D * (P + r + 1) for r in range(k))
            emit("attn_verify_k", f"attn Hq{Hq} Hkv{Hkv} D{D} P{P}", k, us,
                 2 * Hkv * (P + k) * D * 2 + k * (2 * Hq * D * 2 + 2 * Hkv * D * 2 + Hq * D * 4),
                 {"tflops": round(flops / us / 1e6, 2), "caches": n_c, "split": split})
        del caches
        torch.cuda.empty_cache()
    print(json.dumps({"summary": "per-kernel roofline: back-to-back calls, weights or inputs rotated over > 3 x L2",
                      "n": len(lines), "peak": hbm, "peak_kind": peak_kind}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--k", type=int, default=9, help="verify width of the headline number")
    ap.add_argument("--widths", default="1,4,8,9,16,32", help="widths also measured (reported under config.per_k)")
    ap.add_argument("--layers", type=int, default=12)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="",
                    help="with --kernels: comma list of tiny,dense,lm_head,experts,gdn,accept,attn (default all)")
    ap.add_argument("--attn-p", default="4096,65536",
                    help="with --kernels: cached positions of the attention rows (comma list)")
    ap.add_argument("--kernels", action="store_true",
                    help="time each hot-path kernel alone on its own configuration instead (JSON line per kernel)")
    args = ap.parse_args()
    from speculative_decode_verification_gb300 import synth as S
    cfg = dict(S.STACK)
    cfg["layers"] = args.layers
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.kernels:
        return run_kernels(args)
    return run_ours(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
