#!/usr/bin/env python3
"""Benchmark: closed-form tree verify + commit of one GDN layer on a GB300.

One step is one pass of the whole hot path over one batch: tree prep, the
S0 contraction, the masked decayed A/C build, the triangular solve and the
output (one verify call), then the commit of a root-to-leaf accepted path.
Default workload: batched verify, B=16 streams, H=16 heads, dk=dv=128,
T=64-node uniform random trees with depth 4..20, bf16 q/k/v, fp32 S0, fp32
o (synthetic, seeded).  Metric: verified nodes/s (B*T per step) and us per
layer verify.

  python bench.py [--gpus N --steps K --warmup W] [--impl canopy|reference]
  python bench.py --sweep          # crossover map vs the serial replay kernel

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and a
device synchronise on both sides, CUDA events on the launching stream, max
over ranks.  The timed steps are captured once as a CUDA graph of
consecutive steps over the rotating sets and replayed, so the host's per-call
marshalling does not starve the GPU; per-kernel durations come from graphs of
the same launches of one kernel alone.  Inputs rotate over enough independent sets that the data one
step touches is not in L2 (129 MB) when the step starts.  Clocks are sampled
with nvidia-smi during the timed region.  Under torchrun each rank runs the
same per-GPU workload (replicas: the units are independent, no collective in
the data path).
"""

from __future__ import annotations

import argparse
import json
import os
import shutil
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

WORKLOAD = dict(name="batched verify B=16 T=64 H=16 dk=dv=128 random trees depth 4-20 bf16 q/k/v fp32 S0",
                case=2, B=16, T=64, H=16, d=128)
METRIC = "µs per GDN layer tree-verify and verified nodes/s (B=16,T=64); % HBM roofline"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0     # GB300 HBM3e, nominal (context beside the measured copy peak)
# DRAM bytes of one verify launch of the default workload from an ncu capture
# of the current kernel (dram__bytes_read.sum, dram__bytes_write.sum); set to
# None whenever the kernel changes, until it is captured again.  The writes
# (o and U, 16.8 MB) are still in L2 when the launch ends and reach DRAM
# during later launches, so the capture's write figure is far below them.
VERIFY_DRAM_TRAFFIC = {"read": 29_562_368, "write": 100_864}


def verify_bytes(B, T, H, d, in_bytes=2, o_bytes=4):
    """Algorithmic bytes of one verify call: S0, q/k/v, g, beta and parent read;
    o, U, l, depth and the ancestor mask written."""
    W = (T + 31) // 32
    return (B * H * d * d * 4 + B * T * H * d * in_bytes * 3 + B * T * H * 4 * 2 + B * T * 4
            + B * T * H * d * o_bytes + B * T * H * d * 4 + B * T * H * 4 + B * T * 4 + B * T * W * 4)


def commit_bytes(B, T, H, d):
    """S0 read and S_new written (the path's k rows, u entries and gates are
    negligible and not counted)."""
    return 2 * B * H * d * d * 4


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.out = os.path.join("/tmp", f"canopy_clocks_{os.getpid()}.csv")

    def start(self):
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        self.f = open(self.out, "w")
        self.proc = subprocess.Popen([exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                      "-i", str(self.gpu), "-lms", "100"], stdout=self.f,
                                     stderr=subprocess.DEVNULL)
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.out):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        os.remove(self.out)
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "power_w_max": max(r["power"] for r in rows), "samples": len(rows), "reasons": sorted(reasons)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# the CUDA path

def make_sets(nsets, rank, wl, bf16=True):
    import torch

    import synth
    from gated_deltanet_linear_tree_gb300 import canopy
    from synth import trees
    sets = []
    B, T, H, d = wl["B"], wl["T"], wl["H"], wl["d"]
    for s in range(nsets):
        inp = synth.config_inputs(wl["case"], rnd=1000 * rank + s, B=B, T=T, H=H, dk=d, dv=d)
        dev = {}
        for n in ("q", "k", "v"):
            dev[n] = torch.from_numpy(inp[n]).to("cuda", torch.bfloat16 if bf16 else torch.float32)
        for n in ("g", "beta", "S0"):
            dev[n] = torch.from_numpy(inp[n]).cuda()
        dev["parent"] = torch.from_numpy(inp["parent"]).cuda()
        rng = np.random.default_rng(s)
        acc = np.array([rng.choice(trees.leaves(inp["parent"][b])) for b in range(B)], dtype=np.int32)
        dev["acc"] = torch.from_numpy(acc).cuda()
        dev["ws"] = canopy.workspace(B, T, H, d)
        dev["o"] = torch.empty((B, T, H, d), dtype=torch.float32, device="cuda")
        dev["S_new"] = torch.empty_like(dev["S0"])
        dev["host"] = inp
        sets.append(dev)
    return sets


def step(canopy, s, T, solve="fwdsub"):
    canopy.verify(s["q"], s["k"], s["v"], s["g"], s["beta"], s["S0"], s["parent"], s["ws"], solve=solve,
                  out=s["o"])
    canopy.commit(s["acc"], s["S0"], s["k"], s["parent"], s["ws"], out=s["S_new"])


def capture_graph(canopy, sets, T, solve, n, kind):
    """One CUDA graph of n consecutive steps over the rotating input sets:
    kind "step" = verify + commit, "verify" or "commit" = that call alone.
    The host-side argument marshalling runs once, at capture."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            s = sets[i % len(sets)]
            if kind in ("step", "verify"):
                # the kernel before each verify in the graph (a commit or a
                # verify of another input set) never writes its inputs, S0
                # included (commits write S_new)
                canopy.verify(s["q"], s["k"], s["v"], s["g"], s["beta"], s["S0"], s["parent"], s["ws"], solve=solve,
                              out=s["o"], inputs_ready=True, state_ready=True)
            if kind in ("step", "commit"):
                # the kernel before each commit (its verify, or a commit of
                # another set) writes none of S0, the accepted nodes, k and
                # parent
                canopy.commit(s["acc"], s["S0"], s["k"], s["parent"], s["ws"], out=s["S_new"], state_ready=True)
    torch.cuda.synchronize()
    return g


def verify_after_producer(canopy, sets, solve, n, reps):
    """us per verify when the kernel before it is a plain HBM-bound kernel
    that writes the verify's q, k and v (a stand-in for the projection that
    produces them), with no overlap flags: graphs of n x (producer copies)
    and of n x (producer copies, verify), the difference per verify.  The
    verify can then start nothing before the copies complete."""
    import torch
    for s in sets:
        if "src" not in s:
            s["src"] = {c: s[c].clone() for c in ("q", "k", "v")}

    def graph(with_verify):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                s = sets[i % len(sets)]
                for c in ("q", "k", "v"):
                    s[c].copy_(s["src"][c])
                if with_verify:
                    canopy.verify(s["q"], s["k"], s["v"], s["g"], s["beta"], s["S0"], s["parent"], s["ws"],
                                  solve=solve, out=s["o"])
        torch.cuda.synchronize()
        return g

    gp, gpv = graph(False), graph(True)
    tp, tpv = [], []
    for _ in range(reps):
        for g, out in ((gp, tp), (gpv, tpv)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            out.append(a.elapsed_time(b))
    return 1e3 * (statistics.median(tpv) - statistics.median(tp)) / n, 1e3 * statistics.median(tp) / n


def run_canopy(args, world, rank, local):
    import torch

    from gated_deltanet_linear_tree_gb300 import build as bld
    from gated_deltanet_linear_tree_gb300 import canopy
    if rank == 0 or not os.path.exists(bld.LIB):
        bld.build()
    barrier(world)
    canopy.load()
    wl = WORKLOAD
    B, T, H, d = wl["B"], wl["T"], wl["H"], wl["d"]
    sets = make_sets(args.sets, rank, wl)
    for i in range(max(args.warmup, len(sets))):
        step(canopy, sets[i % len(sets)], T, args.solve)
    torch.cuda.synchronize()
    assert canopy.read_device_error(sets[0]["ws"]) == 0
    G = max(len(sets), (args.graph_steps // len(sets)) * len(sets))
    g_step = capture_graph(canopy, sets, T, args.solve, G, "step")
    g_ver = capture_graph(canopy, sets, T, args.solve, G, "verify")
    g_com = capture_graph(canopy, sets, T, args.solve, G, "commit")
    K = args.steps
    reps, rem = divmod(K, G)
    g_rem = capture_graph(canopy, sets, T, args.solve, rem, "step") if rem else None
    for _ in range(max(1, -(-args.warmup // G))):
        g_step.replay()
    if g_rem is not None:
        g_rem.replay()   # a graph's first replay uploads it: keep that out of the timed region
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g_step.replay()
    if g_rem is not None:
        g_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    total_ms = e0.elapsed_time(e1)
    # per-kernel launch durations: the same launches, one kernel kind per graph
    t_verify, t_commit = [], []
    for g, out in ((g_ver, t_verify), (g_com, t_commit)):
        for _ in range(args.kernel_reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            out.append(a.elapsed_time(b) / G)
    clk = clocks.stop()
    # warm: the same input set at every launch, so its 46 MB stay in the
    # 129 MB L2 (reported beside the cold, rotating figure)
    g_warm = capture_graph(canopy, sets[:1], T, args.solve, G, "verify")
    g_warm.replay()
    torch.cuda.synchronize()
    t_warm = []
    for _ in range(args.kernel_reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g_warm.replay()
        b.record()
        torch.cuda.synchronize()
        t_warm.append(a.elapsed_time(b) / G)
    total_ms = max_over_ranks(total_ms, world)
    vp_us, prod_us = verify_after_producer(canopy, sets, args.solve, G, args.kernel_reps)
    errs = [canopy.read_device_error(s["ws"]) for s in sets]
    assert not any(errs), errs

    ms_step = total_ms / K
    nodes = B * T * K * world
    value = nodes / (total_ms / 1e3)
    v_us = 1e3 * statistics.mean(t_verify)
    c_us = 1e3 * statistics.mean(t_commit)
    peak, peak_src = peaks()
    vb = verify_bytes(B, T, H, d)
    cb = commit_bytes(B, T, H, d)
    achieved = vb / (v_us * 1e-6) / 1e9
    # forward substitution: one launch at every T (the fused kernel up to 64
    # nodes, the blocked tensor-core kernel beyond); the Neumann series is
    # one launch up to 64 nodes; otherwise tree prep, the Gram and the solve
    # (two launches for split)
    one_launch = args.solve == "fwdsub" or (T <= 64 and args.solve == "neumann")
    launches_per_step = (1 if one_launch else (4 if args.solve == "split" else 3)) + 1
    kernel = {("fwdsub", True): "tcf::verify_fwd_kernel (fused, tcgen05)",
              ("fwdsub", False): "tcb::verify_big_kernel (blocked, tcgen05)",
              ("neumann", True): "tc::verify_neumann_kernel (fused, tcgen05)"}.get(
                  (args.solve, T <= 64), "tree prep + tensor-core Gram + CUDA-core solve variant")
    traffic = None
    if VERIFY_DRAM_TRAFFIC is not None and T == 64 and args.solve == "fwdsub":
        traffic = VERIFY_DRAM_TRAFFIC["read"] + VERIFY_DRAM_TRAFFIC["write"]

    e2e = run_e2e(canopy, sets, T, args, world)
    e2e_copied = run_e2e(canopy, sets, T, args, world, state_on_device=False)
    line = {
        "metric": METRIC, "value": value, "unit": "verified nodes/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, shapes and distributions of the pages' "
        "batched-verify case; no dataset or weights)",
        "config": bench_config(args, world),
        "us_per_layer_verify": v_us, "us_per_commit": c_us,
        "verify_p10_p50_p90_us": [1e3 * float(np.percentile(t_verify, p)) for p in (10, 50, 90)],
        "timing": f"one CUDA graph of {G} steps (verify + commit, sets rotating) replayed {reps} times "
                  f"(+ a graph of the {rem} remaining steps) between two events; per-kernel durations from graphs of {G} launches of one kernel, "
                  f"{args.kernel_reps} replays each (p10/p50/p90 over replays)",
        "roofline": {"bound": "hbm", "kernel": kernel,
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "frac_nominal": achieved / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS,
                     "traffic": traffic,
                     "traffic_note": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch; o and U "
                                     "are still in L2 when the launch ends, so its writes reach DRAM later"
                                     if traffic is not None else "no capture of the current kernel",
                     "algorithmic_bytes": vb, "peak_source": f"{peak_src} hbm_gbs",
                     "setting": "back to back over rotating input sets, overlap flags set (the preceding "
                                "kernel is a verify or commit of another set)"},
        "roofline_verify_after_producer": {
            "bound": "hbm", "us_per_launch": vp_us, "achieved": vb / (vp_us * 1e-6) / 1e9, "peak": peak,
            "unit": "GB/s", "frac": vb / (vp_us * 1e-6) / 1e9 / peak,
            "frac_nominal": vb / (vp_us * 1e-6) / 1e9 / NOMINAL_HBM_GBS,
            "setting": "each verify follows copy kernels that write its q, k and v (no overlap flags); "
                       f"time of (copies + verify) minus copies alone ({prod_us:.2f} us) per launch"},
        "verify_warm_l2": {"us_per_launch": 1e3 * statistics.mean(t_warm),
                           "algorithmic_GBps": vb / (1e3 * statistics.mean(t_warm) * 1e-6) / 1e9,
                           "setting": "the same input set at every launch (back to back, overlap flags set): "
                                      "its inputs and outputs stay in L2, so this is not an HBM figure"},
        "roofline_commit": {"bound": "hbm", "achieved": cb / (c_us * 1e-6) / 1e9, "peak": peak, "unit": "GB/s",
                            "frac": cb / (c_us * 1e-6) / 1e9 / peak,
                            "frac_nominal": cb / (c_us * 1e-6) / 1e9 / NOMINAL_HBM_GBS, "algorithmic_bytes": cb},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
        "e2e": e2e,
        "e2e_state_copied": e2e_copied,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sets[0]["host"], args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_config(args, world):
    """The workload's config record, the same for both arms."""
    wl = WORKLOAD
    return {"workload": wl["name"], "B": wl["B"], "T": wl["T"], "H": wl["H"], "dk": wl["d"], "dv": wl["d"],
            "o_dtype": "f32", "solve": args.solve, "step": "verify + commit of one accepted leaf per stream",
            "l2": f"inputs and outputs rotate over {args.sets} sets of about 88 MB each, more than the 129 MB L2 "
                  "in total",
            "parallelism": f"replicas x{world}"}


def run_e2e(canopy, sets, T, args, world, state_on_device=True):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory and reads its output o back.  With
    state_on_device (decoding as it runs: the recurrent state never leaves
    the GPU), the inputs are the round's q, k, v, g, beta, parent and accepted
    leaf, and each step verifies against the state and commits into it in
    place; otherwise S0 is copied in and S_new read back every step as well.
    A step's inputs travel as one packed host-to-device copy and its results
    as one packed device-to-host copy, each on a stream of its own, so that
    step i + 1's inputs and step i - 1's results move while step i computes
    (three device buffer sets in rotation; events order every reuse)."""
    import torch
    K = max(10, min(args.e2e_steps, args.steps))
    names = ("q", "k", "v", "g", "beta", "parent", "acc") + (() if state_on_device else ("S0",))
    outs = ("o",) + (() if state_on_device else ("S_new",))

    def packing(fields):
        lay, off = [], 0
        for n, t in fields:
            nb = t.numel() * t.element_size()
            lay.append((n, off, nb, t.dtype, tuple(t.shape)))
            off = (off + nb + 255) // 256 * 256
        return lay, off

    def views(buf, lay):
        return {n: buf[o:o + nb].view(dt).view(sh) for n, o, nb, dt, sh in lay}

    in_lay, in_size = packing([(n, sets[0][n]) for n in names])
    out_lay, out_size = packing([(n, sets[0][n]) for n in outs])
    h2d = sum(nb for _, _, nb, _, _ in in_lay)
    d2h = sum(nb for _, _, nb, _, _ in out_lay)
    host_in = []
    for s in sets[:2]:
        hb = torch.empty(in_size, dtype=torch.uint8).pin_memory()
        hv = views(hb, in_lay)
        for n in names:
            hv[n].copy_(s[n].cpu())
        host_in.append(hb)
    host_out = [torch.empty(out_size, dtype=torch.uint8).pin_memory() for _ in range(2)]
    dev_in = [torch.empty(in_size, dtype=torch.uint8, device="cuda") for _ in range(3)]
    dev_out = [torch.empty(out_size, dtype=torch.uint8, device="cuda") for _ in range(3)]
    din = [views(x, in_lay) for x in dev_in]
    dout = [views(x, out_lay) for x in dev_out]
    state = sets[0]["S0"].clone() if state_on_device else None
    ws = sets[0]["ws"]
    cur = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, computed, out_read = [ev() for _ in range(3)], [ev() for _ in range(3)], [ev() for _ in range(3)]
    for e in computed + out_read:
        e.record(cur)

    def one(i):
        j, hsel = i % 3, i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(computed[j])          # step i - 3 has finished with these inputs
            dev_in[j].copy_(host_in[hsel], non_blocking=True)
            in_ready[j].record(s_in)
        cur.wait_event(in_ready[j])
        cur.wait_event(out_read[j])               # step i - 3's results have left
        d, o = din[j], dout[j]
        S0 = state if state_on_device else d["S0"]
        S_new = state if state_on_device else o["S_new"]
        canopy.verify(d["q"], d["k"], d["v"], d["g"], d["beta"], S0, d["parent"], ws, solve=args.solve,
                      out=o["o"])
        canopy.commit(d["acc"], S0, d["k"], d["parent"], ws, out=S_new)
        computed[j].record(cur)
        with torch.cuda.stream(s_out):
            s_out.wait_event(computed[j])
            host_out[hsel].copy_(dev_out[j], non_blocking=True)
            out_read[j].record(s_out)

    for i in range(6):
        one(i)
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cur)
    s_in.wait_event(a)
    s_out.wait_event(a)
    for i in range(K):
        one(i)
    cur.wait_stream(s_out)
    b.record(cur)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world)
    assert canopy.read_device_error(ws) == 0
    B = sets[0]["parent"].shape[0]
    what = ("q, k, v, g, beta, parent and the accepted leaf in, o out; the recurrent state stays on the GPU and "
            "is committed in place" if state_on_device else
            "q, k, v, g, beta, parent, the accepted leaf and S0 in, o and S_new out")
    return {"value": B * T * K * world / (ms / 1e3), "unit": "verified nodes/s", "steps": K,
            "ms_per_step": ms / K, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": f"per step: {what}; one packed pinned host-to-device copy and one packed device-to-host "
                      "copy, on their own streams, overlapping the neighbouring steps' compute"}


def _oracle_streams(args):
    """Worker of the CPU baseline's process pool: the fp64 oracle replay of
    whole streams (one stream per task, every head of it at once)."""
    import oracle
    parent, q, k, v, g, beta, S0 = args
    oracle.replay(parent, q, k, v, g, beta, S0, keep_states=False)
    return parent.shape[0]


def cpu_baseline(inp, seconds, repeats=3):
    """The fp64 oracle as it stands, on a bounded sample of the workload: the
    first input set's streams, each replayed whole (all heads at once, NumPy
    einsum, no BLAS call), spread over a process pool of one worker per host
    core (spawned: the workers start no CUDA context).  The sample is sized
    so that one pass takes about seconds / repeats; the value is the median
    of `repeats` passes."""
    import multiprocessing as mp
    B = inp["parent"].shape[0]
    T = inp["parent"].shape[1]
    cores = os.cpu_count() or 1
    tasks = [tuple(inp[n][b] for n in ("parent", "q", "k", "v", "g", "beta", "S0")) for b in range(B)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        pool.map(_oracle_streams, tasks[:cores])            # start-up and imports, untimed
        t0 = time.perf_counter()
        pool.map(_oracle_streams, tasks)
        per_pass = time.perf_counter() - t0
        mult = max(1, int(round(seconds / repeats / max(per_pass, 1e-3))))
        rates = []
        for _ in range(repeats):
            t0 = time.perf_counter()
            n = sum(pool.map(_oracle_streams, tasks * mult))
            rates.append(n / (time.perf_counter() - t0))
    return {"value": statistics.median(rates), "unit": "verified nodes/s", "cores": cores, "host_cores": cores,
            "blas_threads": 0, "repeats": repeats, "kind": "oracle",
            "sample": f"{B * mult} whole streams per pass (T={T}, H={inp['q'].shape[2]}, dk=dv={inp['q'].shape[3]}) of the "
                      f"workload's first input set, fp64 NumPy replay, one stream per task over {cores} spawned "
                      f"worker processes; median of {repeats} passes (einsum: no BLAS threads)"}


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores

def run_reference(args, world, rank):
    """The oracle on the host cores: each step replays the first m nodes of
    one stream per host core (a bounded sample of the workload, every head
    at once), the streams spread over spawned worker processes; m is sized
    so that the whole run takes about two minutes."""
    if rank != 0:
        return
    import multiprocessing as mp

    import synth
    wl = WORKLOAD
    inp = synth.config_inputs(wl["case"], rnd=0)
    B, T = inp["parent"].shape
    cores = os.cpu_count() or 1
    names = ("parent", "q", "k", "v", "g", "beta", "S0")

    def tasks(i, m):
        out = []
        for c in range(cores):
            b = (i * cores + c) % B
            out.append(tuple(inp[n][b] if n == "S0" else inp[n][b][:m] for n in names))
        return out

    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        pool.map(_oracle_streams, tasks(0, 8))               # start-up and imports, untimed
        t0 = time.perf_counter()
        pool.map(_oracle_streams, tasks(0, 8))
        t_node = (time.perf_counter() - t0) / 8
        budget = 120.0 / max(1, args.steps + args.warmup)
        m = int(max(1, min(T, budget / max(t_node, 1e-6))))
        for i in range(args.warmup):
            pool.map(_oracle_streams, tasks(i, m))
        t0 = time.perf_counter()
        for i in range(args.steps):
            pool.map(_oracle_streams, tasks(i, m))
        dt = time.perf_counter() - t0
    value = cores * m * args.steps / dt
    sample = (f"first {m} nodes of {cores} streams' trees per step (one stream per spawned worker process; "
              f"H=16, dk=dv=128), fp64 NumPy replay")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "verified nodes/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": bench_config(args, world),
            "cpu_baseline": {"value": value, "unit": "verified nodes/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "verified nodes/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# tables (crossover map, dispatch table, solve strategies, layer shape): each
# output file opens with a record of the machine and closes with the clocks

def _smi(query):
    import subprocess
    try:
        r = subprocess.run(["nvidia-smi", f"--query-gpu={query}", "--format=csv,noheader"], capture_output=True,
                           text=True, timeout=20)
        return r.stdout.strip()
    except (OSError, subprocess.SubprocessError):
        return ""


def env_record(kind):
    import torch
    return {"env": {"table": kind, "gpu": torch.cuda.get_device_name(0), "torch": torch.__version__,
                    "cuda": torch.version.cuda, "driver": _smi("driver_version"),
                    "clocks_before": _smi("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active"),
                    "date_utc": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime())}}


class TableOut:
    """JSON lines to stdout and to --sweep-out (if given), between an
    environment record and a closing clocks record."""

    def __init__(self, args, kind):
        self.f = open(args.sweep_out, "w") if args.sweep_out else None
        self.write(env_record(kind))

    def write(self, rec):
        line = json.dumps(rec)
        print(line, flush=True)
        if self.f:
            self.f.write(line + "\n")

    def close(self):
        self.write({"env_end": {"clocks_after": _smi("clocks.sm,clocks.max.sm,power.draw,"
                                                     "clocks_event_reasons.active")}})
        if self.f:
            self.f.close()


def time_calls(calls, flush, warmup, reps):
    """Each call timed alone after an L2 flush (a 1 GiB fill, which also keeps
    the host ahead of the GPU), the calls interleaved; p10/p50/p90 in us."""
    import torch
    times = {k: [] for k in calls}
    for it in range(warmup + reps):
        for name, fn in calls.items():
            flush.fill_(float(it))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            if it >= warmup:
                times[name].append((a, b))
    torch.cuda.synchronize()
    out = {}
    for name, evs in times.items():
        us = [1e3 * a.elapsed_time(b) for a, b in evs]
        out[name] = {"p10": float(np.percentile(us, 10)), "p50": float(np.percentile(us, 50)),
                     "p90": float(np.percentile(us, 90))}
    return out


def run_dispatch_table(args):
    """Below the crossover: the closed form against the path replay (both
    forced), random trees of 1..8 nodes, B in {1, 2, 4, 8, 16}, 16 key and
    value heads, d = 128, bf16; the library's dispatch rule is checked
    against this table (tests/test_dispatch_table.py)."""
    import torch

    import synth
    from gated_deltanet_linear_tree_gb300 import build as bld
    from gated_deltanet_linear_tree_gb300 import canopy
    from synth import configs, trees
    bld.build()
    canopy.load()
    H, d = 16, 128
    flush = torch.empty(1024 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    Bs = [int(x) for x in args.sweep_b.split(",")] if args.sweep_b else configs.SWEEP_B
    Ts = [int(x) for x in args.sweep_t.split(",")] if args.sweep_t else list(range(1, 9))
    out = TableOut(args, "dispatch: closed form vs path replay, H = HV = 16, d = 128, bf16, random trees")
    for B in Bs:
        for T in Ts:
            rng = np.random.default_rng(100 * B + T)
            inp = synth.make_inputs([trees.family("random", T, rng) for _ in range(B)], H, d, d, True, case=3, rnd=T)
            dev = {n: torch.from_numpy(inp[n]).to("cuda", torch.bfloat16) for n in ("q", "k", "v")}
            for n in ("g", "beta", "S0", "parent"):
                dev[n] = torch.from_numpy(inp[n]).cuda()
            ws = canopy.workspace(B, T, H, d)
            o = torch.empty((B, T, H, d), dtype=torch.float32, device="cuda")
            calls = {f: (lambda f=f: canopy.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"],
                                                   dev["parent"], ws, out=o, force=f))
                     for f in ("closed_form", "path_replay")}
            rec = {"B": B, "T": T, "H": H, "HV": H, **time_calls(calls, flush, args.sweep_warmup, args.sweep_reps)}
            assert canopy.read_device_error(ws) == 0
            out.write(rec)
    out.close()


# ---------------------------------------------------------------------------
# crossover sweep: closed-form verify vs the serial replay kernel

def run_sweep(args):
    """For every (B, T, family) cell: median (p10, p90) µs of the closed-form
    verify and of the serial replay, each call timed alone with CUDA events
    after an L2 flush, the two kernels interleaved; the ratio serial/closed is
    the crossover map."""
    import torch

    import synth
    from gated_deltanet_linear_tree_gb300 import build as bld
    from gated_deltanet_linear_tree_gb300 import canopy
    from synth import configs, trees
    bld.build()
    canopy.load()
    H, d = 16, 128
    # 1 GiB: larger than L2, and long enough (about 0.15 ms) that the host has
    # queued the timed call before the GPU reaches it
    flush = torch.empty(1024 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    Bs = [int(x) for x in args.sweep_b.split(",")] if args.sweep_b else configs.SWEEP_B
    Ts = [int(x) for x in args.sweep_t.split(",")] if args.sweep_t else configs.SWEEP_T
    fams = args.sweep_fam.split(",") if args.sweep_fam else configs.SWEEP_FAMILIES
    out = TableOut(args, "crossover: closed-form verify vs serial replay, H = 16, d = 128, bf16")
    solves = ["fwdsub", "neumann"]
    for B in Bs:
        for T in Ts:
            for fam in fams:
                rng = np.random.default_rng(1000 * B + T)
                parents = [trees.family(fam, T, rng) for _ in range(B)]
                inp = synth.make_inputs(parents, H, d, d, True, case=3, rnd=T)
                dev = {n: torch.from_numpy(inp[n]).to("cuda", torch.bfloat16) for n in ("q", "k", "v")}
                for n in ("g", "beta", "S0"):
                    dev[n] = torch.from_numpy(inp[n]).cuda()
                dev["parent"] = torch.from_numpy(inp["parent"]).cuda()
                ws = canopy.workspace(B, T, H, d)
                snap = torch.empty(canopy.snapshot_bytes(B, T, H, d), dtype=torch.uint8, device="cuda")
                o = torch.empty((B, T, H, d), dtype=torch.float32, device="cuda")
                calls = {"serial": lambda: canopy.serial_replay(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                                                dev["S0"], dev["parent"], ws, snapshot=snap, out=o)}
                for sv in solves:
                    if sv == "neumann" and T > 64:
                        continue
                    calls[sv] = (lambda sv=sv: canopy.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                                             dev["S0"], dev["parent"], ws, solve=sv, out=o))
                rec = {"B": B, "T": T, "family": fam, "depth": int(max(trees.tree_depth(p) for p in parents)),
                       **time_calls(calls, flush, args.sweep_warmup, args.sweep_reps)}
                assert canopy.read_device_error(ws) == 0
                rec["speedup_fwdsub"] = rec["serial"]["p50"] / rec["fwdsub"]["p50"]
                if "neumann" in rec:
                    rec["speedup_neumann"] = rec["serial"]["p50"] / rec["neumann"]["p50"]
                out.write(rec)
    out.close()


def run_solve_table(args):
    """The solve strategies side by side (canopy page, "Design decisions":
    blocked forward substitution, the Neumann series, the squaring form and
    the split design; DFS against level order): for B in {1, 16}, each tree
    family at T = 256 (or --sweep-t) under DFS pre-order and under level
    order, median (p10, p90) µs of every strategy's verify call, timed alone
    after an L2 flush, the strategies interleaved; the serial replay beside
    them for scale."""
    import torch

    import synth
    from gated_deltanet_linear_tree_gb300 import build as bld
    from gated_deltanet_linear_tree_gb300 import canopy
    from synth import trees
    bld.build()
    canopy.load()
    H, d = 16, 128
    flush = torch.empty(1024 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    Bs = [int(x) for x in args.sweep_b.split(",")] if args.sweep_b else [1, 16]
    Ts = [int(x) for x in args.sweep_t.split(",")] if args.sweep_t else [256]
    fams = args.sweep_fam.split(",") if args.sweep_fam else ["top8", "top4", "top2", "random", "skewed", "chain"]
    out = TableOut(args, "solve strategies and DFS vs level order, H = 16, d = 128, bf16")
    for B in Bs:
        for T in Ts:
            for fam in fams:
                rng = np.random.default_rng(1000 * B + T)
                base = [trees.family(fam, T, rng) for _ in range(B)]
                for order_name, order_fn in (("dfs", trees.dfs_preorder), ("level", trees.level_order)):
                    parents = [trees.relabel(p, order_fn(p)) for p in base]
                    inp = synth.make_inputs(parents, H, d, d, True, case=3, rnd=T)
                    dev = {n: torch.from_numpy(inp[n]).to("cuda", torch.bfloat16) for n in ("q", "k", "v")}
                    for n in ("g", "beta", "S0"):
                        dev[n] = torch.from_numpy(inp[n]).cuda()
                    dev["parent"] = torch.from_numpy(inp["parent"]).cuda()
                    ws = canopy.workspace(B, T, H, d)
                    snap = torch.empty(canopy.snapshot_bytes(B, T, H, d), dtype=torch.uint8, device="cuda")
                    o = torch.empty((B, T, H, d), dtype=torch.float32, device="cuda")
                    calls = {"serial": lambda: canopy.serial_replay(dev["q"], dev["k"], dev["v"], dev["g"],
                                                                    dev["beta"], dev["S0"], dev["parent"], ws,
                                                                    snapshot=snap, out=o)}
                    for sv in ("fwdsub", "neumann", "squaring", "split"):
                        calls[sv] = (lambda sv=sv: canopy.verify(dev["q"], dev["k"], dev["v"], dev["g"],
                                                                 dev["beta"], dev["S0"], dev["parent"], ws,
                                                                 solve=sv, out=o))
                    rec = {"B": B, "T": T, "family": fam, "order": order_name,
                           "depth": int(max(trees.tree_depth(p) for p in parents)),
                           **time_calls(calls, flush, args.sweep_warmup, args.sweep_reps)}
                    assert canopy.read_device_error(ws) == 0
                    out.write(rec)
                    del ws, snap, o, dev
    out.close()


def run_layer_shape(args):
    """One GDN layer at the shape the canopy page gives for Qwen3.5-9B (16 key
    heads, 32 value heads of 128 x 128, scale 1/sqrt(128) on q), for the
    batch-1 (4, 2, 1) tree of 16 nodes and for random trees of 64 nodes at
    batch 1 and 16: median (p10, p90) us of the verify alone, of verify +
    commit, and of the serial replay, each timed alone after an L2 flush."""
    import torch

    import synth
    from gated_deltanet_linear_tree_gb300 import build as bld
    from gated_deltanet_linear_tree_gb300 import canopy
    from synth import configs, trees
    bld.build()
    canopy.load()
    H, HV, d = 16, 32, 128
    scale = 1.0 / np.sqrt(d)
    # 1 GiB: larger than L2, and long enough (about 0.15 ms) that the host has
    # queued the timed call before the GPU reaches it
    flush = torch.empty(1024 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    out = TableOut(args, "one GDN layer at 16 key / 32 value heads, d = 128, scale 1/sqrt(128)")
    for B, T, fam in ((1, 16, "schedule421"), (1, 64, "random"), (16, 64, "random")):
        rng = np.random.default_rng(7000 + 100 * B + T)
        parents = [configs.make_tree(fam, T, rng) for _ in range(B)]
        ik = synth.make_inputs(parents, H, d, d, True, case=94, rnd=T)
        iv = synth.make_inputs(parents, HV, d, d, True, case=95, rnd=T)
        dev = {"q": torch.from_numpy(ik["q"]).to("cuda", torch.bfloat16),
               "k": torch.from_numpy(ik["k"]).to("cuda", torch.bfloat16),
               "v": torch.from_numpy(iv["v"]).to("cuda", torch.bfloat16)}
        for n in ("g", "beta", "S0"):
            dev[n] = torch.from_numpy(iv[n]).cuda()
        dev["parent"] = torch.from_numpy(iv["parent"]).cuda()
        rng2 = np.random.default_rng(B * T)
        dev["acc"] = torch.tensor([int(rng2.choice(trees.leaves(p))) for p in parents], dtype=torch.int32,
                                  device="cuda")
        ws = canopy.workspace(B, T, HV, d)
        snap = torch.empty(canopy.snapshot_bytes(B, T, HV, d), dtype=torch.uint8, device="cuda")
        o = torch.empty((B, T, HV, d), dtype=torch.float32, device="cuda")
        S_new = torch.empty_like(dev["S0"])

        def ver():
            canopy.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws,
                          out=o, scale=scale)

        def step():
            ver()
            canopy.commit(dev["acc"], dev["S0"], dev["k"], dev["parent"], ws, out=S_new)

        def ser():
            canopy.serial_replay(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws,
                                 snapshot=snap, out=o, scale=scale)

        # the short convolution before the layer over q, k and v channels
        C = 2 * H * d + HV * d
        xc = torch.randn((B, T, C), device="cuda").to(torch.bfloat16)
        cst = torch.randn((B, C, 3), device="cuda")
        cw = 0.5 * torch.randn((C, 4), device="cuda")
        yc = torch.empty_like(xc)

        def conv():
            canopy.tree_conv(xc, cst, cw, dev["parent"], act="silu", out=yc)

        calls = {"verify": ver, "verify_commit": step, "serial": ser, "tree_conv": conv}
        rec = {"layer": "H=16 key heads, HV=32 value heads, dk=dv=128, scale 1/sqrt(128)", "B": B, "T": T,
               "tree": fam, "depth": int(max(trees.tree_depth(p) for p in parents)),
               **time_calls(calls, flush, args.sweep_warmup, args.sweep_reps)}
        assert canopy.read_device_error(ws) == 0
        rec["speedup_verify"] = rec["serial"]["p50"] / rec["verify"]["p50"]
        conv_bytes = 2 * B * T * C * 2 + B * C * 3 * 4 + C * 4 * 4
        rec["tree_conv_channels"] = C
        rec["tree_conv_GBps"] = conv_bytes / (rec["tree_conv"]["p50"] * 1e3)
        out.write(rec)
    out.close()


def run_memory(args):
    """Transient memory of one tree verify per GDN layer and sequence at the
    canopy page's model shape (32 value heads of 128 x 128), for the serial
    replay's per-node snapshots and for this library: the pseudo-values and
    log gates the commit reads, and the whole workspace as allocated (with
    the T x T scratch of the paths beyond 64 nodes).  Host arithmetic through
    the library's own size functions; no GPU needed."""
    from gated_deltanet_linear_tree_gb300 import build as bld
    from gated_deltanet_linear_tree_gb300 import canopy
    bld.build()
    canopy.load()
    HV, d, layers = 32, 128, 24
    mib = float(1 << 20)
    for T in (16, 64, 100, 128, 256):
        snap = canopy.snapshot_bytes(1, T, HV, d)
        ws = canopy.workspace_bytes(1, T, HV, d)
        factors = T * HV * d * 4 + T * HV * 4          # U and l, what the commit reads
        rec = {"per": "one GDN layer, one sequence (HV=32 value heads, dk=dv=128)", "T": T,
               "snapshots_MiB": snap / mib, "U_and_l_MiB": factors / mib, "workspace_MiB": ws / mib,
               "ratio_snapshots_to_U_and_l": snap / factors, "ratio_snapshots_to_workspace": snap / ws,
               "all_24_layers": {"snapshots_MiB": layers * snap / mib, "workspace_MiB": layers * ws / mib}}
        print(json.dumps(rec), flush=True)


PROFILE_CASES = {
    # name: (what runs, B, T, tree family)
    "verify64": ("verify", 16, 64, "random_depth_4_20"),
    "verify128": ("verify", 16, 128, "random"),
    "verify256": ("verify", 16, 256, "random"),
    "verify256_chain": ("verify", 16, 256, "chain"),
    "neumann64": ("neumann", 16, 64, "random_depth_4_20"),
    "neumann256": ("neumann", 16, 256, "random"),
    "neumann256_top8": ("neumann", 16, 256, "top8"),
    "squaring256": ("squaring", 16, 256, "random"),
    "squaring256_chain": ("squaring", 16, 256, "chain"),
    "split256": ("split", 16, 256, "random"),
    "commit64": ("commit", 16, 64, "random_depth_4_20"),
    "serial64": ("serial", 4, 64, "random_depth_4_20"),
    "path_replay3": ("path_replay", 16, 3, "random"),
    "tree_conv64": ("tree_conv", 16, 64, "random_depth_4_20"),
}


def run_profile_case(args):
    """A small, fixed case of one kernel for profilers: seeded inputs (16 key
    and value heads, d = 128, bf16 q/k/v, fp32 S0 and o), one warm-up call,
    then --profile-reps calls, each after a 256 MB read that evicts L2 (a
    read leaves clean lines, so the call pays no write-back of them).  The
    tree convolution runs over the 8,192 channels of a 16-key / 32-value-head
    layer's q, k and v (K = 4, SiLU).  Device memory stays under 1 GB."""
    import torch

    import synth
    from gated_deltanet_linear_tree_gb300 import build as bld
    from gated_deltanet_linear_tree_gb300 import canopy
    from synth import configs, trees
    bld.build()
    canopy.load()
    kind, B, T, fam = PROFILE_CASES[args.profile_case]
    H, d = 16, 128
    rng = np.random.default_rng(11)
    parents = [configs.make_tree(fam, T, rng) for _ in range(B)]
    inp = synth.make_inputs(parents, H, d, d, True, case=97, rnd=T)
    dev = {n: torch.from_numpy(inp[n]).to("cuda", torch.bfloat16) for n in ("q", "k", "v")}
    for n in ("g", "beta", "S0", "parent"):
        dev[n] = torch.from_numpy(inp[n]).cuda()
    dev["acc"] = torch.tensor([int(rng.choice(trees.leaves(p))) for p in parents], dtype=torch.int32,
                              device="cuda")
    ws = canopy.workspace(B, T, H, d)
    o = torch.empty((B, T, H, d), dtype=torch.float32, device="cuda")
    S_new = torch.empty_like(dev["S0"])
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")

    def ver(solve="fwdsub", force=None):
        canopy.verify(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws,
                      solve=solve, out=o, force=force)

    if kind == "verify":
        fn = ver
    elif kind in ("neumann", "squaring", "split"):
        def fn():
            ver(kind)
    elif kind == "path_replay":
        def fn():
            ver(force="path_replay")
    elif kind == "commit":
        ver()

        def fn():
            canopy.commit(dev["acc"], dev["S0"], dev["k"], dev["parent"], ws, out=S_new)
    elif kind == "serial":
        snap = torch.empty(canopy.snapshot_bytes(B, T, H, d), dtype=torch.uint8, device="cuda")

        def fn():
            canopy.serial_replay(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], dev["S0"], dev["parent"], ws,
                                 snapshot=snap, out=o)
    elif kind == "tree_conv":
        C = 2 * 16 * d + 32 * d
        gen = torch.Generator(device="cuda")
        gen.manual_seed(5)
        xc = torch.randn((B, T, C), device="cuda", generator=gen).to(torch.bfloat16)
        cst = torch.randn((B, C, 3), device="cuda", generator=gen)
        cw = 0.5 * torch.randn((C, 4), device="cuda", generator=gen)
        yc = torch.empty_like(xc)
        # eight input / output pairs (268 MB) for the back-to-back graph below
        xs = [xc] + [torch.randn_like(xc, dtype=torch.float32).to(torch.bfloat16) for _ in range(7)]
        ys = [torch.empty_like(xc) for _ in range(8)]

        def fn():
            canopy.tree_conv(xc, cst, cw, dev["parent"], act="silu", out=yc)

        def rotating(i):
            canopy.tree_conv(xs[i % 8], cst, cw, dev["parent"], act="silu", out=ys[i % 8])
    else:
        raise ValueError(kind)
    fn()
    torch.cuda.synchronize()
    times = []
    flush.fill_(1.0)
    torch.cuda.synchronize()
    for i in range(args.profile_reps):
        flush.sum()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        times.append(1e3 * a.elapsed_time(b))
    assert canopy.read_device_error(ws) == 0
    rec = {"profile_case": args.profile_case, "kind": kind, "B": B, "T": T, "tree": fam,
           "depth": int(max(trees.tree_depth(p) for p in parents)), "us_per_call_after_l2_read": times}
    if kind == "tree_conv":
        # back to back over the eight pairs (each call's data is out of L2):
        # one graph of 64 calls, replayed
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(64):
                rotating(i)
        g.replay()
        torch.cuda.synchronize()
        reps = []
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            reps.append(1e3 * a.elapsed_time(b) / 64)
        rec["us_per_call_back_to_back"] = reps
        # the same bytes moved by a plain device copy (y = x), for scale
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2):
            for i in range(64):
                ys[i % 8].copy_(xs[i % 8])
        g2.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g2.replay()
        b.record()
        torch.cuda.synchronize()
        rec["us_per_plain_copy_of_x_back_to_back"] = 1e3 * a.elapsed_time(b) / 64
    print(json.dumps(rec), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["canopy", "reference"], default="canopy")
    ap.add_argument("--solve", choices=["fwdsub", "neumann", "squaring", "split"], default="fwdsub")
    ap.add_argument("--sets", type=int, default=8)
    ap.add_argument("--graph-steps", type=int, default=200, help="steps per captured graph")
    ap.add_argument("--kernel-reps", type=int, default=5, help="replays of the one-kernel graphs")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="crossover map vs the serial replay kernel")
    ap.add_argument("--memory", action="store_true",
                    help="transient memory per layer: serial snapshots vs this library's workspace")
    ap.add_argument("--layer-shape", action="store_true",
                    help="one GDN layer at 16 key / 32 value heads with the 1/sqrt(dk) q scale")
    ap.add_argument("--solve-table", action="store_true",
                    help="solve strategies and DFS vs level order side by side (T = 256 by default)")
    ap.add_argument("--dispatch-table", action="store_true",
                    help="closed form vs path replay below the crossover (the dispatch rule's data)")
    ap.add_argument("--sweep-b", default="")
    ap.add_argument("--sweep-t", default="")
    ap.add_argument("--sweep-fam", default="")
    ap.add_argument("--sweep-reps", type=int, default=50)
    ap.add_argument("--sweep-warmup", type=int, default=10)
    ap.add_argument("--sweep-out", default="")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default="",
                    help="a small fixed case of one kernel, for ncu")
    ap.add_argument("--profile-reps", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    if args.memory:
        run_memory(args)
        return
    if args.layer_shape:
        run_layer_shape(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.solve_table:
        run_solve_table(args)
        return
    if args.dispatch_table:
        run_dispatch_table(args)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_canopy(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
