"""Benchmark of the GB300 mHC seam (delayed pre + post).

Headline workload: the prefill seam, T = 16384 tokens, n = 4 streams,
C = 5120, 20 Sinkhorn iterations, fused RMSNorm fold on; one step = one
mhc_pre_delayed + one mhc_post over the batch (every step of the seam).
`value` = tokens/s (whole job, all ranks).  Inputs (x 671 MB) are larger than
L2 (129 MB), so no explicit flush is needed between steps.  Secondary keys
carry the decode sweep (T = 1..128: a graph of 20 back-to-back calls, as in a
model step, median of 5 x 50 replays, per call), the 80-seam decode chain (one
graph) and per-kernel HBM roofline figures.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--skip-decode] [--skip-cpu]

`--impl reference` times the CPU oracle (this seam has no other reference
implementation) on the same workload and metric, on a bounded token sample
per step.  Multi-GPU (torchrun): independent replicas, one batch per rank,
no collective on the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "mHC seam µs/call T=1–128 (graph); tokens/s + HBM GB/s vs peak at T=16384"
T_PREFILL, N_STREAMS, HIDDEN, ITERS = 16384, 4, 5120, 20
DECODE_T = (1, 2, 4, 8, 16, 32, 64, 128)
CHAIN_SEAMS, CHAIN_T = 80, 4
DECODE_REPS = 20   # calls per captured graph in the decode sweep

# algorithmic bytes (what the method must move; fn counted once per call)
PRE_BYTES_PER_TOKEN = 40960 + 10240 + 16 + 16 + 16 + 64   # x, layer_input, pre_in, pre, post, comb
PRE_BYTES_FIXED = 24 * 20480 * 4 + 24 * 4 + 12 + 5120 * 2  # fn, bias, alpha, norm_weight
POST_BYTES_PER_TOKEN = 40960 + 10240 + 64 + 16 + 40960     # x, y, comb, post, x_new
PRE_FLOP_PER_TOKEN = 2 * 24 * 20480
# model-entry broadcast seam: x is [T, C], read once for all four streams
PRE_BCAST_BYTES_PER_TOKEN = 10240 + 10240 + 16 + 16 + 16 + 64   # x, layer_input, pre_in, pre, post, comb
POST_BCAST_BYTES_PER_TOKEN = 10240 + 10240 + 64 + 16 + 40960    # x, y, comb, post, x_new


def pre_bytes(T):
    return T * PRE_BYTES_PER_TOKEN + PRE_BYTES_FIXED


def post_bytes(T):
    return T * POST_BYTES_PER_TOKEN


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank scalar over the default process group (the
    timed region's slowest rank); the value itself when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_throughput(tokens_per_rank: int, steps: int, world: int, elapsed_ms_max: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch each step; the
    job time is the slowest rank's."""
    return world * tokens_per_rank * steps / (elapsed_ms_max / 1e3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# sources each kernel is built from: a committed ncu traffic figure is used
# only while these files are unchanged
KERNEL_SOURCES = {
    "mhc_pre_delayed": ("pre_tc.cu", "sm100.cuh", "common.cuh"),
    "mhc_pre_delayed_packed": ("pre_tc.cu", "sm100.cuh", "common.cuh"),
    "mhc_post": ("post.cu", "common.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mhc_hyper_connection_pre_gb300", "csrc")
    for fn in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` at the benchmark's
    size, from the committed ncu summary; None when that kernel's sources
    changed since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    k = d.get("kernels", {}).get(kernel)
    if k is None or k.get("source_hash") != kernel_source_hash(kernel):
        return None
    return k.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        sel = ["-i", str(device_index)]
        try:
            import torch
            props = torch.cuda.get_device_properties(device_index)
            bus_id = "{:08x}:{:02x}:{:02x}.0".format(props.pci_domain_id, props.pci_bus_id,
                                                    props.pci_device_id)
            probe = subprocess.run(["nvidia-smi", "-i", bus_id, "--query-gpu=clocks.max.sm",
                                    "--format=csv,noheader"], capture_output=True, text=True,
                                   timeout=20)
            if probe.returncode == 0 and probe.stdout.strip():
                sel = ["-i", bus_id]
        except Exception:
            pass
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "100"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for name, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_info():
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for l in f:
                if l.lower().startswith(("model name", "cpu part", "hardware")):
                    model = l.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return os.cpu_count() or 1, model


def time_oracle_sample(d, tokens: int, nthreads: int):
    """Oracle pre + post on the first `tokens` rows of the workload; seconds."""
    import numpy as np
    import oracle
    from workloads import bf16_bits
    x = bf16_bits(d["x"][:tokens])
    y = bf16_bits(d["y"][:tokens])
    pre_in = d["pre_in"][:tokens].cpu().numpy()
    fn, bias, alpha = d["fn"].cpu().numpy(), d["bias"].cpu().numpy(), d["alpha"].cpu().numpy()
    nw = bf16_bits(d["norm_w"])
    t0 = time.perf_counter()
    o = oracle.pre_delayed(x, pre_in, fn, bias, alpha, nw, nthreads=nthreads)
    oracle.post(x, y, o["comb"].astype(np.float32), o["post"].astype(np.float32), nthreads=nthreads)
    return time.perf_counter() - t0


# ------------------------------------------------------------ our arm ---

def run_ours(args, rank, world, local):
    import torch
    import mhc_hyper_connection_pre_gb300 as mhc
    from mhc_hyper_connection_pre_gb300.graphs import SeamGraph
    from workloads import seam_inputs, chain_seam_params, chain_stub_delta

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    hbm_peak, peak_kind = load_peaks()
    T = args.tokens
    d = seam_inputs(T, seed=rank, fold=True, with_y=True, device=f"cuda:{local}")
    x, y = d["x"], d["y"]
    pre_in = [d["pre_in"], torch.empty_like(d["pre_in"])]
    outs = [{"pre": torch.empty(T, 4, device=dev), "post": torch.empty(T, 4, device=dev),
             "comb": torch.empty(T, 4, 4, device=dev),
             "layer_input": torch.empty(T, HIDDEN, dtype=torch.bfloat16, device=dev)} for _ in range(2)]
    x_new = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    # --packed: fn's planes packed once ahead (a weight transform, outside the
    # timed region), the pre reading that single copy
    packed = mhc.pre_pack(d["fn"]) if args.packed else None
    pre_name = "mhc_pre_delayed_packed" if args.packed else "mhc_pre_delayed"

    def step(i, ev=None):
        o = outs[i & 1]
        o["pre"] = pre_in[(i + 1) & 1]          # this seam's pre-mix feeds the next step
        if ev is not None:
            ev[0].record(stream)
        if packed is not None:
            mhc.pre_delayed_packed(x, pre_in[i & 1], d["fn"], packed, d["bias"], d["alpha"], d["norm_w"], out=o)
        else:
            mhc.pre_delayed(x, pre_in[i & 1], d["fn"], d["bias"], d["alpha"], d["norm_w"], out=o)
        if ev is not None:
            ev[1].record(stream)
        mhc.post(x, y, o["comb"], o["post"], out=x_new)
        if ev is not None:
            ev[2].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    for i in range(args.warmup):
        step(i)
    barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        t_begin = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_begin.record(stream)
        for i in range(args.steps):
            step(i, evs[i])
        t_end.record(stream)
        barrier()
    elapsed_ms = max_over_ranks(t_begin.elapsed_time(t_end), dev)
    pre_ms = [e[0].elapsed_time(e[1]) for e in evs]
    post_ms = [e[1].elapsed_time(e[2]) for e in evs]
    ms_per_step = elapsed_ms / args.steps
    tokens_per_s = weak_scaling_throughput(T, args.steps, world, elapsed_ms)

    pre_avg = sum(pre_ms) / len(pre_ms)
    post_avg = sum(post_ms) / len(post_ms)
    kernels = {
        pre_name: {"us": pre_avg * 1e3, "bytes": pre_bytes(T),
                            "gbs": pre_bytes(T) / (pre_avg / 1e3) / 1e9},
        "mhc_post": {"us": post_avg * 1e3, "bytes": post_bytes(T),
                     "gbs": post_bytes(T) / (post_avg / 1e3) / 1e9},
    }
    for k in kernels.values():
        k["frac_of_hbm_peak"] = k["gbs"] / hbm_peak
    dom = max(kernels, key=lambda k: kernels[k]["us"])
    roof = {"bound": "hbm", "kernel": dom, "achieved": round(kernels[dom]["gbs"], 1),
            "peak": hbm_peak, "unit": "GB/s", "frac": round(kernels[dom]["gbs"] / hbm_peak, 4),
            "traffic": ncu_traffic(dom), "peak_kind": f"{peak_kind} (STREAM-style copy)"}
    seam_frac = (pre_bytes(T) + post_bytes(T)) / hbm_peak / 1e9 / (ms_per_step / 1e3)

    # ---- end to end through the public API: pinned host in, pinned host out
    e2e = None
    if not args.skip_e2e:
        hx = torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x)
        hy = torch.empty(y.shape, dtype=y.dtype, pin_memory=True).copy_(y)
        hp = torch.empty(pre_in[0].shape, pin_memory=True).copy_(pre_in[0])
        ho = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        hpo = torch.empty(pre_in[0].shape, pin_memory=True)
        ek = max(3, min(20, args.steps))
        hout = {"x_new": ho, "pre": hpo}

        def e2e_step():
            # the library's host-buffer call: chunked copies in and out
            # overlapped with the kernels on its own streams
            mhc.seam_host(hx, hy, hp, d["fn"], d["bias"], d["alpha"], d["norm_w"], out=hout, stream=stream)

        for _ in range(2):
            e2e_step()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(ek):
            e2e_step()
        b.record(stream)
        barrier()
        e_ms = max_over_ranks(a.elapsed_time(b), dev)
        h2d = x.numel() * 2 + y.numel() * 2 + pre_in[0].numel() * 4
        d2h = x_new.numel() * 2 + pre_in[0].numel() * 4
        e2e = {"value": round(weak_scaling_throughput(T, ek, world, e_ms), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e_ms / ek, 4)}
        del hx, hy, hp, ho, hpo

    # ---- the other prefill entry points at the same T (rank 0 only): the
    # model-entry broadcast seam and the non-delayed pre
    other_prefill = None
    if rank == 0 and (not args.skip_decode or args.other_prefill):
        xe = x[:, 0, :].contiguous()
        oe = {k: torch.empty_like(v) for k, v in outs[0].items()}
        xne = torch.empty_like(x)

        def timed(call, reps=20):
            for _ in range(3):
                call()
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            a_ev.record(stream)
            for _ in range(reps):
                call()
            b_ev.record(stream)
            torch.cuda.synchronize(dev)
            return a_ev.elapsed_time(b_ev) * 1e3 / reps

        fixed = PRE_BYTES_FIXED
        cases = {
            "mhc_pre_delayed_broadcast": (lambda: mhc.pre_delayed_broadcast(
                xe, pre_in[0], d["fn"], d["bias"], d["alpha"], d["norm_w"], out=oe),
                T * PRE_BCAST_BYTES_PER_TOKEN + fixed),
            "mhc_post_broadcast": (lambda: mhc.post_broadcast(xe, y, oe["comb"], oe["post"], out=xne),
                                   T * POST_BCAST_BYTES_PER_TOKEN),
            "mhc_pre": (lambda: mhc.pre(x, d["fn"], d["bias"], d["alpha"], d["norm_w"], out=oe), pre_bytes(T)),
            # post of one seam and the next seam's delayed pre in one call; the
            # bytes are the fused op's own (the pre consumes x_new without
            # reading it back), so the fraction shows what a one-pass kernel would gain
            "mhc_post_pre_delayed": (lambda: mhc.post_pre_delayed(
                x, y, outs[0]["comb"], outs[0]["post"], pre_in[0], d["fn"], d["bias"], d["alpha"], d["norm_w"],
                x_new=xne, out=oe), post_bytes(T) + pre_bytes(T) - T * 40960),
            # fn's planes packed once ahead (a weight transform, outside the timing)
            "mhc_pre_delayed_packed": (lambda: mhc.pre_delayed_packed(x, pre_in[0], d["fn"], packed, d["bias"],
                                                                      d["alpha"], d["norm_w"], out=oe),
                                       pre_bytes(T)),
        }
        packed = mhc.pre_pack(d["fn"])
        other_prefill = {}
        for name, (call, nbytes) in cases.items():
            us = timed(call)
            other_prefill[name] = {"us": round(us, 2), "bytes": nbytes, "gbs": round(nbytes / us / 1e3, 1),
                                   "frac_of_hbm_peak": round(nbytes / us / 1e3 / hbm_peak, 4)}
        assert mhc.device_status() == 0, "a bounded in-kernel wait timed out"
        del xe, oe, xne, packed
        # the stress workload: T = 65536, comb logits driven to +-30 and beyond,
        # 1 % of the rows scaled by 1e3 and 1 % all zero
        Ts = 65536
        ds = seam_inputs(Ts, seed=0, fold=True, stress=True, device=f"cuda:{local}")
        os_ = mhc.pre_delayed(ds["x"], ds["pre_in"], ds["fn"], ds["bias"], ds["alpha"], ds["norm_w"])
        us = timed(lambda: mhc.pre_delayed(ds["x"], ds["pre_in"], ds["fn"], ds["bias"], ds["alpha"],
                                           ds["norm_w"], out=os_), reps=10)
        nb = pre_bytes(Ts)
        other_prefill["mhc_pre_delayed_stress_T65536"] = {
            "us": round(us, 2), "bytes": nb, "gbs": round(nb / us / 1e3, 1),
            "frac_of_hbm_peak": round(nb / us / 1e3 / hbm_peak, 4)}
        assert mhc.device_status() == 0, "a bounded in-kernel wait timed out"
        del ds, os_

    # ---- decode sweep and the 80-seam chain (rank 0 only)
    decode = chain = None
    if rank == 0 and not args.skip_decode:
        decode = {}
        s = torch.cuda.Stream(dev)
        for Td in DECODE_T:
            dd = seam_inputs(Td, seed=Td, fold=True, with_y=True, device=f"cuda:{local}")
            o = mhc.pre_delayed(dd["x"], dd["pre_in"], dd["fn"], dd["bias"], dd["alpha"], dd["norm_w"])
            xn = torch.empty_like(dd["x"])
            torch.cuda.synchronize()
            res = {}
            def pre_call(st):
                mhc.pre_delayed(dd["x"], dd["pre_in"], dd["fn"], dd["bias"], dd["alpha"], dd["norm_w"],
                                out=o, stream=st)

            def seam_call(st):
                pre_call(st)
                mhc.post(dd["x"], dd["y"], o["comb"], o["post"], out=xn, stream=st)

            def fused_call(st):
                # post of the previous seam (its gates: o) fused with this pre
                mhc.post_pre_delayed(dd["x"], dd["y"], o["comb"], o["post"], dd["pre_in"], dd["fn"], dd["bias"],
                                     dd["alpha"], dd["norm_w"], x_new=xn, out=o, stream=st)

            xe = dd["x"][:, 0, :].contiguous()

            def entry_call(st):
                # the model-entry broadcast seam: pre and post on x [T, C]
                mhc.pre_delayed_broadcast(xe, dd["pre_in"], dd["fn"], dd["bias"], dd["alpha"], dd["norm_w"],
                                          out=o, stream=st)
                mhc.post_broadcast(xe, dd["y"], o["comb"], o["post"], out=xn, stream=st)

            def nondelayed_call(st):
                # the non-delayed block: collapse with its own pre-mix
                mhc.pre(dd["x"], dd["fn"], dd["bias"], dd["alpha"], dd["norm_w"], out=o, stream=st)

            for name, one, ov in (("pre", pre_call, False), ("seam", seam_call, False),
                                  ("fused_seam", fused_call, False), ("pre_nondelayed", nondelayed_call, False),
                                  ("entry_seam", entry_call, False),
                                  ("pre_overlap", pre_call, True), ("seam_overlap", seam_call, True),
                                  ("fused_seam_overlap", fused_call, True)):
                mhc.set_launch_overlap(ov)
                # DECODE_REPS calls back to back in one graph: the GPU time per
                # call, not the host's graph-launch rate
                g = SeamGraph(lambda st, one=one: [one(st) for _ in range(DECODE_REPS)], s)
                g.replay(5)
                meds = []
                for _ in range(5):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(s)
                    g.replay(50)
                    b.record(s)
                    s.synchronize()
                    meds.append(a.elapsed_time(b) * 1e3 / (50 * DECODE_REPS))
                res[name + "_us"] = round(statistics.median(meds), 3)
                res[name + "_launches"] = g.kernel_nodes / DECODE_REPS
                g.close()
            mhc.set_launch_overlap(False)
            decode[str(Td)] = res
        # 80 seams, each with its own weights, pre-mix carried seam to seam
        params = [chain_seam_params(si, device=f"cuda:{local}") for si in range(CHAIN_SEAMS)]
        deltas = [chain_stub_delta(si, device=f"cuda:{local}") for si in range(CHAIN_SEAMS)]
        c0 = seam_inputs(CHAIN_T, seed=0, device=f"cuda:{local}")
        cx = c0["x"].clone()
        cp = [c0["pre_in"].clone(), torch.empty_like(c0["pre_in"])]
        co = {"post": torch.empty(CHAIN_T, 4, device=dev), "comb": torch.empty(CHAIN_T, 4, 4, device=dev),
              "layer_input": torch.empty(CHAIN_T, HIDDEN, dtype=torch.bfloat16, device=dev)}
        cy = torch.empty(CHAIN_T, HIDDEN, dtype=torch.bfloat16, device=dev)

        def chain_step(st):
            for si in range(CHAIN_SEAMS):
                p = params[si]
                o = dict(co, pre=cp[(si + 1) & 1])
                mhc.pre_delayed(cx, cp[si & 1], p["fn"], p["bias"], p["alpha"], p["norm_w"], out=o, stream=st)
                with torch.cuda.stream(st):
                    torch.add(co["layer_input"], deltas[si], out=cy)   # synthetic sublayer
                mhc.post(cx, cy, co["comb"], co["post"], out=cx, stream=st)

        def chain_step_fused(st):
            # the same step with post(s - 1) fused into pre(s)
            for si in range(CHAIN_SEAMS):
                p = params[si]
                o = dict(co, pre=cp[(si + 1) & 1])
                if si == 0:
                    mhc.pre_delayed(cx, cp[0], p["fn"], p["bias"], p["alpha"], p["norm_w"], out=o, stream=st)
                else:
                    mhc.post_pre_delayed(cx, cy, co["comb"], co["post"], cp[si & 1], p["fn"], p["bias"],
                                         p["alpha"], p["norm_w"], x_new=cx, out=o, stream=st)
                with torch.cuda.stream(st):
                    torch.add(co["layer_input"], deltas[si], out=cy)   # synthetic sublayer
            mhc.post(cx, cy, co["comb"], co["post"], out=cx, stream=st)

        chain_us = {}
        for fused, ov, early in ((False, False, False), (False, True, False), (True, False, False),
                                 (True, True, False), (False, True, True), (True, True, True)):
            mhc.set_launch_overlap(ov)
            step_fn = chain_step_fused if fused else chain_step
            with torch.cuda.stream(s):
                step_fn(s)
            s.synchronize()
            g = SeamGraph(step_fn, s, early_launch=early)
            g.replay(3)
            meds = []
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                g.replay(200)
                b.record(s)
                s.synchronize()
                meds.append(a.elapsed_time(b) * 1e3 / 200)
            chain_us[(fused, ov, early)] = round(statistics.median(meds), 2)
            if fused:
                fused_nodes = g.kernel_nodes
            else:
                nodes = g.kernel_nodes
            g.close()
        mhc.set_launch_overlap(False)
        chain = {"us_per_step": chain_us[(False, False, False)],
                 "us_per_step_overlap": chain_us[(False, True, False)],
                 "us_per_step_fused": chain_us[(True, False, False)],
                 "us_per_step_fused_overlap": chain_us[(True, True, False)],
                 "us_per_step_overlap_early": chain_us[(False, True, True)],
                 "us_per_step_fused_overlap_early": chain_us[(True, True, True)],
                 "us_per_step_best": min(chain_us.values()),
                 "best_config": {(False, False, False): "2 launches/seam", (False, True, False): "2 launches/seam, overlap",
                                 (True, False, False): "fused", (True, True, False): "fused, overlap",
                                 (False, True, True): "2 launches/seam, overlap, early launch",
                                 (True, True, True): "fused, overlap, early launch"}[
                     min(chain_us, key=chain_us.get)],
                 "seams": CHAIN_SEAMS, "T": CHAIN_T, "kernel_nodes": nodes,
                 "launches_per_seam": (nodes - CHAIN_SEAMS) / CHAIN_SEAMS,
                 "launches_per_seam_fused": (fused_nodes - CHAIN_SEAMS) / CHAIN_SEAMS,
                 "l2": "fn of 80 seams = 157 MB > L2"}
        g.close()

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        cores, model = cpu_info()
        probe = 64
        dt = time_oracle_sample(d, probe, cores)
        tokens = int(max(probe, min(T, probe * 12.0 / max(dt, 1e-6))))
        dt = time_oracle_sample(d, tokens, cores)
        cpu = {"value": round(tokens / dt, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"first {tokens} of the {T} tokens, pre + post, fp64 oracle, {cores} threads"
                         + (f" ({model})" if model else "")}
        # the oracle per call at the decode sizes and on a prefill sample, one
        # thread and every core (context for the GPU numbers, not a target)
        by_t = {}
        for Tc in (16, 128):
            dc = seam_inputs(Tc, seed=Tc, fold=True, with_y=True)
            r = {}
            for th in (1, cores):
                r[f"us_per_call_{th}_threads"] = round(time_oracle_sample(dc, Tc, th) * 1e6, 1)
            by_t[str(Tc)] = r
        by_t[str(T) + "_sample_64"] = {"tokens_per_s_1_thread": round(64 / time_oracle_sample(d, 64, 1), 1)}
        cpu["by_T"] = by_t

    line = {
        "metric": METRIC, "value": round(tokens_per_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16/fp32",
        "data": "synthetic (seeded N(0,1) streams, N(0,0.02^2) fn; no checkpoint)",
        "config": workload_config(T, world, pre_name, args.packed),
        "seam_hbm_frac": round(seam_frac, 4),
        "kernels": {k: {kk: round(vv, 3) if isinstance(vv, float) else vv for kk, vv in v.items()}
                    for k, v in kernels.items()},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        # per step: the post, and the pre (from 256 tokens on the tensor-core
        # path: fn's planes packed, then the kernel; one launch with --packed)
        "gpu_launches": (1 + (2 if mhc.pre_plan(T)["kernel"] == 2 and not args.packed else 1)) * args.steps,
        "clocks": clk.summary(),
        "other_prefill": other_prefill,
        "decode_graph": decode,
        "decode_graph_method": (f"per T: {DECODE_REPS} back-to-back calls captured in one CUDA graph, "
                                "replayed 50 times, 5 repeats, median of the repeats / (50 x "
                                f"{DECODE_REPS}) = microseconds per call; a graph holding one call "
                                "would time this host's graph-launch rate (about 14 us), not the GPU"),
        "decode_chain_80": chain,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------ reference arm ---

def workload_config(T: int, world: int, pre_name: str = "mhc_pre_delayed", packed: bool = False) -> dict:
    """The workload both arms time, described the same way (the driver
    compares the two lines' config)."""
    return {"workload": f"prefill seam: {pre_name} (fold) + mhc_post, T={T}, n=4, C=5120, 20 Sinkhorn iters",
            "T": T, "n": N_STREAMS, "C": HIDDEN, "sinkhorn_iters": ITERS, "fold": True, "per_rank_tokens": T,
            "fn": "bf16 planes packed once ahead (mhc_pre_pack)" if packed else "fp32 weights given to every call",
            "l2": f"inputs larger than L2 (x {T * 40960 / 1e6:.0f} MB vs 129 MB), no flush",
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world, local):
    if rank != 0:
        return
    import torch
    from workloads import seam_inputs
    T = T_PREFILL
    d = seam_inputs(T, seed=0, fold=True, with_y=True, device="cpu")
    cores, model = cpu_info()
    probe = 16
    dt = time_oracle_sample(d, probe, cores)
    per_token = dt / probe
    budget = 150.0
    steps_total = args.steps + args.warmup
    tokens = int(max(1, min(T, budget / max(1, steps_total) / per_token)))
    for _ in range(args.warmup):
        time_oracle_sample(d, tokens, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle_sample(d, tokens, cores)
    el = time.perf_counter() - t0
    value = tokens * args.steps / el
    sample = (f"first {tokens} of the {T} tokens per step, pre + post, fp64 oracle, {cores} threads"
              + (f" ({model})" if model else ""))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(T, world),
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    _ = torch


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--packed", action="store_true",
                    help="the timed pre reads fn planes packed once ahead by mhc_pre_pack (a weight transform "
                         "outside the timed region) instead of converting fp32 fn per call")
    ap.add_argument("--other-prefill", action="store_true",
                    help="time the other prefill entry points (broadcast seam, mhc_pre, packed fn, the stress "
                         "workload) even with --skip-decode")
    ap.add_argument("--tokens", type=int, default=T_PREFILL,
                    help="tokens per rank (default 16384; smaller only for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
