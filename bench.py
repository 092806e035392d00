#!/usr/bin/env python
"""Benchmark of the B300 selective scan (S6).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one forward selective scan (fused discretisation, recurrence,
readout, skip and gate, the state carried across time chunks and the final
state returned) over one batch of the headline workload, the largest scan
workload: bf16 I/O, fp32 state, batch 1, 5120 channels, N 16, L 65536, G 1.
Rank 0 prints one JSON line.  `value` is the whole-job rate of compulsory bytes (u, delta, z, y
plus B, C) per second, device-timed with CUDA events around a CUDA graph of K
launches over rotating input sets that together exceed 3x the L2 cache.  The
same line carries the end-to-end rate through the public API with host
buffers, the decode-step rate (tokens/s), the roofline of the scan kernel and
the fp64 CPU oracle timed on this host as a baseline.

--impl reference times the fp64 CPU oracle instead (the reference arm: no
GPU code exists on the pages), on a bounded sample of the same workload.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own independent
batches (weak scaling, no data-path collective); the time is the max over
ranks and `value` sums the bytes of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "scan_bf16_b1_d5120_l65536_final_state"
DECODE = "decode_b256_d5120"
METRIC = "selective-scan fwd GB/s and % of B300 HBM roofline; decode tokens/s"
FALLBACK_HBM_GBS = 6400.0
# One state update (b, d, l, n) needs one MUFU.EX2 (the decay) and four fp32
# FMA-pipe operations (Delta*A, Delta*u*B, the FMA of the recurrence, the FMA
# of the readout).  The arithmetic roofline is the rate at which the slower of
# the two pipes can supply that, measured live on the GPU by
# ssm_probe_alu_rates (nominal B300 rates: 32 ex2 and 128 FMA per SM per
# clock, i.e. 32 updates per SM per clock from either pipe).
NOMINAL_UPDATES_PER_SM_CLK = 32.0
# Nominal HBM3e bandwidth the scan's memory target is stated against (the
# measured copy bandwidth of the peaks file is the roofline's denominator).
NOMINAL_HBM_GBS = 8000.0


# ---------------------------------------------------------------------------
# distributed plumbing (host-side; tested with gloo on CPU)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self, t0, t1):
        sm, mx, reasons, power = [], None, set(), []
        for ts, line in self.lines:
            if ts < t0 or ts > t1:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"], parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "sm_max_mhz": 2032.0}, "fallback"


# Device sources of the chunked forward call's kernels (summary, carry and
# fused passes): a DRAM-traffic record stays valid while these and the launch
# plan are unchanged.
FWD_SCAN_SOURCES = ("scan_tma.cuh", "tma.cuh", "ssm_device.cuh")


def kernel_source_hash(names=FWD_SCAN_SOURCES):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_109_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name in names:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def ncu_record(kernel_key: str, plan=None):
    """The committed ncu record of one call (DRAM bytes and serialised time per
    kernel), if it was taken on the current kernel sources and launch plan;
    else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(kernel_key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    if plan is not None and rec.get("plan") != plan:
        return None
    return rec


def n_rotating_sets(bytes_per_set: int, l2_bytes: int) -> int:
    return max(2, math.ceil(3 * l2_bytes / max(1, bytes_per_set)))


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def bench_scan_device(ssm, I, torch, w, steps, warmup, sampler=None, preroll_s=1.0, pass_reps=0):
    """Device-timed forward scan over rotating input sets (> 3x L2).  With
    pass_reps > 0, afterwards times the call's fused pass alone: that many
    eager calls with CUDA events recorded by the library around the fused
    pass's launch (on the call's stream)."""
    dev = torch.device("cuda")
    props = torch.cuda.get_device_properties(dev)
    nbytes = I.compulsory_bytes_scan(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"], w["io"])
    nsets = n_rotating_sets(nbytes, props.L2_cache_size)
    sets = [I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"], io=w["io"],
                               recipe=w["recipe"], seed=s, device=dev) for s in range(nsets)]
    outs = [torch.empty_like(x.u) for x in sets]
    # The timed call is the chunked entry point (time-parallel chunks with the
    # carried state, final state returned): the whole forward path.
    hfs = [torch.empty((w["batch"], w["dim"], w["dstate"]), dtype=torch.float32, device=dev)
           for _ in range(nsets)]
    need = ssm.chunked_workspace_size(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"],
                                      sets[0].u.dtype)
    ws = [ssm.alloc_workspace(need, dev) for _ in range(nsets)]

    def launch(i):
        x = sets[i]
        ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias,
                             out=outs[i], h_final=hfs[i], workspace=ws[i])

    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        for i in range(nsets):
            launch(i)  # eager warm-up (also loads the module)
    torch.cuda.synchronize(dev)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                launch(i % nsets)
        return g

    full = capture(nsets)
    rem = steps % nsets
    part = capture(rem) if rem else None
    for _ in range(max(1, math.ceil(warmup / nsets))):
        full.replay()
    torch.cuda.synchronize(dev)
    t_pre = time.time()
    if preroll_s > 0:  # keeps the GPU busy while the clock sampler settles
        while time.time() - t_pre < preroll_s:
            full.replay()
            torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps // nsets):
            full.replay()
        if part is not None:
            part.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    ms = e0.elapsed_time(e1)
    ms_pass = None
    if pass_reps > 0:
        pb = torch.cuda.Event(enable_timing=True)
        pe = torch.cuda.Event(enable_timing=True)
        tot = 0.0
        with torch.cuda.stream(stream):
            pb.record(stream)  # creates the events on this device
            pe.record(stream)
            ssm.set_pass_timer(pb, pe)
            try:
                for i in range(pass_reps):
                    launch(i % nsets)
                    torch.cuda.synchronize(dev)
                    tot += pb.elapsed_time(pe)
            finally:
                ssm.set_pass_timer()
        ms_pass = tot / pass_reps
    plan = ssm.scan_plan(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"], sets[0].u.dtype)
    return dict(ms_total=ms, ms_per_launch=ms / steps, bytes_per_step=nbytes, nsets=nsets, plan=plan,
                ms_fused_pass=ms_pass,
                t_window=(t_pre, t_end), upd_per_step=w["batch"] * w["dim"] * w["seqlen"] * w["dstate"],
                bdl_per_step=w["batch"] * w["dim"] * w["seqlen"])


def bench_scan_e2e(ssm, I, torch, w, steps, warmup):
    """End to end through the public API: every step copies its inputs from
    pinned host memory to the device, runs the chunked scan and copies y back
    to pinned host memory.  Steps are pipelined over three streams (copy-in,
    compute, copy-out) with two device buffer sets, so that the copies of one
    step overlap the compute and copies of its neighbours; every copy of every
    step is inside the timed region."""
    dev = torch.device("cuda")
    x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"], io=w["io"],
                           recipe=w["recipe"], seed=100, device="cpu")
    names = ["u", "delta", "z", "B", "C"]
    host = {n: getattr(x, n).pin_memory() for n in names}
    params = {n: getattr(x, n).to(dev) for n in ["A", "D", "dt_bias"]}
    nbuf = 2
    devt = [{n: torch.empty_like(host[n], device=dev) for n in names} for _ in range(nbuf)]
    y_dev = [torch.empty_like(devt[0]["u"]) for _ in range(nbuf)]
    y_host = [torch.empty_like(host["u"]).pin_memory() for _ in range(nbuf)]
    hf_dev = [torch.empty((w["batch"], w["dim"], w["dstate"]), dtype=torch.float32, device=dev)
              for _ in range(nbuf)]
    need = ssm.chunked_workspace_size(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"],
                                      host["u"].dtype)
    ws = [ssm.alloc_workspace(need, dev) for _ in range(nbuf)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = y_host[0].numel() * y_host[0].element_size()
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]
    ev_cmp = [torch.cuda.Event() for _ in range(nbuf)]
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]
    for e in ev_cmp + ev_out:
        e.record(torch.cuda.current_stream(dev))

    def step(i):
        k = i % nbuf
        s_in.wait_event(ev_cmp[k])           # the compute that last read this buffer set is done
        with torch.cuda.stream(s_in):
            for n in names:
                devt[k][n].copy_(host[n], non_blocking=True)
            ev_in[k].record(s_in)
        s_cmp.wait_event(ev_in[k])
        s_cmp.wait_event(ev_out[k])          # y of this buffer set has been read back
        with torch.cuda.stream(s_cmp):
            d = devt[k]
            ssm.scan_fwd_chunked(d["u"], d["delta"], params["A"], d["B"], d["C"], z=d["z"], D=params["D"],
                                 dt_bias=params["dt_bias"], out=y_dev[k], h_final=hf_dev[k], workspace=ws[k])
            ev_cmp[k].record(s_cmp)
        s_out.wait_event(ev_cmp[k])
        with torch.cuda.stream(s_out):
            y_host[k].copy_(y_dev[k], non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_stream(s_in)
    s_out.wait_stream(s_in)
    for i in range(steps):
        step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    return dict(ms_per_step=ms / steps, h2d=h2d, d2h=d2h)


def bench_decode_device(ssm, I, torch, w, steps, warmup):
    """Decode step on the full batch; states rotate so the 80 MiB state is
    read from HBM each step (cold); also a warm figure on one state."""
    dev = torch.device("cuda")
    props = torch.cuda.get_device_properties(dev)
    b, d, n = w["batch"], w["dim"], w["dstate"]
    per = I.compulsory_bytes_decode(b, d, n)
    nsets = n_rotating_sets(per, props.L2_cache_size)
    prm = I.decode_params(d, n, recipe=w["recipe"], seed=0, device=dev)
    states = [I.make_decode_state(b, d, n, seed=s, device=dev) for s in range(nsets)]
    toks = [I.make_decode_token(b, d, n, s, io=w["io"], recipe=w["recipe"], seed=0, device=dev)
            for s in range(nsets)]
    ys = [torch.empty((b, d), dtype=toks[0]["u"].dtype, device=dev) for _ in range(nsets)]

    def launch(i, k):
        t = toks[k]
        ssm.state_update(states[i], t["u"], t["delta"], prm["A"], t["B"], t["C"], z=t["z"],
                         D=prm["D"], dt_bias=prm["dt_bias"], out=ys[k])

    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    res = {}
    for mode in ("cold", "warm"):
        with torch.cuda.stream(stream):
            for i in range(nsets):
                launch(i if mode == "cold" else 0, i)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsets):
                launch(i if mode == "cold" else 0, i)
        reps = max(1, steps // nsets)
        for _ in range(max(1, math.ceil(warmup / nsets))):
            g.replay()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / (reps * nsets)
        res[mode] = dict(us_per_step=ms * 1e3, tokens_per_s=b / (ms * 1e-3),
                         state_gbs=per / (ms * 1e-3) / 1e9, launches=reps * nsets)
    return res


def bench_graph(torch, launch, nsets, reps, warmup=3):
    """Mean device time of one launch: CUDA events around `reps` replays of a
    CUDA graph that calls launch(i) for i in range(nsets)."""
    dev = torch.device("cuda")
    stream = torch.cuda.Stream(dev)
    stream.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(stream):
        for i in range(nsets):
            launch(i)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(nsets):
            launch(i)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / (reps * nsets)


def bench_conv(ssm, I, torch, peaks, width=4):
    """The short causal convolution (+ silu) in front of the scan, on the
    three scan shapes (bf16), and its decode step on the decode shape: device
    time per launch over rotating inputs (> 3x L2)."""
    dev = torch.device("cuda")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}
    for name in ("scan_bf16_b2_d1536_l2048", "scan_bf16_b8_d2048_l4096", "scan_bf16_b1_d5120_l65536_final_state"):
        w = I.WORKLOADS[name]
        nbytes = I.compulsory_bytes_conv(w["batch"], w["dim"], w["seqlen"], w["io"])
        nsets = n_rotating_sets(nbytes, l2)
        ins = [I.make_conv_inputs(w["batch"], w["dim"], w["seqlen"], width, io=w["io"], seed=s, device=dev)
               for s in range(nsets)]
        outs = [torch.empty_like(c["x"]) for c in ins]

        def launch(i, ins=ins, outs=outs):
            c = ins[i]
            ssm.causal_conv1d(c["x"], c["w"], c["bias"], out=outs[i])

        ms = bench_graph(torch, launch, nsets, reps=max(3, 60 // nsets))
        gbs = nbytes / (ms * 1e-3) / 1e9
        key = "conv1d_w%d_%s" % (width, name.replace("scan_", "").replace("_final_state", ""))
        res[key] = dict(GBps=round(gbs, 1), us_per_launch=round(ms * 1e3, 2),
                        frac_of_hbm_measured=round(gbs / peaks["hbm_gbs"], 4))
        del ins, outs
    wd = I.WORKLOADS[DECODE]
    b, d = wd["batch"], wd["dim"]
    es = 2
    per = b * d * es * (2 * (width - 1) + 2)  # state read + written, token read, out written
    nsets = n_rotating_sets(per, l2)
    ins = [I.make_conv_inputs(b, d, 1, width, io=wd["io"], seed=s, device=dev, with_prev=True) for s in range(nsets)]
    toks = [c["x"][:, :, 0].contiguous() for c in ins]
    outs = [torch.empty_like(t) for t in toks]

    def launch_dec(i):
        c = ins[i]
        ssm.causal_conv1d_update(c["x_prev"], toks[i], c["w"], c["bias"], out=outs[i])

    ms = bench_graph(torch, launch_dec, nsets, reps=max(3, 200 // nsets))
    res["conv1d_update_w%d_b%d_d%d" % (width, b, d)] = dict(
        us_per_step=round(ms * 1e3, 3), GBps=round(per / (ms * 1e-3) / 1e9, 1),
        frac_of_hbm_measured=round(per / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4))
    return res


VARLEN_SHAPE = dict(dim=1536, dstate=16, nseq=64, mean=64)   # serving prefill: 64 sequences, mean 64 tokens


def bench_varlen(ssm, I, torch, peaks):
    """Packed variable-length scan (64 bf16 sequences of mixed lengths, 1536
    channels) and the decode step on a pool of state slots (the decode shape,
    rows mapped to a permutation of the slots): device time per launch over
    rotating inputs (> 3x L2)."""
    dev = torch.device("cuda")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}
    vs = VARLEN_SHAPE
    lengths = I.varlen_lengths(vs["nseq"], vs["mean"], seed=0)
    T = sum(lengths)
    nbytes = I.compulsory_bytes_scan(1, vs["dim"], vs["dstate"], T, 1, "bf16")
    nsets = n_rotating_sets(nbytes, l2)
    # Rows padded to a multiple of 8 steps (the 16-byte packet) after the last sequence.
    ins = [I.make_varlen_inputs(vs["dim"], vs["dstate"], lengths, io="bf16", seed=s, device=dev, with_h0=True,
                                row_multiple=8) for s in range(nsets)]
    outs = [torch.empty_like(x["u"]) for x in ins]
    hfs = [torch.empty((vs["nseq"], vs["dim"], vs["dstate"]), device=dev) for _ in ins]

    def launch(i):
        x = ins[i]
        ssm.scan_fwd_varlen(x["u"], x["delta"], x["A"], x["B"], x["C"], x["cu_seqlens"], z=x["z"], D=x["D"],
                            dt_bias=x["dt_bias"], h0=x["h0"], out=outs[i], h_final=hfs[i])

    ms = bench_graph(torch, launch, nsets, reps=max(3, 60 // nsets))
    gbs = nbytes / (ms * 1e-3) / 1e9
    res["scan_varlen_bf16_d%d_n%d_mean%d" % (vs["dim"], vs["nseq"], vs["mean"])] = dict(
        tokens=T, GBps=round(gbs, 1), us_per_launch=round(ms * 1e3, 2),
        frac_of_hbm_measured=round(gbs / peaks["hbm_gbs"], 4))
    del ins, outs, hfs
    wd = I.WORKLOADS[DECODE]
    b, d, n = wd["batch"], wd["dim"], wd["dstate"]
    per = I.compulsory_bytes_decode(b, d, n)
    nsets = n_rotating_sets(per, l2)
    prm = I.decode_params(d, n, recipe=wd["recipe"], seed=0, device=dev)
    pools = [I.make_decode_state(b, d, n, seed=s, device=dev) for s in range(nsets)]
    g = torch.Generator().manual_seed(0)
    perm = torch.randperm(b, generator=g).to(torch.int32).to(dev)
    toks = [I.make_decode_token(b, d, n, s, io=wd["io"], recipe=wd["recipe"], seed=0, device=dev)
            for s in range(nsets)]
    ys = [torch.empty((b, d), dtype=toks[0]["u"].dtype, device=dev) for _ in range(nsets)]

    def launch_dec(i):
        t = toks[i]
        ssm.state_update(pools[i], t["u"], t["delta"], prm["A"], t["B"], t["C"], z=t["z"], D=prm["D"],
                         dt_bias=prm["dt_bias"], out=ys[i], state_indices=perm)

    ms = bench_graph(torch, launch_dec, nsets, reps=max(3, 200 // nsets))
    res["decode_pooled_b%d_d%d" % (b, d)] = dict(
        us_per_step=round(ms * 1e3, 3), state_GBps=round(per / (ms * 1e-3) / 1e9, 1),
        frac_of_hbm_measured=round(per / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4))
    return res


def bench_ssd(ssm, I, torch, peaks, name="ssd_bf16_b2_h64_p64_n128_l2048"):
    """The SSD (Mamba-2) layer on the tensor cores: device time per launch over
    rotating inputs (> 3x L2); compulsory bytes per second and the chunked
    evaluation's dense-contraction FLOPs against the measured bf16 tensor peak."""
    dev = torch.device("cuda")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    w = I.WORKLOADS[name]
    args = (w["batch"], w["nheads"], w["headdim"], w["dstate"], w["seqlen"], w["ngroups"])
    nbytes = I.compulsory_bytes_ssd(*args)
    flops = I.flops_ssd_chunked(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["seqlen"])
    nsets = n_rotating_sets(nbytes, l2)
    xs = [I.make_ssd_inputs(*args, seed=s, device=dev) for s in range(nsets)]
    ys = [torch.empty_like(x["x"]) for x in xs]
    hfs = [torch.empty((w["batch"], w["nheads"] * w["headdim"], w["dstate"]), device=dev) for _ in xs]

    def launch(i):
        x = xs[i]
        ssm.ssd_fwd(x["x"], x["delta"], x["A"], x["B"], x["C"], z=x["z"], D=x["D"], dt_bias=x["dt_bias"],
                    headdim=w["headdim"], out=ys[i], h_final=hfs[i])

    ms = bench_graph(torch, launch, nsets, reps=max(3, 60 // nsets))
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks.get("bf16_tflops", 1800.0)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del xs, ys, hfs
    return {name: dict(us_per_launch=round(ms * 1e3, 2), GBps=round(gbs, 1),
                       frac_of_hbm_measured=round(gbs / peaks["hbm_gbs"], 4), TFLOPs=round(tflops, 1),
                       roofline={"bound": "tensor", "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
                                 "frac": round(tflops / peak, 4),
                                 "peak_source": "bf16_tflops of MEASURED_PEAKS.json (cuBLAS bf16 GEMM, burst)"},
                       kernel="ssd_fwd_kernel (tcgen05.mma, TMEM accumulators, TMA)")}


def bench_bwd(ssm, I, torch, peaks, names=("scan_bf16_b2_d1536_l2048", "scan_bf16_b8_d2048_l4096",
                                           "scan_bf16_b2_d1536_l2048_n256")):
    """Backward pass (every gradient, no final-state gradient) on the scan
    shapes: device time per call over rotating inputs (> 3x L2)."""
    dev = torch.device("cuda")
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}
    for name in names:
        w = I.WORKLOADS[name]
        b, d, n, L, G = w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"]
        nbytes = I.compulsory_bytes_bwd(b, d, n, L, G, w["io"])
        nsets = n_rotating_sets(nbytes, l2)
        xs = [I.make_scan_inputs(b, d, n, L, G, io=w["io"], recipe=w["recipe"], seed=s, device=dev)
              for s in range(nsets)]
        dys = [I.make_scan_inputs(b, d, n, L, G, io=w["io"], recipe=w["recipe"], seed=100 + s, device=dev).u
               for s in range(nsets)]
        outs = [None] * nsets
        ws = ssm.alloc_workspace(ssm.bwd_workspace_size(b, d, n, L, G, xs[0].u.dtype), dev)

        def launch(i):
            x = xs[i]
            outs[i] = ssm.scan_bwd(x.u, x.delta, x.A, x.B, x.C, dys[i], z=x.z, D=x.D, dt_bias=x.dt_bias,
                                   out=outs[i], workspace=ws, want_dh0=False)

        for i in range(nsets):
            launch(i)  # allocates the outputs outside the captured graph
        ms = bench_graph(torch, launch, nsets, reps=max(3, 40 // nsets))
        gbs = nbytes / (ms * 1e-3) / 1e9
        res["scan_bwd_" + name[len("scan_"):]] = dict(
            GBps=round(gbs, 1), us_per_launch=round(ms * 1e3, 2), frac_of_hbm_measured=round(gbs / peaks["hbm_gbs"], 4),
            Gupd_per_s=round(b * d * n * L / (ms * 1e-3) / 1e9, 1))
        del xs, dys, outs, ws
    return res


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

# Channels of the headline workload in one oracle sample: the oracle's cost
# per channel does not depend on the values, so a sample of channels with the
# workload's per-channel shape (L, N) and recipe is timed instead of all 5120.
ORACLE_SAMPLE_CHANNELS = 512


def oracle_sample_inputs(I, w, nd):
    """fp64 inputs of `nd` channels with the workload's batch, L, N, groups and
    recipe (seed 0), for timing the oracle."""
    return I.make_scan_inputs(w["batch"], nd, w["dstate"], w["seqlen"], w["ngroups"], io=w["io"],
                              recipe=w["recipe"], seed=0, device="cpu").as_f64()


def oracle_baseline(I, w, budget_s=10.0):
    import oracle
    nd = min(w["dim"], ORACLE_SAMPLE_CHANNELS)
    x = oracle_sample_inputs(I, w, nd)
    threads = oracle.default_threads()
    nbytes = I.compulsory_bytes_scan(w["batch"], nd, w["dstate"], w["seqlen"], w["ngroups"], w["io"])
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.scan(**x, nthreads=threads, return_final_state=True)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    gbs = reps * nbytes / el / 1e9
    return dict(value=gbs, unit="GB/s", cores=threads, kind="oracle",
                sample=f"{reps} passes over {nd} of the {w['dim']} channels of the {HEADLINE} workload "
                       f"(batch {w['batch']}, L {w['seqlen']}, N {w['dstate']}; fp64 C oracle, {threads} threads "
                       f"over channels) in {el:.1f} s",
                seconds=el, passes=reps)


# ---------------------------------------------------------------------------

def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    from selective_state_space_109_b300 import inputs as I
    from selective_state_space_109_b300 import ssm

    w = I.WORKLOADS[HEADLINE]
    peaks, peak_src = measured_peaks()
    alu = ssm.probe_alu_rates(dev)  # the arithmetic pipes' rates on this GPU, for the roofline
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    r = bench_scan_device(ssm, I, torch, w, args.steps, args.warmup, pass_reps=max(3, min(args.steps, 20)))
    torch.cuda.synchronize(dev)
    barrier(world)
    sampler.stop()
    clocks = sampler.summary(*r["t_window"])
    ms_total = max_over_ranks(r["ms_total"], world, dev)
    total_bytes = sum_over_ranks(r["bytes_per_step"] * args.steps, world, dev)
    value = total_bytes / (ms_total * 1e-3) / 1e9
    per_launch_s = r["ms_per_launch"] * 1e-3
    achieved = r["bytes_per_step"] / per_launch_s / 1e9

    e2e = bench_scan_e2e(ssm, I, torch, w, max(3, min(args.steps, 50)), 3)
    e2e_ms = max_over_ranks(e2e["ms_per_step"], world, dev)
    e2e_value = sum_over_ranks(r["bytes_per_step"], world, dev) / (e2e_ms * 1e-3) / 1e9

    dec = None
    if not args.skip_decode:
        dec = bench_decode_device(ssm, I, torch, I.WORKLOADS[DECODE], max(args.steps, 64), args.warmup)

    extra = {}
    if not args.skip_extra and world == 1:
        for name in ("scan_bf16_b2_d1536_l2048", "scan_bf16_b8_d2048_l4096",
                     "scan_bf16_b2_d1536_l2048_n64", "scan_bf16_b2_d1536_l2048_n128",
                     "scan_bf16_b2_d1536_l2048_n256"):
            wx = I.WORKLOADS[name]
            rx = bench_scan_device(ssm, I, torch, wx, max(4, min(args.steps, 40)), 3, preroll_s=0.0)
            extra[name] = dict(GBps=round(rx["bytes_per_step"] / (rx["ms_per_launch"] * 1e-3) / 1e9, 1),
                               us_per_launch=round(rx["ms_per_launch"] * 1e3, 2),
                               frac_of_hbm_measured=round(rx["bytes_per_step"] / (rx["ms_per_launch"] * 1e-3)
                                                          / 1e9 / peaks["hbm_gbs"], 4),
                               Gupd_per_s=round(rx["upd_per_step"] / (rx["ms_per_launch"] * 1e-3) / 1e9, 1),
                               plan=rx["plan"])
        # The time-segmented variant (time split inside each warp by an
        # associative scan over (Abar, Bbar x) pairs), measured beside the
        # default plans it loses to.
        for name, lanes, seg in (("scan_bf16_b2_d1536_l2048", 4, 4),
                                 ("scan_bf16_b1_d5120_l65536_final_state", 4, 2)):
            os.environ["SSM_FORCE_SEG"], os.environ["SSM_FORCE_LANES"] = str(seg), str(lanes)
            try:
                wx = I.WORKLOADS[name]
                rx = bench_scan_device(ssm, I, torch, wx, max(4, min(args.steps, 20)), 3, preroll_s=0.0)
            finally:
                del os.environ["SSM_FORCE_SEG"], os.environ["SSM_FORCE_LANES"]
            extra[f"{name}_segmented_l{lanes}s{seg}"] = dict(
                GBps=round(rx["bytes_per_step"] / (rx["ms_per_launch"] * 1e-3) / 1e9, 1),
                us_per_launch=round(rx["ms_per_launch"] * 1e3, 2),
                Gupd_per_s=round(rx["upd_per_step"] / (rx["ms_per_launch"] * 1e-3) / 1e9, 1),
                plan={"lanes": lanes, "segments": seg, "kernels": 1, "staged": True})
        extra.update(bench_conv(ssm, I, torch, peaks))
        extra.update(bench_varlen(ssm, I, torch, peaks))
        extra.update(bench_bwd(ssm, I, torch, peaks))
        extra.update(bench_ssd(ssm, I, torch, peaks))

    base = None
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        base = oracle_baseline(I, w, budget_s=args.cpu_seconds)

    if rank != 0:
        return
    sm_max = peaks.get("sm_max_mhz", 2032.0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_achieved = r["upd_per_step"] / per_launch_s / 1e9
    upd_per_sm_ns = min(alu["ex2_per_sm_ns"], alu["ffma_per_sm_ns"] / 4.0)
    alu_peak = sms * upd_per_sm_ns  # Gupd/s
    rec = ncu_record("scan_chunked_call/" + HEADLINE, r["plan"])
    traffic = rec.get("dram_bytes_per_launch") if rec else None
    # The dominant kernel is the fused pass (the kernel that writes y): the
    # largest share of the call in the committed ncu launch record, and the
    # call's only kernel on single-pass plans.  Its duration is measured live
    # (CUDA events the library records around its launch); its algorithmic
    # work is one pass's state updates (and the call's compulsory bytes).
    fused_name, share = None, None
    if rec and rec.get("kernel_ns"):
        tot = sum(rec["kernel_ns"].values())
        fused_name, ns = max(rec["kernel_ns"].items(), key=lambda kv: kv[1])
        share = ns / tot
    t_fused = r["ms_fused_pass"] * 1e-3
    fused_alu = r["upd_per_step"] / t_fused / 1e9
    fused_traffic = rec["kernels"].get(fused_name) if rec and fused_name else None
    if isinstance(fused_traffic, dict):
        fused_traffic = fused_traffic.get("dram_bytes")
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_total / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": HEADLINE, "batch": w["batch"], "dim": w["dim"], "dstate": w["dstate"],
                   "seqlen": w["seqlen"], "ngroups": w["ngroups"], "io": "bf16", "state": "f32",
                   "final_state": bool(w.get("final_state", False)),
                   "recipe": w["recipe"], "l2": f"inputs larger than L2: {r['nsets']} rotating input sets "
                                                f"({r['nsets'] * r['bytes_per_step'] / 1e6:.0f} MB)",
                   "timing": "CUDA events around a CUDA graph of the K launches",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "frac_of_hbm": round(value / world / peaks["hbm_gbs"], 4),
        "tokens_channels_per_s": round(r["bdl_per_step"] / per_launch_s, 1),
        "roofline": {"bound": "alu", "achieved": round(fused_alu, 1), "peak": round(alu_peak, 1),
                     "unit": "Gupd/s", "frac": round(fused_alu / alu_peak, 4), "traffic": fused_traffic,
                     "kernel": ("scan_tma_kernel fused pass (ScanMode::Full), the dominant kernel of the "
                                "chunked call" if r["plan"]["kernels"] > 1
                                else "scan_ws_kernel fused pass (the call's only kernel)"),
                     "us_per_launch": round(t_fused * 1e6, 1),
                     "timing": f"CUDA events recorded by the library around the fused pass's launch, mean of "
                               f"{max(3, min(args.steps, 20))} calls over the rotating input sets",
                     "share_of_call_ncu": round(share, 4) if share is not None else None,
                     "plan": r["plan"],
                     "peak_basis": (f"measured live by ssm_probe_alu_rates: MUFU.EX2 "
                                    f"{alu['ex2_per_sm_ns']:.2f} and fp32 FMA {alu['ffma_per_sm_ns']:.2f} per SM "
                                    f"per ns; one ex2 and four FMA-pipe operations per state update -> "
                                    f"{upd_per_sm_ns:.2f} updates per SM per ns x {sms} SMs (nominal: "
                                    f"{NOMINAL_UPDATES_PER_SM_CLK:.0f}/SM/clk x {sm_max:.0f} MHz = "
                                    f"{sms * sm_max * 1e-3 * NOMINAL_UPDATES_PER_SM_CLK:.0f} Gupd/s)"),
                     "update_mix_ceiling": {"achieved_by_bare_mix": round(alu["mix_updates_per_sm_ns"] * sms, 1),
                                            "unit": "Gupd/s",
                                            "frac_of_peak": round(alu["mix_updates_per_sm_ns"] / upd_per_sm_ns, 4),
                                            "note": "the scan's per-state instruction mix alone (no per-step "
                                                    "scalars, loads or stores), eight warps per scheduler"},
                     "whole_call": {"achieved": round(alu_achieved, 1), "frac": round(alu_achieved / alu_peak, 4),
                                    "traffic": traffic,
                                    "note": "the whole chunked call (summary, carry and fused passes) against "
                                            "one pass's updates; the summary pass recomputes the decays of "
                                            "all chunks but the last"}},
        "hbm_roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "peak_source": peak_src, "traffic": traffic,
                         "nominal_peak": NOMINAL_HBM_GBS,
                         "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": args.steps * r["plan"]["kernels"],
        "clocks": clocks,
    }
    if dec is not None:
        out["decode"] = {"workload": DECODE, "tokens_per_s": round(dec["cold"]["tokens_per_s"], 1),
                         "us_per_step": round(dec["cold"]["us_per_step"], 3),
                         "state_GBps": round(dec["cold"]["state_gbs"], 1),
                         "frac_of_hbm": round(dec["cold"]["state_gbs"] / peaks["hbm_gbs"], 4),
                         "frac_of_nominal_hbm": round(dec["cold"]["state_gbs"] / NOMINAL_HBM_GBS, 4),
                         "warm_l2_us_per_step": round(dec["warm"]["us_per_step"], 3),
                         "warm_l2_tokens_per_s": round(dec["warm"]["tokens_per_s"], 1)}
    if extra:
        out["other_workloads"] = extra
    if base is not None:
        out["cpu_baseline"] = {k: base[k] for k in ("value", "unit", "cores", "kind", "sample")}
        out["cpu_baseline"]["value"] = round(base["value"], 3)
    print(json.dumps(out), flush=True)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from selective_state_space_109_b300 import inputs as I
    w = I.WORKLOADS[HEADLINE]
    import oracle
    threads = oracle.default_threads()
    # Each step: the oracle over a bounded sample (a block of channels with the
    # workload's per-channel shape and recipe), sized so that K + W steps end
    # within a few minutes.
    nd = max(1, min(w["dim"], int(os.environ.get("SSM_REF_CHANNELS", "256"))))
    sub = oracle_sample_inputs(I, w, nd)
    sub_bytes = I.compulsory_bytes_scan(w["batch"], nd, w["dstate"], w["seqlen"], w["ngroups"], w["io"])
    for _ in range(args.warmup):
        oracle.scan(**sub, nthreads=threads, return_final_state=True)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan(**sub, nthreads=threads, return_final_state=True)
    el = time.perf_counter() - t0
    value = sub_bytes * args.steps / el / 1e9
    sample = (f"{nd} of {w['dim']} channels x batch {w['batch']} x L {w['seqlen']} per step "
              f"(the workload's per-channel shape and recipe, seed 0)")
    out = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": HEADLINE, "batch": w["batch"], "dim": w["dim"], "dstate": w["dstate"],
                      "seqlen": w["seqlen"], "ngroups": w["ngroups"], "io": "bf16-rounded values in fp64",
                      "final_state": True},
           "impl": "reference",
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_profile_case(args):
    """W + K eager launches of one workload on one input set, nothing else:
    the command profiled by ncu."""
    import torch
    from selective_state_space_109_b300 import inputs as I
    from selective_state_space_109_b300 import ssm
    dev = torch.device("cuda")
    if args.profile.startswith("conv1d_"):
        # conv1d_w4_<scan workload>: the short convolution on that scan shape;
        # conv1d_update_w4_<decode workload>: its decode step on that shape.
        upd = args.profile.startswith("conv1d_update_")
        rest = args.profile[len("conv1d_update_w") if upd else len("conv1d_w"):]
        width, name = int(rest.split("_", 1)[0]), rest.split("_", 1)[1]
        w = I.WORKLOADS[name]
        L = 1 if upd else w["seqlen"]
        c = I.make_conv_inputs(w["batch"], w["dim"], L, width, io=w["io"], device=dev, with_prev=upd)
        if upd:
            tok = c["x"][:, :, 0].contiguous()
            for _ in range(args.warmup + args.steps):
                ssm.causal_conv1d_update(c["x_prev"], tok, c["w"], c["bias"])
        else:
            out = torch.empty_like(c["x"])
            for _ in range(args.warmup + args.steps):
                ssm.causal_conv1d(c["x"], c["w"], c["bias"], out=out)
        torch.cuda.synchronize(dev)
        print(json.dumps({"profile_case": args.profile, "launches": args.warmup + args.steps}))
        return
    if args.profile == "scan_varlen":
        vs = VARLEN_SHAPE
        x = I.make_varlen_inputs(vs["dim"], vs["dstate"], I.varlen_lengths(vs["nseq"], vs["mean"], seed=0),
                                 io="bf16", device=dev, with_h0=True, row_multiple=8)
        for _ in range(args.warmup + args.steps):
            ssm.scan_fwd_varlen(x["u"], x["delta"], x["A"], x["B"], x["C"], x["cu_seqlens"], z=x["z"], D=x["D"],
                                dt_bias=x["dt_bias"], h0=x["h0"], return_final_state=True)
        torch.cuda.synchronize(dev)
        print(json.dumps({"profile_case": args.profile, "launches": args.warmup + args.steps}))
        return
    if args.profile.startswith("ssd_"):
        w = I.WORKLOADS[args.profile]
        x = I.make_ssd_inputs(w["batch"], w["nheads"], w["headdim"], w["dstate"], w["seqlen"], w["ngroups"],
                              device=dev)
        y = torch.empty_like(x["x"])
        for _ in range(args.warmup + args.steps):
            ssm.ssd_fwd(x["x"], x["delta"], x["A"], x["B"], x["C"], z=x["z"], D=x["D"], dt_bias=x["dt_bias"],
                        headdim=w["headdim"], out=y)
        torch.cuda.synchronize(dev)
        print(json.dumps({"profile_case": args.profile, "launches": args.warmup + args.steps}))
        return
    if args.profile.startswith("scan_bwd_"):
        # scan_bwd_<scan workload>: the backward pass on that shape.
        w = I.WORKLOADS["scan_" + args.profile[len("scan_bwd_"):]]
        x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"], io=w["io"],
                               recipe=w["recipe"], device=dev)
        dy = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"], io=w["io"],
                                recipe=w["recipe"], seed=1, device=dev).u
        out = None
        for _ in range(args.warmup + args.steps):
            out = ssm.scan_bwd(x.u, x.delta, x.A, x.B, x.C, dy, z=x.z, D=x.D, dt_bias=x.dt_bias, out=out)
        torch.cuda.synchronize(dev)
        print(json.dumps({"profile_case": args.profile, "launches": args.warmup + args.steps}))
        return
    w = I.WORKLOADS[args.profile]
    if w["kind"] == "decode":
        prm = I.decode_params(w["dim"], w["dstate"], recipe=w["recipe"], device=dev)
        st = I.make_decode_state(w["batch"], w["dim"], w["dstate"], device=dev)
        tok = I.make_decode_token(w["batch"], w["dim"], w["dstate"], 0, io=w["io"], recipe=w["recipe"],
                                  device=dev)
        for _ in range(args.warmup + args.steps):
            ssm.state_update(st, tok["u"], tok["delta"], prm["A"], tok["B"], tok["C"], z=tok["z"],
                             D=prm["D"], dt_bias=prm["dt_bias"])
    else:
        # The same call the benchmark times: the chunked entry point with a
        # preallocated workspace and final-state buffer.
        x = I.make_scan_inputs(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"], io=w["io"],
                               recipe=w["recipe"], device=dev)
        y = torch.empty_like(x.u)
        hf = torch.empty((w["batch"], w["dim"], w["dstate"]), dtype=torch.float32, device=dev)
        ws = ssm.alloc_workspace(ssm.chunked_workspace_size(w["batch"], w["dim"], w["dstate"], w["seqlen"],
                                                            w["ngroups"], x.u.dtype), dev)
        for _ in range(args.warmup + args.steps):
            ssm.scan_fwd_chunked(x.u, x.delta, x.A, x.B, x.C, z=x.z, D=x.D, dt_bias=x.dt_bias, out=y,
                                 h_final=hf, workspace=ws)
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile_case": args.profile, "launches": args.warmup + args.steps}))


def write_traffic(csv_path, workload):
    """Reads an ncu --csv metrics log (dram__bytes_read.sum, dram__bytes_write.sum
    per launch) of `bench.py --profile <workload>` and records the DRAM bytes of
    one chunked call (all of its kernels) in profiles/traffic.json, keyed by the
    current kernel-source hash so that a later kernel change voids it."""
    import csv
    per_kernel = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(f) if r]
    hdr = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    cols = rows[hdr]
    launches, times = {}, {}
    for r in rows[hdr + 1:]:
        if len(r) != len(cols):
            continue
        d = dict(zip(cols, r))
        if not any(k in d["Kernel Name"] for k in ("scan_tma_kernel", "scan_fwd_kernel", "scan_carry_kernel",
                                                    "scan_ws_kernel")):
            continue
        name = d["Kernel Name"].split("(")[0]
        unit = d.get("Metric Unit", "byte")
        key = (d["ID"], name)
        launches.setdefault(key, 0.0)
        if d["Metric Name"] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}.get(unit, 1)
            launches[key] += float(d["Metric Value"].replace(",", "")) * scale
        elif d["Metric Name"] == "gpu__time_duration.sum":
            scale = {"ns": 1, "nsecond": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6}.get(unit, 1)
            times[key] = float(d["Metric Value"].replace(",", "")) * scale
    per_time = {}
    for (i, name), b in launches.items():
        per_kernel.setdefault(name, []).append(b)
        if (i, name) in times:
            per_time.setdefault(name, []).append(times[(i, name)])
    kernels = {k: sum(v) / len(v) for k, v in per_kernel.items()}
    kernel_ns = {k: sum(v) / len(v) for k, v in per_time.items()}
    from selective_state_space_109_b300 import inputs as I
    from selective_state_space_109_b300 import ssm
    w = I.WORKLOADS[workload]
    plan = ssm.scan_plan(w["batch"], w["dim"], w["dstate"], w["seqlen"], w["ngroups"], I.io_torch_dtype(w["io"]))
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        data = {}
    data["scan_chunked_call/" + workload] = {
        "dram_bytes_per_launch": round(sum(kernels.values())),
        "kernels": {k: round(v) for k, v in kernels.items()},
        "kernel_ns": {k: round(v) for k, v in kernel_ns.items()},
        "source_hash": kernel_source_hash(),
        "plan": plan,
        "from": os.path.basename(csv_path)}
    with open(path, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
    print(json.dumps(data["scan_chunked_call/" + workload]))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-extra", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", metavar="WORKLOAD", default=None,
                    help="only run W+K launches of one named workload (for ncu)")
    ap.add_argument("--write-traffic", metavar="NCU_CSV", default=None,
                    help="record the DRAM bytes of the headline call from an ncu metrics log")
    args = ap.parse_args(argv)
    if args.write_traffic:
        write_traffic(args.write_traffic, args.profile or HEADLINE)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
