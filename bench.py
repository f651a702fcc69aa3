#!/usr/bin/env python
"""Throughput of the gated delta rule kernels on one GB300 (or N, weak scaling).

One step = one chunked prefill of the Qwen3-Next-shaped workload (batch 1,
4096 tokens, 16 key heads over 32 value heads, 128 x 128 heads, bf16 q/k/v,
fp32 decays/beta, zero initial state) through the C ABI.  The JSON line's
``value`` is prefill tokens/s over all ranks; the decode step (B=256, state
[256,32,128,128] fp32 in place), the packed varlen prefill, the long-context
prefill and the per-token state emission are measured in the same run and
reported as sub-objects with their own rooflines.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Inputs are seeded synthetic tensors resident in HBM before timing; between
timed prefill iterations a 256 MiB buffer is written to flush the 129 MB L2
(the decode state, 512 MiB, is larger than L2 by itself).  Kernel times are
CUDA-event times on the launching stream.  ``--impl reference`` times the fp64
CPU oracle on the host cores instead (bounded sample of the same workload).
"""
import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "GDN prefill tokens/s and decode steps/s (1 GB300) + % of roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def measured_traffic(profile, source):
    """DRAM bytes per call (dram__bytes_read.sum + dram__bytes_write.sum) from the ncu
    summary in profiles/, or None when the kernel source changed since the capture (the
    summary records the sha256 of the source it profiled)."""
    import hashlib
    try:
        fields = {}
        with open(os.path.join(ROOT, "profiles", profile)) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 2 and parts[0] in ("traffic_bytes_per_call", "source_sha256"):
                    fields[parts[0]] = parts[1]
        with open(os.path.join(ROOT, "gated_deltanet_mixer_delta_gb300", "csrc", source), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except OSError:
        return None
    if fields.get("source_sha256") != digest or "traffic_bytes_per_call" not in fields:
        return None
    return int(fields["traffic_bytes_per_call"])


# ---------------------------------------------------------------- algorithmic work
def prefill_bytes(B_tokens, HK, HV, D, elt, n_states_in, n_states_out, states_tokens=0):
    """Bytes a prefill must move at least once: q, k, v, o (elt bytes), g and beta (fp32),
    initial states read, final states written, per-token states written."""
    io = B_tokens * (2 * HK * D * elt + 2 * HV * D * elt + 2 * HV * 4)
    st = (n_states_in + n_states_out) * HV * D * D * 4
    return io + st + states_tokens * HV * D * D * 4


def prefill_flops(tokens, HV, D, C=64):
    """Chunked-form flops per token per value head: five C x C x D and three C x D x D
    products per chunk -> 10 C D + 6 D^2."""
    return tokens * HV * (10 * C * D + 6 * D * D)


def decode_bytes(B, HK, HV, D, elt):
    return B * HV * D * D * 4 * 2 + B * (2 * HK * D * elt + 2 * HV * D * elt + 2 * HV * 4)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index
        self.out = os.path.join("/tmp", f"gdn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.out):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 power=float(parts[3]) if parts[3] not in ("[N/A]", "") else 0.0,
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        os.unlink(self.out)
        if not rows:
            return None
        smax = max(r["smax"] for r in rows)
        load = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(load)}


# ---------------------------------------------------------------- timing helpers
class Timer:
    """Per-iteration CUDA-event timing on the current stream, L2 flushed in between."""

    def __init__(self, flush=True):
        self.flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda") \
            if flush else None
        self.times = []

    def run(self, fn, iters, warmup):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        evs = []
        for _ in range(iters):
            if self.flush_buf is not None:
                self.flush_buf.fill_(1.0)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            evs.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]   # ms


def bench_prefill(gdn, w, iters, warmup, states=False, T_override=None, gated=False):
    """One prefill call of workload w; ``gated``: followed by the gated RMS norm of the
    output (gdn_prefill_gated / gdn_prefill_varlen_gated)."""
    d = workloads.workload_inputs(w, device="cuda", T_override=T_override)
    q, k, v, g, b = d["queries"], d["keys"], d["values"], d["decays"], d["beta"]
    s0 = d["initial_state"]
    dev = q.device
    if w.n_seqs:
        cu = d["cu_seqlens"]
        N, T_total = w.n_seqs, q.shape[1]
    else:
        N, T_total = w.B, w.B * q.shape[1]
    HV, D = w.HV, w.Dk
    out = torch.empty_like(v)
    fin = torch.empty(N, HV, D, D, dtype=torch.float32, device=dev)
    st = torch.empty(*v.shape[:-1], D, D, dtype=torch.float32, device=dev) if states else None
    ws = torch.empty(gdn.workspace_size(T_total, N, HV, D, D, dtype=q.dtype), dtype=torch.uint8, device=dev)
    gk = {}
    if gated:
        gen = torch.Generator(device="cuda").manual_seed(7)
        gk = dict(gate=torch.randn(v.shape, generator=gen, device=dev).to(v.dtype),
                  norm_weight=1.0 + 0.3 * torch.randn(D, generator=gen, device=dev))
    if w.n_seqs:
        fn = lambda: gdn.prefill_varlen(q, k, v, g, b, cu, s0, out=out, final_state=fin,
                                        states=st, workspace=ws, **gk)
    else:
        fn = lambda: gdn.prefill(q, k, v, g, b, s0, out=out, final_state=fin, states=st,
                                 workspace=ws, **gk)
    times = Timer(flush=True).run(fn, iters, warmup)
    elt = q.element_size()
    nbytes = prefill_bytes(T_total, w.HK, HV, D, elt, N if s0 is not None else 0, N,
                           T_total if states else 0)
    if gated:
        nbytes += T_total * HV * D * elt + D * 4             # the gate z and the gain
    flops = prefill_flops(T_total, HV, D)
    res = dict(tokens=T_total, ms=statistics.mean(times), ms_min=min(times), bytes=nbytes,
               flops=flops, launches_per_call=(3 if w.n_seqs else 2) + (2 if states else 0))
    del q, k, v, g, b, s0, out, fin, st, ws, d, gk
    torch.cuda.empty_cache()
    return res


def bench_decode(gdn, w, iters, warmup):
    d = workloads.decode_inputs(w, steps=16, device="cuda")
    state = d["initial_state"]
    out = torch.empty(w.B, w.HV, w.Dv, dtype=w.dtype, device="cuda")
    i = [0]

    def fn():
        s = i[0] % 16
        i[0] += 1
        gdn.decode_step(d["queries"][s], d["keys"][s], d["values"][s], d["decays"][s],
                        d["beta"][s], state, out=out)

    # the 512 MiB state is larger than L2: no flush needed between steps
    times = Timer(flush=False).run(fn, iters, warmup)
    nbytes = decode_bytes(w.B, w.HK, w.HV, w.Dk, 2)
    res = dict(ms=statistics.mean(times), ms_min=min(times), bytes=nbytes)
    del d, state, out
    torch.cuda.empty_cache()
    return res


def bench_decode_gated(gdn, w, iters, warmup):
    """The decode step with the gated RMS norm fused in (gdn_decode_step_gated)."""
    d = workloads.decode_inputs(w, steps=16, device="cuda")
    state = d["initial_state"]
    out = torch.empty(w.B, w.HV, w.Dv, dtype=w.dtype, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(4)
    z = torch.randn(16, w.B, w.HV, w.Dv, generator=gen, device="cuda").to(w.dtype)
    wt = 1.0 + 0.3 * torch.randn(w.Dv, generator=gen, device="cuda")
    i = [0]

    def fn():
        s = i[0] % 16
        i[0] += 1
        gdn.decode_step(d["queries"][s], d["keys"][s], d["values"][s], d["decays"][s],
                        d["beta"][s], state, out=out, gate=z[s], norm_weight=wt)

    times = Timer(flush=False).run(fn, iters, warmup)
    nbytes = decode_bytes(w.B, w.HK, w.HV, w.Dk, 2) + w.B * w.HV * w.Dv * 2 + w.Dv * 4
    res = dict(ms=statistics.mean(times), ms_min=min(times), bytes=nbytes)
    del d, state, out, z, wt
    torch.cuda.empty_cache()
    return res


def bench_gated_norm(gdn, w, iters, warmup, copies=4):
    """The gated RMS norm on the outputs of `copies` prefills of workload w (y, gate in, out
    back): y and the gate together are larger than L2, so no flush is needed."""
    gen = torch.Generator(device="cuda").manual_seed(5)
    shape = (w.B * copies, w.T, w.HV, w.Dv)
    y = torch.randn(shape, generator=gen, device="cuda").to(w.dtype)
    z = torch.randn(shape, generator=gen, device="cuda").to(w.dtype)
    wt = 1.0 + 0.3 * torch.randn(w.Dv, generator=gen, device="cuda")
    out = torch.empty_like(y)
    fn = lambda: gdn.gated_rmsnorm(y, z, wt, out=out)
    times = Timer(flush=False).run(fn, iters, warmup)
    rows = w.B * copies * w.T * w.HV
    nbytes = rows * w.Dv * y.element_size() * 3 + w.Dv * 4
    res = dict(rows=rows, ms=statistics.mean(times), ms_min=min(times), bytes=nbytes)
    del y, z, wt, out
    torch.cuda.empty_cache()
    return res


def bench_prologue(gdn, w, iters, warmup, copies=4):
    """The step before the rule from Qwen3-Next's fused projections of `copies` prompts of
    workload w (regroup, conv + SiLU, gates, z copied out): the projections are larger
    than L2, so no flush is needed."""
    gen = torch.Generator(device="cuda").manual_seed(6)
    HK, HV, D, T = w.HK, w.HV, w.Dk, w.B * w.T * copies
    r = HV // HK
    C = 2 * HK * D + HV * D
    W = HK * (2 * D + 2 * r * D)
    proj = torch.randn(copies, T // copies, W, generator=gen, device="cuda").to(w.dtype)
    ba = torch.randn(copies, T // copies, 2 * HV, generator=gen, device="cuda").to(w.dtype)
    cw = torch.randn(C, 4, generator=gen, device="cuda") * 0.5
    al = torch.randn(HV, generator=gen, device="cuda") * 0.5
    db = torch.randn(HV, generator=gen, device="cuda") * 0.5
    fn = lambda: gdn.conv_gate_prologue(proj, ba, None, cw, al, db, HK=HK, HV=HV, Dk=D, Dv=D,
                                        layout="qkvz")
    times = Timer(flush=False).run(fn, iters, warmup)
    elt = proj.element_size()
    nbytes = T * (W * elt + 2 * HV * elt + C * elt + HV * D * elt + 2 * HV * 4) + C * 16 + HV * 8
    res = dict(tokens=T, ms=statistics.mean(times), bytes=nbytes)
    del proj, ba, cw, al, db
    torch.cuda.empty_cache()
    return res


def bench_e2e(gdn, w, iters, warmup):
    """Public API end to end: every step copies its inputs from pinned host memory to the
    device, runs the prefill and copies the output and the final state back to pinned
    host memory.  Consecutive steps are pipelined the way a serving loop runs them: step
    i + 1's inputs go in and step i - 1's results come out while step i computes (two
    buffer sets, one stream each for copies in, compute and copies out, ordered by
    events).  The wall-clock time of all steps, to the last result on the host, is
    divided by the steps."""
    d = workloads.workload_inputs(w, device="cpu")
    names = ("queries", "keys", "values", "decays", "beta")
    host = {n: d[n].pin_memory() for n in names}
    B, T = w.B, w.T
    nb = 2
    dev = [{n: torch.empty_like(host[n], device="cuda") for n in names} for _ in range(nb)]
    out_h = [torch.empty(B, T, w.HV, w.Dv, dtype=w.dtype).pin_memory() for _ in range(nb)]
    fin_h = [torch.empty(B, w.HV, w.Dk, w.Dv, dtype=torch.float32).pin_memory() for _ in range(nb)]
    out_d = [torch.empty_like(out_h[0], device="cuda") for _ in range(nb)]
    fin_d = [torch.empty_like(fin_h[0], device="cuda") for _ in range(nb)]
    ws = torch.empty(gdn.workspace_size(B * T, B, w.HV, w.Dk, w.Dv, dtype=w.dtype), dtype=torch.uint8,
                     device="cuda")
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nb)]
    ev_run = [torch.cuda.Event() for _ in range(nb)]
    ev_out = [torch.cuda.Event() for _ in range(nb)]
    started = [False] * nb

    def step(i):
        b = i % nb
        if started[b]:
            s_in.wait_event(ev_run[b])              # step i - 2 has read buffer set b
        with torch.cuda.stream(s_in):
            for n in names:
                dev[b][n].copy_(host[n], non_blocking=True)
        ev_in[b].record(s_in)
        s_run.wait_event(ev_in[b])
        if started[b]:
            s_run.wait_event(ev_out[b])             # step i - 2's results have left
        gdn.prefill(dev[b]["queries"], dev[b]["keys"], dev[b]["values"], dev[b]["decays"],
                    dev[b]["beta"], None, out=out_d[b], final_state=fin_d[b], workspace=ws,
                    stream=s_run)
        ev_run[b].record(s_run)
        s_out.wait_event(ev_run[b])
        with torch.cuda.stream(s_out):
            out_h[b].copy_(out_d[b], non_blocking=True)
            fin_h[b].copy_(fin_d[b], non_blocking=True)
        ev_out[b].record(s_out)
        started[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(iters):
        step(warmup + i)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / iters
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = out_h[0].numel() * out_h[0].element_size() + fin_h[0].numel() * 4
    return dict(s=dt, h2d=h2d, d2h=d2h, tokens=B * T)


# ---------------------------------------------------------------- CPU oracle baseline
class OracleSample:
    """The fp64 oracle on a bounded sample of a workload: whole (sequence, value head)
    chains, as many as run in about `target_s` seconds on the host cores.  Inputs are
    drawn once; each call of run() times the same sample."""

    def __init__(self, w, target_s=12.0):
        import oracle
        self.oracle = oracle
        self.w = w
        self.d = workloads.workload_inputs(w, device="cpu", T_override=min(w.T, 4096) if w.T else None)
        self.T = self.d["queries"].shape[1]
        self.cores = oracle.default_threads()
        t0 = time.perf_counter()
        oracle.forward(*(self.d[k][:1] for k in ("queries", "keys", "values", "decays", "beta")),
                       chains=[0], n_threads=1)
        one = time.perf_counter() - t0
        self.n = max(1, min(w.B * w.HV, int(target_s * self.cores / max(one, 1e-6))))
        self.desc = (f"{self.n} (sequence, value head) chains x {self.T} tokens of {w.name}, "
                     f"fp64, {self.cores} threads")

    def run(self):
        """Tokens/s (all value heads of a token counted once) of one timed pass."""
        d = self.d
        t0 = time.perf_counter()
        self.oracle.forward(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                            chains=list(range(self.n)), n_threads=self.cores)
        el = time.perf_counter() - t0
        return (self.n / self.w.HV) * self.T / el


def oracle_chain_rate(w, target_s=6.0, want_states=False):
    """The fp64 oracle on whole (sequence, value head) chains of workload w, as many as
    run in about `target_s` seconds on the host cores (packed batches use their own
    sequences).  Returns (tokens/s with all value heads of a token counted once, cores,
    description of the sample)."""
    import concurrent.futures as cf
    import oracle
    d = workloads.workload_inputs(w, device="cpu")
    cores = oracle.default_threads()
    r = w.HV // w.HK
    if w.n_seqs:
        cu = [int(x) for x in d["cu_seqlens"].tolist()]
        spans = [(0, cu[i], cu[i + 1]) for i in range(w.n_seqs)]
    else:
        spans = [(b, 0, d["queries"].shape[1]) for b in range(w.B)]
    order = [(s, h) for h in range(w.HV) for s in range(len(spans))]  # spread over sequences

    def one(sh):
        s, h = sh
        b, a, e = spans[s]
        s0 = d.get("initial_state")
        oracle.chain(d["queries"][b, a:e, h // r], d["keys"][b, a:e, h // r], d["values"][b, a:e, h],
                     d["decays"][b, a:e, h], d["beta"][b, a:e, h],
                     initial_state=None if s0 is None else s0[s, h], want_states=want_states)
        return e - a

    t0 = time.perf_counter()
    first = one(order[0])
    t_one = max(time.perf_counter() - t0, 1e-6)
    per_token = t_one / max(first, 1)
    budget = target_s * cores / per_token                  # chain-tokens in the budget
    chosen, tok = [], 0
    for sh in order[1:]:
        n = spans[sh[0]][2] - spans[sh[0]][1]
        if chosen and tok + n > budget:
            break
        chosen.append(sh)
        tok += n
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        done = sum(ex.map(one, chosen)) if chosen else 0
    el = time.perf_counter() - t0
    if not chosen:
        done, el = first, t_one
    desc = (f"{len(chosen) or 1} (sequence, value head) chains ({done} chain-tokens) of {w.name}"
            f"{' with per-token states' if want_states else ''}, fp64, {cores} threads")
    return (done / w.HV) / el, cores, desc


def oracle_decode_rate(w, target_s=6.0, n_seq=32):
    """The fp64 oracle's decode step on `n_seq` of the workload's sequences (all value
    heads), consecutive steps carrying the state; the rate is scaled to steps of the full
    batch (sequences are independent, so a step's work is proportional to the batch)."""
    import oracle
    d = workloads.decode_inputs(w, steps=16, device="cpu")
    cores = oracle.default_threads()
    n_seq = min(n_seq, w.B)
    st = d["initial_state"][:n_seq].contiguous()
    names = ("queries", "keys", "values", "decays", "beta")
    step = lambda i, st: oracle.decode_step(*(d[n][i][:n_seq].contiguous() for n in names), st,
                                            n_threads=cores)[1]
    t0 = time.perf_counter()
    st = step(0, st)
    t1 = max(time.perf_counter() - t0, 1e-6)
    k = max(1, min(15, int(target_s / t1)))
    t0 = time.perf_counter()
    for i in range(k):
        st = step(1 + i, st)
    el = time.perf_counter() - t0
    return (k / el) * n_seq / w.B, cores, (f"{k} consecutive decode steps of {n_seq} of the {w.B} sequences "
                                           f"of {w.name} (all heads; rate scaled to the full batch), "
                                           f"fp64, {cores} threads")


def oracle_norm_rate(w, target_s=4.0):
    """The oracle's gated RMS norm over rows of workload w's output shape; rows/s."""
    import oracle
    gen = torch.Generator().manual_seed(5)
    rows = w.T * w.HV
    y = torch.randn(rows, w.Dv, generator=gen).to(w.dtype)
    z = torch.randn(rows, w.Dv, generator=gen).to(w.dtype)
    wt = 1.0 + 0.3 * torch.randn(w.Dv, generator=gen)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.gated_rmsnorm(y, z, wt)
        n += 1
        el = time.perf_counter() - t0
        if el > target_s or n >= 50:
            break
    return n * rows / el, 1, f"{n} passes over {rows} rows of {w.Dv} ({w.name} outputs), fp64, 1 thread"


def oracle_prologue_rate(w, target_s=4.0):
    """The oracle's regroup of Qwen3-Next's fused projections, conv + SiLU and gates over
    one prompt of workload w; tokens/s."""
    import oracle
    gen = torch.Generator().manual_seed(6)
    HK, HV, D, T = w.HK, w.HV, w.Dk, w.T
    r = HV // HK
    C = 2 * HK * D + HV * D
    proj = torch.randn(1, T, HK * (2 * D + 2 * r * D), generator=gen).to(w.dtype)
    ba = torch.randn(1, T, 2 * HV, generator=gen).to(w.dtype)
    cw = torch.randn(C, 4, generator=gen) * 0.5
    al = torch.randn(HV, generator=gen) * 0.5
    db = torch.randn(HV, generator=gen) * 0.5
    import numpy as np
    t0 = time.perf_counter()
    n = 0
    while True:
        q, k, v, z, b, a = oracle.regroup_qkvz(proj, ba, HK, HV, D, D)
        x = np.concatenate([q.reshape(1, T, -1), k.reshape(1, T, -1), v.reshape(1, T, -1)], axis=-1)
        oracle.conv_gate(x, b, a, cw, al, db)
        n += 1
        el = time.perf_counter() - t0
        if el > target_s or n >= 20:
            break
    return n * T / el, 1, f"{n} prompts of {T} tokens of {w.name} (fused layout), fp64, 1 thread"


def oracle_decode_gated_rate(w, target_s=6.0, n_seq=32):
    """The oracle's decode step followed by the gated RMS norm of its output, on `n_seq`
    sequences; steps/s scaled to the full batch."""
    import oracle
    d = workloads.decode_inputs(w, steps=16, device="cpu")
    cores = oracle.default_threads()
    n_seq = min(n_seq, w.B)
    st = d["initial_state"][:n_seq].contiguous()
    gen = torch.Generator().manual_seed(4)
    z = torch.randn(n_seq, w.HV, w.Dv, generator=gen).to(w.dtype)
    wt = 1.0 + 0.3 * torch.randn(w.Dv, generator=gen)
    names = ("queries", "keys", "values", "decays", "beta")

    def step(i, st):
        o, st = oracle.decode_step(*(d[n][i][:n_seq].contiguous() for n in names), st, n_threads=cores)
        oracle.gated_rmsnorm(o, z, wt)
        return st

    t0 = time.perf_counter()
    st = step(0, st)
    t1 = max(time.perf_counter() - t0, 1e-6)
    k = max(1, min(15, int(target_s / t1)))
    t0 = time.perf_counter()
    for i in range(k):
        st = step(1 + i, st)
    el = time.perf_counter() - t0
    return (k / el) * n_seq / w.B, cores, (f"{k} consecutive gated decode steps of {n_seq} of the {w.B} "
                                           f"sequences of {w.name} (rate scaled to the full batch), fp64, "
                                           f"{cores} threads")


def oracle_prefill_gated_rate(w, target_s=6.0):
    """The oracle's prefill of whole chains of workload w followed by the gated RMS norm of
    their outputs; tokens/s with all value heads of a token counted once."""
    import oracle
    d = workloads.workload_inputs(w, device="cpu")
    cores = oracle.default_threads()
    gen = torch.Generator().manual_seed(7)
    zf = torch.randn(w.T, w.Dv, generator=gen).to(w.dtype)
    wt = 1.0 + 0.3 * torch.randn(w.Dv, generator=gen)
    t0 = time.perf_counter()
    o, _, _ = oracle.forward(*(d[k][:1] for k in ("queries", "keys", "values", "decays", "beta")),
                             chains=[0], n_threads=1)
    one = max(time.perf_counter() - t0, 1e-6)
    n = max(1, min(w.HV, int(target_s * cores / one)))
    t0 = time.perf_counter()
    o, _, _ = oracle.forward(d["queries"], d["keys"], d["values"], d["decays"], d["beta"],
                             chains=list(range(n)), n_threads=cores)
    for h in range(n):
        oracle.gated_rmsnorm(o[0, :, h], zf, wt)
    el = time.perf_counter() - t0
    return (n / w.HV) * w.T / el, cores, (f"{n} value-head chains x {w.T} tokens of {w.name}, each output "
                                          f"then gated-normed, fp64, {cores} threads")


# ---------------------------------------------------------------- main
def dist_setup(backend="nccl"):
    """One process per GPU (torchrun): rank, local rank and world size from the env."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def max_over_ranks(x, ws, device="cuda"):
    """Slowest rank's time: the job is done when every replica is."""
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, seconds_max, ws):
    """Whole-job throughput of a weak-scaled run: every rank processes its own batch."""
    return ws * units_per_rank / seconds_max


def barrier(ws, cuda=True):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    if cuda:
        torch.cuda.synchronize()


def run_reference(args, ws, rank):
    """Reference arm: the fp64 CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    w = workloads.WORKLOADS["next_prefill_T4096_hk16_hv32_d128"]
    # each step a bounded sample, sized so that all steps take about two minutes
    sample = OracleSample(w, target_s=max(1.0, 120.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        sample.run()
    vals = [sample.run() for _ in range(args.steps)]
    value = statistics.mean(vals)
    cores, desc = sample.cores, sample.desc
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * 4096 / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "HK": w.HK, "HV": w.HV,
                       "Dk": w.Dk, "Dv": w.Dv},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline and decode only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="",
                    help="comma list of prologue, gated_norm, decode_gated_norm, states, headline, "
                         "varlen, long, hv48, hv16, f32, tiny: time just those steps and print one "
                         "line each (profiling; not the bench line)")
    ap.add_argument("--prefill-T", type=int, default=0,
                    help="override the headline prefill length (profiling a case larger than L2); "
                         "with --only states, the per-token-state workload's length")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return

    import gated_deltanet_mixer_delta_gb300 as gdn
    gdn.load_library(build_if_missing=True)
    torch.cuda.set_device(local)
    P, peak_src = peaks()
    hbm = P["hbm_gbs"]
    clocks = ClockSampler(local)
    clocks.start()

    W = workloads.WORKLOADS
    head_w = W["next_prefill_T4096_hk16_hv32_d128"]
    if args.only:
        runs = {"prologue": lambda: bench_prologue(gdn, head_w, args.steps, args.warmup),
                "gated_norm": lambda: bench_gated_norm(gdn, head_w, args.steps, args.warmup),
                "decode_gated_norm": lambda: bench_decode_gated(gdn, W["decode_B256_hk16_hv32_d128"],
                                                                args.steps, args.warmup),
                "states": lambda: bench_prefill(gdn, W["states_B4_T1024_hk16_hv32_d128"], args.steps,
                                                args.warmup, states=True,
                                                T_override=args.prefill_T or None),
                "headline": lambda: bench_prefill(gdn, head_w, args.steps, args.warmup),
                "varlen": lambda: bench_prefill(gdn, W["varlen8_512to8192_hk16_hv32_d128"], args.steps,
                                                args.warmup),
                "long": lambda: bench_prefill(gdn, W["long_prefill_B2_T65536_hk16_hv32_d128"],
                                              args.steps, args.warmup),
                "hv48": lambda: bench_prefill(gdn, W["qwen35_27b_prefill_T4096_hk16_hv48_d128"],
                                              args.steps, args.warmup),
                "hv16": lambda: bench_prefill(gdn, W["qwen35_0p8b_prefill_T4096_hk16_hv16_d128"],
                                              args.steps, args.warmup),
                # the CUDA-core prefill: fp32 inputs at the headline shape, and the tiny case
                "f32": lambda: bench_prefill(gdn, dataclasses.replace(head_w, dtype=torch.float32,
                                                                      name=head_w.name + "_f32"),
                                             args.steps, args.warmup),
                "tiny": lambda: bench_prefill(gdn, W["tiny_T64_H2_d32_f32"], args.steps, args.warmup)}
        for name in args.only.split(","):
            r = runs[name]()
            if rank == 0:
                print(json.dumps({"only": name, "ms": r["ms"], "bytes": r["bytes"],
                                  "hbm_frac": r["bytes"] / (r["ms"] * 1e-3) / 1e9 / hbm}))
        clocks.stop()
        return
    barrier(ws)
    head = bench_prefill(gdn, head_w, args.steps, args.warmup, T_override=args.prefill_T or None)
    barrier(ws)
    ms = max_over_ranks(head["ms"], ws)
    value = job_rate(head["tokens"], ms * 1e-3, ws)
    dec = bench_decode(gdn, W["decode_B256_hk16_hv32_d128"], max(args.steps, 20), args.warmup)
    dec_ms = max_over_ranks(dec["ms"], ws)

    # end to end right after the headline, before the larger workloads churn memory
    e2e = bench_e2e(gdn, head_w, max(5, min(args.steps, 20)), 2)
    e2e_s = max_over_ranks(e2e["s"], ws)

    subs = {}
    if not args.quick:
        for key, name, kw in (("varlen", "varlen8_512to8192_hk16_hv32_d128", {}),
                              ("long_prefill", "long_prefill_B2_T65536_hk16_hv32_d128", {}),
                              ("states", "states_B4_T1024_hk16_hv32_d128", {"states": True}),
                              ("prefill_hv48", "qwen35_27b_prefill_T4096_hk16_hv48_d128", {}),
                              ("prefill_hv16", "qwen35_0p8b_prefill_T4096_hk16_hv16_d128", {})):
            r = bench_prefill(gdn, W[name], max(3, min(args.steps, 5)), 3, **kw)
            r_ms = max_over_ranks(r["ms"], ws)
            subs[key] = dict(workload=name, tokens=r["tokens"], ms=r_ms,
                             tokens_per_s=ws * r["tokens"] / (r_ms * 1e-3),
                             roofline={"bound": "hbm", "achieved": r["bytes"] / (r_ms * 1e-3) / 1e9,
                                       "peak": hbm, "unit": "GB/s",
                                       "frac": r["bytes"] / (r_ms * 1e-3) / 1e9 / hbm,
                                       "algorithmic_bytes": r["bytes"]})
        dg = bench_decode_gated(gdn, W["decode_B256_hk16_hv32_d128"], max(args.steps, 20),
                                args.warmup)
        subs["decode_gated_norm"] = dict(
            workload="decode_B256_hk16_hv32_d128 + gated RMS norm fused", ms=dg["ms"],
            steps_per_s=1e3 / dg["ms"],
            roofline={"bound": "hbm", "achieved": dg["bytes"] / (dg["ms"] * 1e-3) / 1e9, "peak": hbm,
                      "unit": "GB/s", "frac": dg["bytes"] / (dg["ms"] * 1e-3) / 1e9 / hbm,
                      "algorithmic_bytes": dg["bytes"]})
        r = bench_prefill(gdn, head_w, max(3, min(args.steps, 20)), 3, gated=True)
        subs["prefill_gated_norm"] = dict(
            workload=head_w.name + " followed by the gated RMS norm (gdn_prefill_gated)",
            tokens=r["tokens"], ms=r["ms"], tokens_per_s=r["tokens"] / (r["ms"] * 1e-3),
            roofline={"bound": "hbm", "achieved": r["bytes"] / (r["ms"] * 1e-3) / 1e9, "peak": hbm,
                      "unit": "GB/s", "frac": r["bytes"] / (r["ms"] * 1e-3) / 1e9 / hbm,
                      "algorithmic_bytes": r["bytes"]})
        pr = bench_prologue(gdn, head_w, max(args.steps, 20), args.warmup)
        subs["prologue"] = dict(
            workload="conv + gates from the fused projections of 4 next_prefill_T4096_hk16_hv32_d128 "
                     "prompts (400 MB, larger than L2: no flush)",
            tokens=pr["tokens"], ms=pr["ms"],
            roofline={"bound": "hbm", "achieved": pr["bytes"] / (pr["ms"] * 1e-3) / 1e9, "peak": hbm,
                      "unit": "GB/s", "frac": pr["bytes"] / (pr["ms"] * 1e-3) / 1e9 / hbm,
                      "algorithmic_bytes": pr["bytes"]})
        gn = bench_gated_norm(gdn, head_w, max(args.steps, 20), args.warmup)
        subs["gated_norm"] = dict(
            workload="gated RMS norm of 4 next_prefill_T4096_hk16_hv32_d128 outputs "
                     "(y and gate 268 MB, larger than L2: no flush)", rows=gn["rows"],
            ms=gn["ms"],
            roofline={"bound": "hbm", "achieved": gn["bytes"] / (gn["ms"] * 1e-3) / 1e9, "peak": hbm,
                      "unit": "GB/s", "frac": gn["bytes"] / (gn["ms"] * 1e-3) / 1e9 / hbm,
                      "algorithmic_bytes": gn["bytes"]})
    clk = clocks.stop()

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        sample = OracleSample(head_w)
        cpu = {"value": sample.run(), "unit": "tokens/s", "cores": sample.cores, "kind": "oracle",
               "sample": sample.desc}
        # the oracle on the other rows: a bounded sample of each workload
        rate, cores, desc = oracle_decode_rate(W["decode_B256_hk16_hv32_d128"])
        dec["cpu_baseline"] = {"value": rate, "unit": "steps/s", "cores": cores, "kind": "oracle",
                               "sample": desc}
        for key, wants in (("varlen", False), ("long_prefill", False), ("states", True),
                           ("prefill_hv48", False), ("prefill_hv16", False)):
            if key in subs:
                rate, cores, desc = oracle_chain_rate(W[subs[key]["workload"]], want_states=wants)
                subs[key]["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores,
                                             "kind": "oracle", "sample": desc}
        for key, fn, unit in (("decode_gated_norm", lambda: oracle_decode_gated_rate(
                                    W["decode_B256_hk16_hv32_d128"]), "steps/s"),
                              ("prefill_gated_norm", lambda: oracle_prefill_gated_rate(head_w), "tokens/s"),
                              ("prologue", lambda: oracle_prologue_rate(head_w), "tokens/s"),
                              ("gated_norm", lambda: oracle_norm_rate(head_w), "rows/s")):
            if key in subs:
                rate, cores, desc = fn()
                subs[key]["cpu_baseline"] = {"value": rate, "unit": unit, "cores": cores,
                                             "kind": "oracle", "sample": desc}

    if rank != 0:
        return
    achieved = head["bytes"] / (head["ms"] * 1e-3) / 1e9
    # traffic of the headline workload's call (ncu capture at T = 4096 only)
    traffic = (measured_traffic("prefill_kernels_T4096.md", "gdn_prefill_tc.cu")
               if not args.prefill_T else None)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": head_w.name, "B": head_w.B, "T": head_w.T, "HK": head_w.HK,
                   "HV": head_w.HV, "Dk": head_w.Dk, "Dv": head_w.Dv,
                   "l2": "flushed between timed iterations (256 MiB write)",
                   "parallelism": f"replicas x{ws} (independent batches)"},
        "roofline": {"bound": "hbm", "kernel": "gdn_prefill (prep + scan)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic, "peak_source": peak_src,
                     "algorithmic_bytes": head["bytes"], "flops": head["flops"]},
        # the same call against the tensor pipe (HBM binds: this figure is context)
        "roofline_tensor": {"bound": "tensor", "achieved": head["flops"] / (head["ms"] * 1e-3) / 1e12,
                            "peak": P["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": head["flops"] / (head["ms"] * 1e-3) / 1e12 / P["bf16_tflops"],
                            "peak_source": peak_src + " (bf16 burst)"},
        "decode": {"workload": "decode_B256_hk16_hv32_d128", "value": 1e3 / dec_ms * ws,
                   "unit": "steps/s", "ms_per_step": dec_ms,
                   "roofline": {"bound": "hbm", "kernel": "decode_kernel",
                                "achieved": dec["bytes"] / (dec_ms * 1e-3) / 1e9,
                                "peak": hbm, "unit": "GB/s",
                                "frac": dec["bytes"] / (dec_ms * 1e-3) / 1e9 / hbm,
                                "traffic": measured_traffic("decode_kernel_B256.md", "gdn_decode.cu"),
                                "algorithmic_bytes": dec["bytes"]},
                   "cpu_baseline": dec.get("cpu_baseline")},
        "e2e": {"value": e2e["tokens"] / e2e_s * ws, "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": args.steps * head["launches_per_call"],
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    line.update(subs)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
