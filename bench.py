#!/usr/bin/env python
"""Benchmark of the GDN-2 chunked prefill forward on one or more GB300s.

One "step" is one full forward (every kernel of the launch sequence) over one
batch of the workload, inputs resident in HBM.  Default workload: the
long-context configuration B=4 x T=32768, H=HV=32, K=V=128 (131072 tokens per
step), whose inputs (8.6 GB) exceed the 129 MB L2, so no flush is needed
between steps.

Prints ONE JSON line (rank 0).  Besides the throughput it reports
 * roofline: the dominant kernel's algorithmic HBM bytes per launch over its
   CUDA-event time on the launching stream, against the measured HBM peak;
 * e2e: the same metric through the public API from pinned HOST buffers,
   host->device and device->host copies inside the timed region;
 * cpu_baseline: the FP64 oracle on the host cores over a bounded sample;
 * clocks sampled with nvidia-smi during the timed region.

``--impl reference`` times the oracle instead (the reference arm).
Multi-GPU (torchrun): every rank runs its own batch (weak scaling, no
collective on the data path); time = max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN-2 prefill tokens/s at H32/D128 bf16; fraction of roofline"
FALLBACK_HBM_GBS = 6800.0
DEFAULT_WORKLOAD = 5


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 30 prefill forwards, 500 decode steps)")
    ap.add_argument("--warmup", type=int, default=None,
                    help="warm-up steps (default: 3 prefill forwards; decode: >= 3 steps and >= 0.3 s)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["prefill", "decode"], default="prefill",
                    help="prefill: the chunked forward (default); decode: the token-by-token "
                         "recurrence from a carried state (gdn2_recurrent_fwd)")
    ap.add_argument("--decode-batch", type=int, default=128)
    ap.add_argument("--decode-tokens", type=int, default=1)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD)
    ap.add_argument("--kernels", choices=["tc", "simt"], default=os.environ.get("GDN2_BENCH_KERNELS", "tc"))
    ap.add_argument("--e2e-steps", type=int, default=7)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other D=128 workloads (2-4) in the line's `configs` object")
    ap.add_argument("--config-steps", type=int, default=20)
    ap.add_argument("--config-cpu-seconds", type=float, default=4.0)
    ap.add_argument("--segments", type=int, default=0,
                    help="segments per sequence of the chunk-parallel state pass (0: the library's choice)")
    ap.add_argument("--seqs", type=int, default=0,
                    help="keep only the workload's first SEQS sequences (a smaller case of the same "
                         "shape, for profiler captures); 0 = all")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 500 if args.op == "decode" else 30
    if args.warmup is None:
        args.warmup = 3
    return args


# ---------------------------------------------------------------------------
# byte accounting (per launch): the algorithmic bytes a stage must move, each
# of its inputs read once and each output written once; the roofline's
# `achieved` is these bytes over the stage's CUDA-event time
# ---------------------------------------------------------------------------
def n_chunks(wl):
    return sum((L + 63) // 64 for L in wl.lens)


def fused_min_bytes(wl, has_h0, write_state=True):
    """The whole operator's minimum HBM traffic: every input read once, the
    output written once, states in/out."""
    T, H, HV, K, V = wl.T_tot, wl.H, wl.HV, wl.K, wl.V
    b = T * H * K * 2 * 2                      # q, k
    b += T * HV * V * 2 * 3                    # v, w, o
    b += T * HV * K * (4 + 2)                  # g fp32, beta bf16
    st = wl.N * HV * K * V * 4
    return b + (st if has_h0 else 0) + (st if write_state else 0)


def stage_bytes(wl, impl, has_h0, write_state=True, l2norm=False):
    """Algorithmic bytes each stage of the launch sequence must move: its own
    inputs read once and outputs written once (intermediates in bf16, G in
    fp32)."""
    T, H, HV, K, V = wl.T_tot, wl.H, wl.HV, wl.K, wl.V
    NC = n_chunks(wl)
    st = wl.N * HV * K * V * 4
    qk1 = T * H * K * 2            # one of q / k
    kh = T * HV * K                # per-(token, value head) key-channel elements
    vh = T * HV * V
    hb = NC * HV * K * V * 2       # bf16 chunk states
    out = {}
    if impl == "tc":
        rec = (73728 + 512 + 1023) // 1024 * 1024 if K == 128 else (40960 + 256 + 1023) // 1024 * 1024
        rec_read = (rec - 1024 + 4 * K) if K == 128 else (rec - 1024 + 4 * K)
        out["chunk_map"] = 0
        out["intra"] = 2 * qk1 + vh * 2 * 2 + kh * 4 + kh * 2 + NC * HV * rec
        out["state_output"] = NC * HV * rec_read + vh * 2 + (st if has_h0 else 0) + (st if write_state else 0)
        return out
    out["prep"] = kh * 4 * 2 + (4 * qk1 if l2norm else 0)
    out["intra"] = qk1 + kh * 4 + kh * 2 + vh * 2 * 2 + kh * 2 + vh * 2
    out["state"] = kh * 2 + vh * 2 + qk1 + kh * 4 + hb + vh * 2 + (st if has_h0 else 0) + (
        st if write_state else 0)
    out["output"] = 2 * qk1 + kh * 4 + hb + vh * 2 + vh * 2
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def strip_comments(src):
    """C/C++ source without comments and blank lines (string literals kept)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == '"' or c == "'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            while i < n and src[i] != "\n":
                i += 1
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return "\n".join(ln for ln in lines if ln.strip())


# The source files of the kernels each profiled stage runs (besides every
# shared header): a committed ncu summary stays valid while these are unchanged.
STAGE_SOURCES = {
    "intra": ["gdn2_tc_intra.cu"],
    "state_output": ["gdn2_tc_state_la.cu"],  # the lookahead kernels (the long workloads' sequential pass)
    "recurrent": ["gdn2_recurrent.cu"],
}


def kernel_source_sha(read=None, files=None):
    """Hash of the CUDA sources' code (comments and blank lines ignored): of
    every source, or of the headers and the named .cu files.  It tells whether
    a committed ncu summary was taken on the current kernels."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_prefill_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith(".cuh") or (f.endswith(".cu") and (files is None or f in files)):
            txt = read(f) if read else open(os.path.join(csrc, f), encoding="utf-8").read()
            h.update(f.encode() + b"\0" + strip_comments(txt).encode() + b"\0")
    return h.hexdigest()[:16]


def stage_source_sha(stage):
    """kernel_source_sha over the headers and the stage's own kernel sources."""
    return kernel_source_sha(files=STAGE_SOURCES.get(stage))


def ncu_traffic(stage, impl, workload_name):
    """DRAM bytes per launch of a stage's kernel from a committed ncu summary
    (profiles/*.md with lines 'traffic_bytes_per_launch: <n>' and
    'source_sha: <sha>', the stage_source_sha of the sources it was taken
    on); None when absent or taken on other kernel sources."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    sha = stage_source_sha(stage)
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        txt = open(os.path.join(pdir, f)).read()
        m_stage = re.search(r"^stage:\s*(\S+)", txt, re.M)
        m_impl = re.search(r"^impl:\s*(\S+)", txt, re.M)
        m_wl = re.search(r"^workload:\s*(\S+)", txt, re.M)
        m_b = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt, re.M)
        m_sha = re.search(r"^source_sha:\s*(\S+)", txt, re.M)
        if not (m_stage and m_impl and m_b and m_sha and m_wl):
            continue
        if m_stage.group(1) == stage and m_impl.group(1) == impl and m_wl.group(1) == workload_name:
            return float(m_b.group(1)) if m_sha.group(1) == sha else None
    return None


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index):
        self.dev = dev_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.1)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pc=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in rows:
            if r["hw"].startswith("Active"):
                reasons.add("hw_slowdown")
            if r["hwt"].startswith("Active"):
                reasons.add("hw_thermal_slowdown")
            if r["swt"].startswith("Active"):
                reasons.add("sw_thermal_slowdown")
            if r["pc"].startswith("Active"):
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(loaded)}


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and reference arm)
# ---------------------------------------------------------------------------
def unit_batch(d, wl, units, n_tokens=None):
    """Stand-alone float64 host problem made of whole (sequence, value head)
    units (or their first n_tokens): unit i becomes packed sequence i with
    one key head and one value head."""
    import numpy as np
    cu = d["cu_seqlens"].tolist()
    group = wl.HV // wl.H
    parts = {k: [] for k in ("q", "k", "v", "g", "beta", "w", "h0")}
    lens = []
    for n, hv in units:
        a = cu[n]
        b = cu[n + 1] if n_tokens is None else min(cu[n + 1], a + n_tokens)
        h = hv // group
        for key, head in (("q", h), ("k", h), ("v", hv), ("g", hv), ("beta", hv), ("w", hv)):
            parts[key].append(d[key][a:b, head:head + 1].double().cpu().numpy())
        if d["h0"] is not None:
            parts["h0"].append(d["h0"][n:n + 1, hv:hv + 1].double().cpu().numpy())
        lens.append(b - a)
    out = {k: (np.concatenate(v) if v else None) for k, v in parts.items()}
    out["cu_seqlens"] = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    out["scale"] = d["scale"]
    out["tokens"] = int(sum(lens))
    return out


def time_oracle(b, threads):
    """Wall time of the oracle's C call on a prepared float64 batch."""
    import oracle
    t0 = time.perf_counter()
    oracle.gdn2_forward(b["q"], b["k"], b["v"], b["g"], b["beta"], b["w"], scale=b["scale"],
                        initial_state=b["h0"], cu_seqlens=b["cu_seqlens"], threads=threads)
    return time.perf_counter() - t0


def cpu_baseline(d, wl, seconds):
    """The oracle, as it stands, on the host cores over a bounded sample:
    whole (sequence, value head) units in order, one batch of `threads`
    units at a time, until about `seconds` of oracle time is spent."""
    threads = max(1, min(os.cpu_count() or 1, wl.N * wl.HV))
    all_units = [(n, hv) for n in range(wl.N) for hv in range(wl.HV)]
    total_t, tokens, done = 0.0, 0, 0
    while done < len(all_units) and total_t < seconds:
        batch = unit_batch(d, wl, all_units[done:done + threads])
        total_t += time_oracle(batch, threads)
        tokens += batch["tokens"]
        done += min(threads, len(all_units) - done)
    return {"value": tokens / wl.HV / total_t, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "FP64 oracle on %d of %d whole (sequence, value head) units (%d token-heads), "
                      "%.1f s on %d threads; tokens/s = token-heads / HV / s"
                      % (done, len(all_units), tokens, total_t, threads)}


# ---------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    from gated_deltanet_prefill_gb300 import inputs
    import oracle
    oracle.build()
    wl = inputs.workload(args.workload)
    # a bounded host-generated slice of the workload (same recipe)
    small_lens = (min(wl.lens[0], 16384),)
    wl_s = inputs.Workload(wl.name + "_slice", small_lens, wl.H, wl.HV, wl.K, wl.V, g_max=wl.g_max,
                           beta_max=wl.beta_max, h0_std=wl.h0_std, seed=wl.seed, scale=wl.scale)
    d = inputs.generate(wl_s)
    threads = max(1, min(os.cpu_count() or 1, wl.HV))
    units = [(0, hv) for hv in range(threads)]
    per_step = max(2.0, 90.0 / max(1, args.steps + args.warmup))
    probe = time_oracle(unit_batch(d, wl_s, units, 256), threads) / 256
    n_tok = max(64, min(wl_s.lens[0], int(per_step / max(probe, 1e-9)) // 64 * 64))
    b = unit_batch(d, wl_s, units, n_tok)
    for _ in range(args.warmup):
        time_oracle(b, threads)
    times = [time_oracle(b, threads) for _ in range(args.steps)]
    dt = sum(times) / len(times)
    val = n_tok * threads / wl.HV / dt
    units = threads
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.N, "T": wl.lens[0], "H": wl.H, "HV": wl.HV,
                       "K": wl.K, "V": wl.V,
                       "sample_per_step": "sequence 0 tokens [0,%d) x %d value heads" % (n_tok, units)},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": units, "kind": "oracle",
                             "sample": "FP64 oracle per step: %d tokens x %d of %d value heads"
                                       % (n_tok, units, wl.HV)},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def gpu_numa_cpus(dev):
    """Host CPUs local to CUDA device `dev` (from sysfs), or None."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(dev)
        bus = "%04x:%02x:%02x.0" % (getattr(pr, "pci_domain_id", 0), pr.pci_bus_id, pr.pci_device_id)
        txt = open("/sys/bus/pci/devices/%s/local_cpulist" % bus).read().strip()
    except Exception:
        return None
    cpus = set()
    for part in txt.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    return cpus or None


def measure(wl, args, K, warmup, seed_rank=0, world=1, clocks_dev=None):
    """Time K steps of one workload exactly as the headline is timed: inputs
    resident in HBM, >= 3 warm-up steps, CUDA events on the launching stream,
    a 512 MB L2 flush between steps (outside the per-step events) when the
    inputs are under 1 GB.  Returns the timing record and the live buffers."""
    import torch
    from gated_deltanet_prefill_gb300 import dist as gdist
    from gated_deltanet_prefill_gb300 import gdn2, inputs

    wl_r = inputs.with_seed(wl, gdist.rank_seed(wl.seed, seed_rank))  # each rank: its own batch
    d = inputs.generate(wl_r, device="cuda")
    T, HV, V = wl.T_tot, wl.HV, wl.V
    out = torch.empty((T, HV, V), dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((wl.N, HV, wl.K, V), dtype=torch.float32, device="cuda")
    dims = gdn2.make_dims(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], out, d["cu_seqlens"],
                          False, args.kernels)
    dims.state_segments = args.segments
    ws = torch.empty(gdn2.workspace_bytes(dims), dtype=torch.uint8, device="cuda")
    names = gdn2.stage_names(dims)
    stream = torch.cuda.current_stream()

    def step(evs=None):
        gdn2.chunk_gdn2_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                            initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], out=out, final_state=fs,
                            workspace=ws, impl=args.kernels, stage_events=evs, state_segments=args.segments)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    stage_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(K)]
    for evs in stage_evs:  # materialise the CUDA events
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # inputs within a few L2 sizes: write a 512 MB buffer between steps, outside
    # each step's events, and time the steps one by one
    fmin = fused_min_bytes(wl, d["h0"] is not None)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda") if fmin < 1e9 else None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clk = Clocks(clocks_dev) if clocks_dev is not None else None
    if clk:
        clk.__enter__()
    # The steps are timed as a user runs them: no event between their kernels,
    # so each kernel's launch overlaps its predecessor's tail (programmatic
    # dependent launches).  The per-stage times come from K more steps with an
    # event between the stages, which serialises the stage boundaries.
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in step_evs:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(K):
        if flush is not None:
            flush.zero_()
        step_evs[i][0].record(stream)
        step()
        step_evs[i][1].record(stream)
    end.record(stream)
    for i in range(K):
        if flush is not None:
            flush.zero_()
        step(stage_evs[i])
    torch.cuda.synchronize()
    if clk:
        clk.__exit__()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if flush is None:
        ms = gdist.max_over_ranks(start.elapsed_time(end) / K, device="cuda")
    else:
        per_step = [a.elapsed_time(b) for a, b in step_evs]
        ms = gdist.max_over_ranks(sum(per_step) / K, device="cuda")
        del flush
    stage_ms = {n: sum(ev[i].elapsed_time(ev[i + 1]) for ev in stage_evs) / K for i, n in enumerate(names)}
    staged_ms = sum(ev[0].elapsed_time(ev[-1]) for ev in stage_evs) / K
    status = gdn2.device_status(ws)
    peak, peak_kind = load_peaks()
    sb = stage_bytes(wl, args.kernels, d["h0"] is not None, True, False)
    stages = {n: {"ms": stage_ms[n], "algorithmic_bytes": sb.get(n),
                  "gbs": (sb[n] / (stage_ms[n] * 1e-3) / 1e9) if sb.get(n) else None,
                  "frac_of_peak": (sb[n] / (stage_ms[n] * 1e-3) / 1e9 / peak) if sb.get(n) else None,
                  "share": stage_ms[n] / max(sum(stage_ms.values()), 1e-12)} for n in names}
    whole = {"min_bytes": fmin, "achieved_gbs": fmin / (ms * 1e-3) / 1e9,
             "frac": fmin / (ms * 1e-3) / 1e9 / peak}
    rec = {"ms": ms, "staged_ms": staged_ms, "stage_ms": stage_ms, "stages": stages, "whole_op": whole, "sb": sb,
           "peak": peak,
           "peak_kind": peak_kind, "fmin": fmin, "dims": dims, "status": status,
           "clocks": clk.summary() if clk else None}
    return rec, dict(d=d, out=out, fs=fs, ws=ws)


def l2_note(fmin):
    return ("inputs (%.1f GB) larger than L2 (129 MB); no flush" % (fmin / 1e9) if fmin >= 1e9 else
            "inputs (%.2f GB) near the L2 size: a 512 MB buffer written between steps, outside the "
            "per-step events" % (fmin / 1e9))


def host_link(torch, h2d_bytes, d2h_bytes, reps=3):
    """Plain pinned-memory copies on this GPU's host link, the floor an
    end-to-end step cannot beat: one cudaMemcpyAsync each way of the step's
    bytes, alone and both directions at once (best of `reps`)."""
    src = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(h2d_bytes, dtype=torch.uint8, device="cuda")
    dsrc = torch.empty(d2h_bytes, dtype=torch.uint8, device="cuda")
    ddst = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn):
        best = None
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            t = a.elapsed_time(b)
            best = t if best is None else min(best, t)
        return best

    def both():
        cur = torch.cuda.current_stream()
        s1.wait_stream(cur)
        s2.wait_stream(cur)
        with torch.cuda.stream(s1):
            dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(s2):
            ddst.copy_(dsrc, non_blocking=True)
        cur.wait_stream(s1)
        cur.wait_stream(s2)

    h_ms = timed(lambda: dst.copy_(src, non_blocking=True))
    d_ms = timed(lambda: ddst.copy_(dsrc, non_blocking=True))
    b_ms = timed(both)
    del src, dst, dsrc, ddst
    return {"h2d_gbs": h2d_bytes / (h_ms * 1e-3) / 1e9, "d2h_gbs": d2h_bytes / (d_ms * 1e-3) / 1e9,
            "h2d_ms": h_ms, "d2h_ms": d_ms, "both_ms": b_ms,
            "how": "one pinned cudaMemcpyAsync of the step's bytes each way, alone and both at once "
                   "(two streams); best of %d" % reps}


def run_ours(args):
    import torch
    import torch.distributed as dist
    from gated_deltanet_prefill_gb300 import build as gbuild
    from gated_deltanet_prefill_gb300 import dist as gdist
    from gated_deltanet_prefill_gb300 import gdn2, inputs

    rank, world, local = gdist.rank_world()
    torch.cuda.set_device(local)
    # host threads and first-touch host pages near this GPU (pinned buffers of
    # the end-to-end leg land on the GPU's own NUMA node)
    near = gpu_numa_cpus(local)
    numa = None
    if near:
        try:
            os.sched_setaffinity(0, near)
            numa = "bound to the %d CPUs local to the GPU (sysfs local_cpulist)" % len(near)
        except Exception:
            numa = None
    if world > 1:
        dist.init_process_group("nccl")
    if rank == 0 or world == 1:
        gbuild.build()
    if world > 1:
        dist.barrier()
    gdn2.load()

    wl = inputs.workload(args.workload)
    if args.seqs > 0 and args.seqs < wl.N:
        import dataclasses
        wl = dataclasses.replace(wl, name="%s_first%d" % (wl.name, args.seqs), lens=wl.lens[:args.seqs])
    T = wl.T_tot
    K = args.steps
    rec, buf = measure(wl, args, K, args.warmup, seed_rank=rank, world=world, clocks_dev=local)
    d, ms, stage_ms, stages, whole = buf["d"], rec["ms"], rec["stage_ms"], rec["stages"], rec["whole_op"]
    dims, fmin, peak, peak_kind, sb = rec["dims"], rec["fmin"], rec["peak"], rec["peak_kind"], rec["sb"]
    stream = torch.cuda.current_stream()

    # roofline of the dominant kernel
    dom = max(stage_ms, key=stage_ms.get)
    ach = sb[dom] / (stage_ms[dom] * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
            "traffic": ncu_traffic(dom, args.kernels, wl.name), "kernel": dom,
            "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind if peak_kind == "measured"
            else "fallback 6.8 TB/s"}
    del buf["out"], buf["fs"], buf["ws"]

    # end-to-end from pinned host buffers through the public API
    e2e = None
    if not args.no_e2e:
        host = {k: (v.cpu().pin_memory() if torch.is_tensor(v) else v) for k, v in d.items()}
        runner = gdn2.HostRunner(host, impl=args.kernels)
        for _ in range(2):
            runner()
        torch.cuda.synchronize()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
        if world > 1:
            dist.barrier()
        evs[0].record(stream)
        for i in range(args.e2e_steps):
            runner()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        # the host link is shared with the machine's other GPUs: a step can
        # stall on a neighbour's copies, so the value uses the median step and
        # the mean, minimum and maximum are reported beside it
        per = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.e2e_steps)]
        ems = gdist.max_over_ranks(statistics.median(per), device="cuda")
        h2d, d2h = runner.h2d_bytes, runner.d2h_bytes
        del runner, host
        link = host_link(torch, h2d, d2h)
        # the step cannot beat the slower copy direction or the device step
        floor = max(link["h2d_ms"], link["d2h_ms"], ms)
        link["floor_ms"] = floor
        link["frac"] = floor / ems
        link["numa"] = numa or "not bound (no sysfs local_cpulist)"
        e2e = {"value": gdist.aggregate_throughput(T, world, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ems, "stat": "median of %d steps" % args.e2e_steps, "steps": args.e2e_steps,
               "warmup": 2, "ms_mean": evs[0].elapsed_time(evs[-1]) / args.e2e_steps,
               "ms_min": min(per), "ms_max": max(per), "ms_all": per, "host_link": link}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(d, wl, args.cpu_seconds)
    del d, buf

    # the other D = 128 workloads, timed the same way (the headline stays on
    # the long workload)
    configs = None
    if world == 1 and not args.no_configs:
        configs = {}
        for idx in (2, 3, 4):
            if idx == args.workload:
                continue
            wli = inputs.workload(idx)
            r, b = measure(wli, args, args.config_steps, args.warmup)
            c = {"workload": wli.name, "ms_per_step": r["ms"], "ms_per_step_staged": r["staged_ms"],
                 "tokens_per_s": wli.T_tot / (r["ms"] * 1e-3),
                 "steps": args.config_steps, "warmup": max(3, args.warmup), "l2": l2_note(r["fmin"]),
                 "stages": {n: {"ms": v["ms"], "frac_of_peak": v["frac_of_peak"]} for n, v in r["stages"].items()},
                 "whole_op_frac": r["whole_op"]["frac"], "device_status": r["status"],
                 "cpu_baseline": None if args.no_cpu_baseline else
                 cpu_baseline(b["d"], wli, args.config_cpu_seconds)}
            configs[wli.name] = c
            del b
            torch.cuda.empty_cache()

    if rank == 0:
        line = {"metric": METRIC, "value": gdist.aggregate_throughput(T, world, ms), "unit": "tokens/s",
                "n_gpus": world,
                "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if args.kernels == "tc" else "f32", "data": "synthetic",
                "config": {"workload": wl.name, "B": wl.N, "T": wl.lens[0], "H": wl.H, "HV": wl.HV,
                           "K": wl.K, "V": wl.V, "tokens_per_step_per_gpu": T, "kernels": args.kernels,
                           "g": "-U(0,%g)" % wl.g_max, "beta": "U(0,%g)" % wl.beta_max,
                           "initial_state": "N(0,%g)" % wl.h0_std if wl.h0_std else "zero",
                           "output_final_state": True, "l2": l2_note(fmin),
                           "state_segments": args.segments if args.segments else "chosen by the library",
                           "parallelism": "replicas x%d (independent batches)" % world},
                "ms_per_step_staged": rec["staged_ms"],
                "timing": "ms_per_step: steps with no event between their kernels (each launch overlaps its "
                          "predecessor's tail); stages: K more steps with an event between the stages, "
                          "ms_per_step_staged their sum",
                "roofline": roof, "stages": stages, "whole_op": whole, "e2e": e2e,
                "cpu_baseline": cpu, "gpu_launches": gdn2.launch_count(dims) * K,
                "device_status": rec["status"], "configs": configs,
                "clocks": rec["clocks"], "source_sha": kernel_source_sha()}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def decode_bytes(wl):
    """Algorithmic HBM bytes of one recurrent call: the state read and written
    once per (sequence, value head), each token's inputs read once (q, k per
    key head) and its output written once."""
    K, V = wl.K, wl.V
    per_tok_hv = V * 2 + V * 2 + K * 2 + K * 4 + V * 2          # v, w, beta, g, o
    per_tok_h = 2 * K * 2                                         # q, k
    state = (2 if wl.h0_std else 1) * wl.N * wl.HV * K * V * 4
    return state + wl.T_tot * (wl.HV * per_tok_hv + wl.H * per_tok_h)


def run_decode(args):
    """The token-by-token recurrence (decode) on one GPU: one JSON line with
    its own metric, roofline and oracle baseline (not the headline)."""
    import torch
    from gated_deltanet_prefill_gb300 import build as gbuild
    from gated_deltanet_prefill_gb300 import gdn2, inputs

    torch.cuda.set_device(0)
    gbuild.build()
    gdn2.load()
    wl = inputs.decode_workload(args.decode_batch, args.decode_tokens)
    d = inputs.generate(wl, device="cuda")
    out = torch.empty((wl.T_tot, wl.HV, wl.V), dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((wl.N, wl.HV, wl.K, wl.V), dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        gdn2.recurrent_gdn2_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["w"], scale=d["scale"],
                                initial_state=d["h0"], cu_seqlens=d["cu_seqlens"], out=out, final_state=fs,
                                workspace=ws)

    # warm up for >= 0.3 s as well as >= W steps: a decode step is ~0.1 ms, and
    # a few steps leave the GPU at its idle clocks when the timed region starts
    W, t0 = 0, time.perf_counter()
    while W < max(3, args.warmup) or time.perf_counter() - t0 < 0.3:
        for _ in range(50):
            step()
        W += 50
        torch.cuda.synchronize()
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(0) as clk:
        start.record(stream)
        for _ in range(K):
            step()
        end.record(stream)
        torch.cuda.synchronize()
    ms = start.elapsed_time(end) / K
    # the same step captured once into a CUDA graph and replayed K times
    # (launch overheads hidden: the way a serving loop would run it)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step()
    for _ in range(20):
        graph.replay()
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(K):
        graph.replay()
    end.record(stream)
    torch.cuda.synchronize()
    g_ms = start.elapsed_time(end) / K
    peak, peak_kind = load_peaks()
    nbytes = decode_bytes(wl)
    ach = nbytes / (ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
            "traffic": ncu_traffic("recurrent", "recurrent", wl.name), "kernel": "recurrent",
            "timed": "whole call (cu_seqlens check + recurrence), CUDA events",
            "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind if peak_kind == "measured"
            else "fallback 6.8 TB/s"}
    cpu = None if args.no_cpu_baseline else cpu_baseline(d, wl, args.cpu_seconds)
    line = {"metric": "GDN-2 decode tokens/s (token-by-token from a carried state)",
            "value": wl.T_tot / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": K,
            "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.N, "T": wl.lens[0], "H": wl.H, "HV": wl.HV, "K": wl.K,
                       "V": wl.V, "initial_state": "N(0,%g)" % wl.h0_std,
                       "l2": "state in + out (%.2f GB) larger than L2 (129 MB); no flush" % (nbytes / 1e9)},
            "roofline": roof, "e2e": None, "cpu_baseline": cpu, "gpu_launches": 2 * K,
            "graph": {"ms_per_step": g_ms, "value": wl.T_tot / (g_ms * 1e-3), "unit": "tokens/s",
                      "frac": nbytes / (g_ms * 1e-3) / 1e9 / peak},
            "clocks": clk.summary(), "source_sha": kernel_source_sha()}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "decode":
        run_decode(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
