"""Benchmark of the ReplaySSM GDN decode hot path on GB300.

One step = one pass of the hot path over one batch: the ReplaySSM decode of one
layer (tensor-core replay) and the cursor advance, in one launch
(gdn_replayssm_decode_advance, the call for a forward's last layer).  Workload (the metric's
configuration): HV=32, HK=16, K=V=128, L=16, fp32 checkpoint, fp16 d/k ring,
bf16 mixed_qkv and output, B=256 rows of a 512-slot pool, cursors staggered
uniformly over [0, L) so flush and append rows mix in every launch.  Every step
reads 512 MiB of checkpoint (4x the 129 MB L2), so no L2 flush is needed.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       [--workload headline|qwen3next_layer|kda_layer|kda_layer:L:f16|f32|stack30|stack30:B|sweep:B:L:f16|f32] [--recon tensor|ffma|output]
       [--kernel-only]   (timed decode loop only: for profiling and sweeps)
       [--sweep [--sweep-batches 1,8,...] [--sweep-lens 1,4,...]]  (one JSON line per point)
       [--spec [--spec-batches 64,256] [--spec-windows 2,4,8] [--spec-accept 0.7]]
                         (speculative verify window + commit + fold, one JSON line per point)
       [--graph [--graph-batches 1,8,64,256] [--graph-layers 30]]  (CUDA-graph replay vs one-by-one launches)
       [--lossless [--spec-batches ...] [--spec-windows ...]]
                         (lossless verify + exact-order commit, one JSON line per point)
Under torchrun each rank runs an independent replica on its own GPU (the
path has no exchange step); rank 0 prints one JSON line.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN decode head-steps/s & HBM GB/s vs 8 TB/s (HV=32,K=V=128,L=16,B=256)"
UNIT = "head-steps/s"
FALLBACK_HBM_GBS = 6800.0
PROFILE = os.path.join(ROOT, "profiles", "gdn_replayssm_decode_tc_B256_L16.md")
# everything the profiled kernel's code and launch depend on: a change to any
# of these marks the stored ncu traffic stale
KERNEL_SOURCES = ([os.path.join(ROOT, "linear_attention_decode_gb300", "csrc", f)
                   for f in ("gdn_tcp.cu", "gdn_tc_common.cuh", "gdn_common.cuh", "gdn_kernels.h", "gdn_tc.cu",
                             "gdn_api.cu")]
                  + [os.path.join(ROOT, "include", "gdnreplay.h")])


# ---------------------------------------------------------------------------
# Algorithmic bytes (host logic, also checked by the CPU tests).
# ---------------------------------------------------------------------------

def head_step_parts(K, V, G, p, flush, rb, ib, ob, kda=False):
    """Bytes one (row, value head) must move, by part: the checkpoint read and
    (on a flush) write, the p valid ring entries read plus the append, the
    inputs, the output.  A key head's ring entries and inputs are shared by
    its G value heads."""
    g_entry = 4 * K if kda else 4
    ring_entry = V * rb + K * rb / G + g_entry
    return {"state": 4 * V * K + (4 * V * K if flush else 0),
            "ring": p * ring_entry + (0 if flush else ring_entry),
            "inputs": 2 * K * ib / G + V * ib + g_entry + 4,
            "output": V * ob}


def head_step_bytes(K, V, G, p, flush, rb, ib, ob, kda=False):
    return sum(head_step_parts(K, V, G, p, flush, rb, ib, ob, kda).values())


def packed_head_step_bytes(K, V, G, ib, ob, kda=False):
    """Packed decode: the state is read and written every step."""
    g_entry = 4 * K if kda else 4
    return 8 * V * K + 2 * K * ib / G + V * ib + g_entry + 4 + V * ob


def spec_head_bytes(K, V, G, p, T, rb, ib, ob, kda=False):
    """Bytes one (row, value head) must move in a verify window of T tokens at
    cursor p: the checkpoint read, the p committed ring entries read, the T
    window entries written, T tokens of inputs and of output."""
    g_entry = 4 * K if kda else 4
    ring_entry = V * rb + K * rb / G + g_entry
    return (4 * V * K + (p + T) * ring_entry + T * (2 * K * ib / G + V * ib + g_entry + 4)
            + T * V * ob)


def fold_head_bytes(K, V, G, p, rb, kda=False):
    """Bytes of folding p ring entries of one (slot, value head) into its
    checkpoint: the checkpoint read and written, the entries read."""
    g_entry = 4 * K if kda else 4
    return 8 * V * K + p * (V * rb + K * rb / G + g_entry)


def lossless_verify_head_bytes(K, V, G, T, ib, ob, kda=False):
    """Bytes one (row, value head) must move in a lossless verify of T tokens:
    the state read once, T tokens of inputs and of output, T fp32 tuples
    written (u per value head, k once per key head, g)."""
    g_entry = 4 * K if kda else 4
    return (4 * V * K + T * (2 * K * ib / G + V * ib + g_entry + 4 + V * ob)
            + T * (4 * V + 4 * K / G + g_entry))


def lossless_commit_head_bytes(K, V, G, a, kda=False):
    """Exact-order commit of a tuples into one (slot, value head) in place: the
    state read and written and the a tuples read; nothing when a = 0."""
    if a <= 0:
        return 0.0
    g_entry = 4 * K if kda else 4
    return 8 * V * K + a * (4 * V + 4 * K / G + g_entry)


def launch_bytes(w, p_rows, flush_rows, ob, n_pad, cursors=True):
    """Algorithmic bytes of one decode (+ cursor advance) launch; padding rows
    only write zeros; each live row's cursor is read and written once."""
    rb = 4 if w.ring_dtype == 0 else 2
    ib = 4 if w.qkv_dtype == 0 else 2
    G = w.HV // w.HK
    kda = w.gate == 1
    total = 0.0
    for p, f in zip(p_rows, flush_rows):
        total += w.HV * head_step_bytes(w.K, w.V, G, int(p), bool(f), rb, ib, ob, kda)
    return total + n_pad * w.HV * w.V * ob + (8 * len(p_rows) if cursors else 0)


# ---------------------------------------------------------------------------
# Environment helpers.
# ---------------------------------------------------------------------------

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != kernel_source_hash():
        return None
    return float(m_b.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Arms.
# ---------------------------------------------------------------------------

def max_over_ranks(x: float, device) -> float:
    """The slowest rank's time (the job is done when every replica is done)."""
    import torch
    import torch.distributed as dist
    if not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world_size: int, max_elapsed_s: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return world_size * units_per_rank / max_elapsed_s


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class OracleSample:
    """The CPU oracle as it stands (single thread) on a small pool of the
    workload's shapes: each call decodes `rows` rows x HV heads for one step."""

    def __init__(self, w, pool_rows=16, seed_offset=0):
        import numpy as np

        import oracle as O
        from linear_attention_decode_gb300 import inputs as I

        oracle_dt = {0: O.F32, 1: O.BF16, 2: O.F16}[w.ring_dtype]
        self.w, self.np, self.O, self.I = w, np, O, I
        self.pool = pool_rows
        self.sw = I.with_(w, N=pool_rows, B=pool_rows, n_pad=0)
        self.gen = I.generator(w.seed + 100 + seed_offset, "cpu")
        wp = I.write_pos(self.gen, self.sw, "cpu")
        c = I.cache(self.gen, self.sw, wp, "cpu")
        self.G = O.geom(pool_rows, w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, state_dtype=O.F32,
                        ring_dtype=oracle_dt)
        self.cache = O.Cache.from_arrays(c.state, c.ring_d, c.ring_k, c.ring_g)
        self.wp = wp.numpy().astype(np.int32).copy()
        self.inputs = [I.step_inputs(self.gen, self.sw, "cpu") for _ in range(4)]
        self.next_row = 0
        self.calls = 0

    def step(self, rows):
        np, O = self.np, self.O
        idx = (self.next_row + np.arange(rows)) % self.pool
        self.next_row = int((self.next_row + rows) % self.pool)
        si = self.inputs[self.calls % len(self.inputs)]
        self.calls += 1
        t0 = time.perf_counter()
        O.replay_decode(self.G, self.cache, self.wp, idx.astype(np.int32), None, si.mixed_qkv[idx],
                        si.g[idx], si.beta[idx])
        O.replay_advance(self.pool, idx.astype(np.int32), None, self.w.L, self.wp)
        return time.perf_counter() - t0


def host_cpu_info():
    """The host's thread count (what std::thread::hardware_concurrency reports),
    the threads this process may use, and the CPU model from /proc/cpuinfo."""
    info = {"hardware_concurrency": os.cpu_count(), "usable_threads": len(os.sched_getaffinity(0))}
    model = None
    try:
        text = open("/proc/cpuinfo").read()
        m = re.search(r"^model name\s*:\s*(.+)$", text, re.M)
        if m:
            model = m.group(1).strip()
        else:  # Arm: the implementer and part codes
            imp = re.search(r"^CPU implementer\s*:\s*(\S+)", text, re.M)
            part = re.search(r"^CPU part\s*:\s*(\S+)", text, re.M)
            if imp and part:
                known = {("0x41", "0xd4f"): "Arm Neoverse-V2"}
                model = known.get((imp.group(1), part.group(1)),
                                  f"CPU implementer {imp.group(1)}, part {part.group(1)}")
    except OSError:
        pass
    info["model"] = model or "unknown"
    return info


def cpu_oracle_timing(w, seconds_target=10.0, rows=16, threads=1):
    """The oracle as it stands on a bounded sample of the workload: `threads`
    host threads, each decoding its own pool of `rows` slots step after step
    (the oracle's C code runs with the GIL released, so the threads use
    separate cores) for about seconds_target of wall time.  Head-steps per
    second of wall time, Python marshalling included."""
    samples = [OracleSample(w, pool_rows=rows, seed_offset=i) for i in range(threads)]
    counts = [0] * threads
    go = threading.Barrier(threads + 1)
    stop_at = [0.0]

    def work(i):
        go.wait()
        while time.perf_counter() < stop_at[0]:
            samples[i].step(rows)
            counts[i] += 1

    pool = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
    for t in pool:
        t.start()
    t0 = time.perf_counter()
    stop_at[0] = t0 + seconds_target
    go.wait()
    for t in pool:
        t.join()
    wall = time.perf_counter() - t0
    steps = sum(counts)
    ring = {0: "fp32", 1: "bf16", 2: "fp16"}[w.ring_dtype]
    return {"value": rows * w.HV * steps / wall, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{threads} thread(s) x {rows} rows x {w.HV} heads, {steps} steps in all, of the "
                      f"workload's shapes (K=V={w.K}, L={w.L}, {ring} ring, staggered cursors), {wall:.1f} s"}


def cpu_baseline_report(w, seconds=8.0, rows=16):
    """cpu_baseline of the bench line: the oracle on the workload over all the
    host's usable threads, and single-threaded, plus the same pair on the tiny
    configuration and the one-layer configuration (shorter samples)."""
    from linear_attention_decode_gb300 import inputs as I
    host = host_cpu_info()
    n = host["usable_threads"]
    main = cpu_oracle_timing(w, seconds, rows, threads=n)
    main["single_thread"] = cpu_oracle_timing(w, seconds, rows, threads=1)
    main["host"] = host
    by = {}
    for name, wc, r in (("tiny_N8_B4_HV4_K64_L4_fp32", I.with_(I.TINY, staggered=True), 64),
                        ("one_layer_B64_HV32_K128_L16_fp16", I.with_(I.QWEN3NEXT_LAYER, staggered=True), rows)):
        by[name] = {"all_threads": cpu_oracle_timing(wc, seconds / 3, r, threads=n),
                    "single_thread": cpu_oracle_timing(wc, seconds / 3, r, threads=1)}
    main["by_config"] = by
    return main


def run_reference(args):
    """Reference arm: the CPU oracle timed step by step on the same workload;
    each step is a bounded sample (rows per step sized so the run stays within
    about a minute)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from linear_attention_decode_gb300 import inputs as I
    oracle.build()
    w = I.HEADLINE
    host = host_cpu_info()
    nth = host["usable_threads"]
    # each step: every thread decodes `rows` rows of its own 16-slot pool (the
    # threads run the oracle's C code side by side on separate cores)
    samples = [OracleSample(w, seed_offset=i) for i in range(nth)]
    t_row = max(samples[0].step(1) for _ in range(max(3, args.warmup)))
    rows = int(min(16, max(1, args.ref_budget / max(1, args.steps) / t_row)))

    def one_step():
        ths = [threading.Thread(target=smp.step, args=(rows,)) for smp in samples]
        for t in ths:
            t.start()
        for t in ths:
            t.join()

    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    t_total = time.perf_counter() - t0
    value = args.steps * nth * rows * w.HV / t_total
    cpu = {"value": value, "unit": UNIT, "cores": nth, "kind": "oracle", "host": host,
           "sample": f"{args.steps} steps x {nth} threads x {rows} rows x {w.HV} heads (a pool of 16 slots "
                     f"of the workload's shapes per thread), {t_total:.1f} s"}
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "rows_per_step": rows * nth},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def pick_workload(name):
    from linear_attention_decode_gb300 import inputs as I
    from linear_attention_decode_gb300.constants import BF16, F16, F32
    if name == "headline":
        return I.HEADLINE
    if name == "qwen3next_layer":
        return I.with_(I.QWEN3NEXT_LAYER, staggered=True)
    if name == "kda_layer":
        return I.with_(I.KDA_LAYER, staggered=True)
    if name.startswith("kda_layer:"):  # the KDA layer with another ring length / ring type
        _, L, rd = name.split(":")
        tag = {"f16": "fp16", "f32": "fp32", "bf16": "bf16"}[rd]
        return I.with_(I.KDA_LAYER, staggered=True, L=int(L), ring_dtype={"f16": F16, "f32": F32, "bf16": BF16}[rd],
                       name=f"KDA layer: N=256 B=128 HV=HK=32 K=V=128 L={L} {tag} ring bf16 qkv")
    if name == "stack30":
        return I.with_(I.STACK30, staggered=True)
    if name.startswith("stack30:"):  # the 30-layer stack at another batch (same 320-slot pool)
        B = int(name.split(":")[1])
        N = max(I.STACK30.N, B)
        return I.with_(I.STACK30, staggered=True, B=B, N=N,
                       name=f"30-layer stack: N={N} B={B} HV=32 HK=16 K=V=128 L=16 fp16 ring bf16 qkv")
    if name.startswith("sweep:"):
        _, B, L, rd = name.split(":")
        return I.sweep_point(int(B), int(L), {"f16": F16, "f32": F32, "bf16": BF16}[rd])
    raise SystemExit(f"unknown workload {name}")


def measure_replay(w, K, warmup, recon, dev, layers=1, overlap=False, extra_flags=0):
    """Kernel-only timing of K steps of `layers` layers sharing one cursor array:
    gdn_replayssm_decode on every layer but the last, gdn_replayssm_decode_advance
    on the last.  Inputs are resident on the device; nothing else runs between
    launches.  overlap: every layer but the first is launched with
    STEP_OVERLAP_PREVIOUS (true here: the launch before it is another layer's
    decode, which writes neither this layer's cache nor the cursors; the first
    layer follows the advance and waits).  Returns per-launch and per-step
    figures with the algorithmic bytes."""
    import numpy as np
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import inputs as I

    gen = I.generator(w.seed, dev)
    wp = I.write_pos(gen, w, dev)
    caches = []
    for _ in range(layers):
        c = I.cache(gen, w, wp, dev)
        caches.append(Bd.Cache(c.state, c.ring_d, c.ring_k, c.ring_g))
    idx = I.indices(gen, w.B, w.N, w.n_pad, dev)
    rows = idx.shape[0]
    desc = Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, ring_dtype=w.ring_dtype)
    pool = [I.step_inputs(gen, w, dev) for _ in range(4)]
    out = torch.empty((rows, w.HV, w.V), dtype=torch.bfloat16, device=dev)
    steps_in = [Bd.Step(b.mixed_qkv, b.g, b.beta, idx, out, flags=extra_flags) for b in pool]
    steps_ov = [Bd.Step(b.mixed_qkv, b.g, b.beta, idx, out, flags=Bd.STEP_OVERLAP_PREVIOUS | extra_flags)
                for b in pool]
    stream = torch.cuda.current_stream()
    adv_ws = Bd.decode_advance_workspace(dev)
    idx_h = idx.cpu().numpy()
    wp_h = wp.cpu().numpy().copy()
    ob = 2

    # every call checked and packed once (prepared calls), as a serving loop
    # would: small batches then time the launches, not the Python marshalling
    calls = []
    for j in range(len(steps_in)):
        si = steps_in[j]
        so = steps_ov[j] if overlap else si
        row = [Bd.prepare_replayssm_decode(desc, caches[layer], wp, None, si if layer == 0 else so, recon)
               for layer in range(layers - 1)]
        row.append(Bd.prepare_replayssm_decode(desc, caches[-1], wp, None, si if layers == 1 else so, recon, adv_ws))
        calls.append(row)
    h = stream.cuda_stream

    def step(i):
        for c in calls[i % len(calls)]:
            c.run(h)

    def host_advance():
        live = idx_h[idx_h >= 0]
        p = wp_h[live]
        wp_h[live] = np.where(p == w.L - 1, 0, p + 1)

    # host bookkeeping (the warm-up steps' cursor moves, then every timed
    # launch's bytes) before the warm-up launches, which then run right before
    # the timed region: a GPU left idle even for milliseconds pays extra on its
    # next launch
    for i in range(warmup):
        host_advance()
    total = 0.0
    for i in range(K):
        live = idx_h[idx_h >= 0]
        p = wp_h[live]
        per_layer = launch_bytes(w, p, p == w.L - 1, ob, int((idx_h < 0).sum()), cursors=False)
        total += layers * per_layer + 8 * len(live)
        host_advance()
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(K):
        step(i)
    b.record(stream)
    torch.cuda.synchronize()
    assert np.array_equal(wp.cpu().numpy(), wp_h), "device cursors diverged from the advance rule"
    step_s = a.elapsed_time(b) / 1e3 / K
    launch_s = step_s / layers
    peak, _ = measured_hbm_peak()
    gbs = total / K / step_s / 1e9
    r0 = Bd.gdn_replayssm_decode_kernel(desc, caches[0], steps_in[0], recon)
    kname = {Bd.KERNEL_PERSISTENT_TC: "persistent_tc", Bd.KERNEL_PER_HEAD_TC: "per_head_tc",
             Bd.KERNEL_CUDA_CORE: "cuda_core", Bd.KERNEL_SMALL_BATCH: "small_batch"}[r0]
    return {"workload": w.name, "kernel": kname, "layers": layers, "overlap_previous": bool(overlap and layers > 1),
            "B": w.B, "L": w.L,
            "ring": {0: "f32", 1: "bf16", 2: "f16"}[w.ring_dtype], "steps": K,
            "ms_per_step": step_s * 1e3, "ms_per_launch": launch_s * 1e3,
            "head_steps_per_s_per_layer": w.B * w.HV / launch_s, "tokens_per_s_per_layer": w.B / launch_s,
            "algorithmic_bytes_per_step": total / K, "hbm_gbs_algorithmic": gbs, "frac": gbs / peak,
            "frac_of_8tbs": gbs / 8000.0}


def measure_packed(w, K, dev):
    """The in-repo packed decode (reads and writes the state every step) on the
    workload's shapes: kernel-only, K launches back to back.  The state pool
    holds at least four times the batch's slots and consecutive launches use
    four disjoint slot sets in turn, so no launch finds its states in L2."""
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import inputs as I

    gen = I.generator(w.seed + 7, dev)
    N = max(w.N, 4 * w.B)
    st = I.state(gen, N, w.HV, w.V, w.K, dev)
    perm = torch.randperm(N, generator=gen, device=dev).to(torch.int32)
    sets = []
    for j in range(4):
        idx = torch.full((w.B + w.n_pad,), -1, dtype=torch.int32, device=dev)
        live = torch.randperm(w.B + w.n_pad, generator=gen, device=dev)[:w.B]
        idx[live] = perm[j * w.B:(j + 1) * w.B]
        sets.append(idx)
    rows = w.B + w.n_pad
    desc = Bd.layer_desc(N, w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, ring_dtype=w.ring_dtype)
    si = I.step_inputs(gen, w, dev)
    out = torch.empty((rows, w.HV, w.V), dtype=torch.bfloat16, device=dev)
    steps = [Bd.Step(si.mixed_qkv, si.g, si.beta, idx, out) for idx in sets]
    stream = torch.cuda.current_stream()
    calls = [Bd.prepare_packed_decode(desc, st, stp) for stp in steps]  # as the replay side: prepared calls
    h = stream.cuda_stream
    for i in range(8):
        calls[i % 4].run(h)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(K):
        calls[i % 4].run(h)
    b.record(stream)
    torch.cuda.synchronize()
    s = a.elapsed_time(b) / 1e3 / K
    nbytes = (w.B * w.HV * packed_head_step_bytes(w.K, w.V, w.HV // w.HK, 2, 2, w.gate == Bd.GATE_PER_K)
              + (rows - w.B) * w.HV * w.V * 2)
    peak, _ = measured_hbm_peak()
    return {"ms_per_launch": s * 1e3, "head_steps_per_s": w.B * w.HV / s, "tokens_per_s": w.B / s,
            "hbm_gbs_algorithmic": nbytes / s / 1e9, "frac": nbytes / s / 1e9 / peak}


def run_packed(args):
    """Kernel-only timing of the in-repo packed decode (gdn_packed_decode, the
    read + write baseline) on the workload's shapes: one JSON line."""
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import build as cuda_build

    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    cuda_build.build()
    Bd.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = pick_workload(args.workload)
    r = measure_packed(w, args.steps, dev)
    r.update({"workload": w.name, "kernel": "gdn_packed_decode", "steps": args.steps})
    print(json.dumps(r))
    return 0


def run_sweep(args):
    """Batch x ring-length x ring-dtype sweep of one GDN layer (HV=32, HK=16,
    K=V=128, staggered cursors): one JSON line per point, the replay decode +
    advance beside the packed decode on the same batch size."""
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import build as cuda_build
    from linear_attention_decode_gb300 import inputs as I
    from linear_attention_decode_gb300.constants import F16, F32

    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    cuda_build.build()
    Bd.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    batches = [int(x) for x in args.sweep_batches.split(",")]
    lens = [int(x) for x in args.sweep_lens.split(",")]
    rings = [{"f16": F16, "f32": F32}[x] for x in args.sweep_rings.split(",")]
    packed = {}
    for B in batches:
        for L in lens:
            for ring in rings:
                w = I.sweep_point(B, L, ring)
                K = max(2 * L * 8, 128) // args.sweep_layers + 1
                r = measure_replay(w, K, max(args.warmup, 2 * L), Bd.RECON_TENSOR, dev, layers=args.sweep_layers,
                                   overlap=args.sweep_layers > 1 and not args.no_overlap,
                                   extra_flags=Bd.STEP_PERSISTENT_KERNEL if args.persistent_kernel else 0)
                if B not in packed:
                    packed[B] = measure_packed(w, 64, dev)
                r["packed"] = packed[B]
                r["replay_speedup_vs_packed"] = packed[B]["ms_per_launch"] / r["ms_per_launch"]
                print(json.dumps(r), flush=True)
                torch.cuda.empty_cache()
    return 0


def acceptance_pool(rng, n, rows, T, rate):
    """Accepted counts per row for n windows: drafts are accepted one by one
    with probability `rate` until the first rejection (a in [0, T])."""
    import numpy as np
    acc = np.zeros((n, rows), dtype=np.int32)
    alive = np.ones((n, rows), dtype=bool)
    for _ in range(T):
        alive &= rng.random((n, rows)) < rate
        acc += alive
    return acc


def measure_spec(B, T, K, warmup, dev, rate=0.7, L=16, recon=None):
    """One layer of speculative decoding at the benchmark's layer shape
    (HV=32, HK=16, K=V=128, fp16 ring, bf16 inputs and output), B rows: each
    timed window is gdn_replayssm_spec_verify of T tokens per row, the commit of
    a seeded acceptance draw, and the fold + cursor reset of the slots the
    commit lists.  Kernel-only (inputs resident).  Also times the verify launch
    alone and T single-token decode + advance steps for comparison."""
    import numpy as np
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import inputs as I

    recon = Bd.RECON_TENSOR if recon is None else recon
    w = I.Workload(f"spec window: N={max(B, 512)} B={B} T={T} HV=32 HK=16 K=V=128 L={L} fp16 ring bf16 qkv",
                   N=max(B, 512), B=B, HV=32, HK=16, K=128, L=L, ring_dtype=Bd.F16, qkv_dtype=Bd.BF16, seed=5)
    gen = I.generator(w.seed, dev)
    wp = torch.randint(0, L - T, (w.N,), generator=gen, device=dev, dtype=torch.int32)
    c = I.cache(gen, w, wp, dev)
    cache = Bd.Cache(c.state, c.ring_d, c.ring_k, c.ring_g)
    idx = I.indices(gen, w.B, w.N, 0, dev)
    desc = Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, ring_dtype=w.ring_dtype)
    pool = [I.step_inputs(gen, w, dev, rows=B * T) for _ in range(4)]
    out = torch.empty((B * T, w.HV, w.V), dtype=torch.bfloat16, device=dev)
    steps_in = [Bd.Step(b.mixed_qkv, b.g, b.beta, idx, out) for b in pool]
    acc_h = acceptance_pool(np.random.default_rng(w.seed), 16, B, T, rate)
    acc_dev = [torch.from_numpy(a).to(dev) for a in acc_h]
    fs = torch.empty(B, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    idx_h = idx.cpu().numpy()
    wp_h = wp.cpu().numpy().copy()
    G = w.HV // w.HK

    def window(i):
        Bd.gdn_replayssm_spec_verify(desc, cache, wp, T, steps_in[i % 4], recon, status, stream)
        Bd.gdn_replayssm_spec_commit(idx, acc_dev[i % 16], T, w.N, L, wp, fs, status, stream)
        Bd.gdn_replayssm_flush(desc, cache, wp, fs, status, stream)
        Bd.gdn_replayssm_reset_slots(wp, fs, status, stream)

    def host_window(i):
        """The window's algorithmic bytes; moves the host copy of the cursors."""
        p = wp_h[idx_h]
        nb = w.HV * sum(spec_head_bytes(w.K, w.V, G, int(x), T, 2, 2, 2) for x in p)
        a = acc_h[i % 16]
        nb += 16 * B  # commit: cursor read + write, accepted read, fold-list write
        q = p + a
        fold = q + T > L - 1
        nb += w.HV * sum(fold_head_bytes(w.K, w.V, G, int(x), 2) for x in q[fold]) + 4 * int(fold.sum())
        wp_h[idx_h] = np.where(fold, 0, q)
        return nb, int(a.sum()), int(fold.sum())

    for i in range(warmup):
        window(i)
        host_window(i)
    total = accepted = folds = 0
    for i in range(warmup, warmup + K):
        nb, na, nf = host_window(i)
        total += nb
        accepted += na
        folds += nf
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record(stream)
    for i in range(warmup, warmup + K):
        window(i)
    ev[1].record(stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    assert np.array_equal(wp.cpu().numpy(), wp_h), "device cursors diverged from the commit rule"
    win_s = ev[0].elapsed_time(ev[1]) / 1e3 / K
    # the verify launch alone, at the cursors the loop left (verify moves none)
    vb = w.HV * sum(spec_head_bytes(w.K, w.V, G, int(x), T, 2, 2, 2) for x in wp_h[idx_h])
    nv = max(K // 2, 16)
    ev[2].record(stream)
    for i in range(nv):
        Bd.gdn_replayssm_spec_verify(desc, cache, wp, T, steps_in[i % 4], recon, status, stream)
    ev[3].record(stream)
    torch.cuda.synchronize()
    ver_s = ev[2].elapsed_time(ev[3]) / 1e3 / nv
    peak, _ = measured_hbm_peak()
    dec = measure_replay(I.sweep_point(B, L, Bd.F16), max(K, 2 * L), 2 * L, Bd.RECON_TENSOR, dev)
    return {"workload": w.name, "B": B, "T": T, "L": L, "acceptance_rate_per_draft": rate, "windows": K,
            "ms_per_window": win_s * 1e3, "mean_accepted": accepted / K / B, "folds_per_window": folds / K,
            "verified_tokens_per_s": B * T / win_s, "accepted_tokens_per_s": accepted / K / win_s,
            "algorithmic_bytes_per_window": total / K, "window_hbm_gbs_algorithmic": total / K / win_s / 1e9,
            "verify_ms_per_launch": ver_s * 1e3, "verify_hbm_gbs_algorithmic": vb / ver_s / 1e9,
            "verify_frac": vb / ver_s / 1e9 / peak, "verify_frac_of_8tbs": vb / ver_s / 1e9 / 8000.0,
            "decode_ms_per_step": dec["ms_per_launch"],
            "window_vs_T_decode_steps": T * dec["ms_per_launch"] / (win_s * 1e3)}


def run_spec(args):
    """Speculative-window sweep: one JSON line per (batch, window)."""
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import build as cuda_build

    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    cuda_build.build()
    Bd.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    for B in [int(x) for x in args.spec_batches.split(",")]:
        for T in [int(x) for x in args.spec_windows.split(",")]:
            if args.recon == "output":
                raise SystemExit("--spec verifies with --recon tensor or ffma")
            recon = Bd.RECON_FFMA if args.recon == "ffma" else Bd.RECON_TENSOR
            r = measure_spec(B, T, max(args.steps, 32), args.warmup, dev, rate=args.spec_accept, recon=recon)
            r["recon"] = args.recon
            print(json.dumps(r), flush=True)
            torch.cuda.empty_cache()
    return 0


def measure_lossless(B, T, K, warmup, dev, rate=0.7):
    """Lossless verify + exact-order commit of one GDN layer (HV=32, HK=16,
    K=V=128, fp32 state, bf16 inputs and output), B rows of T tokens: each timed
    window is gdn_lossless_verify and gdn_lossless_commit of a seeded acceptance
    draw, in place.  Four disjoint slot sets rotate so no window finds its
    states in L2.  Kernel-only (inputs resident); also times each launch alone
    and one packed decode step."""
    import numpy as np
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import inputs as I

    N = 4 * B
    w = I.Workload(f"lossless window: N={N} B={B} T={T} HV=32 HK=16 K=V=128 fp32 state bf16 qkv",
                   N=N, B=B, HV=32, HK=16, K=128, L=1, ring_dtype=Bd.F32, qkv_dtype=Bd.BF16, seed=6)
    gen = I.generator(w.seed, dev)
    state = I.state(gen, w.N, w.HV, w.V, w.K, dev)
    perm = torch.randperm(N, generator=gen, device=dev).to(torch.int32)
    idx_sets = [perm[i * B:(i + 1) * B].contiguous() for i in range(4)]
    desc = Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, 1)
    pool = [I.step_inputs(gen, w, dev, rows=B * T) for _ in range(4)]
    out = torch.empty((B * T, w.HV, w.V), dtype=torch.bfloat16, device=dev)
    su, sk, sg = Bd.tuple_shapes(desc, B, T)
    tu, tk, tg = (torch.empty(su, device=dev), torch.empty(sk, device=dev), torch.empty(sg, device=dev))
    acc_h = acceptance_pool(np.random.default_rng(w.seed), 16, B, T, rate)
    acc_dev = [torch.from_numpy(a).to(dev) for a in acc_h]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    G = w.HV // w.HK

    def verify(i):
        b = pool[i % 4]
        Bd.gdn_lossless_verify(desc, state, T, Bd.Step(b.mixed_qkv, b.g, b.beta, idx_sets[i % 4], out),
                               tu, tk, tg, status, stream)

    def commit(i):
        Bd.gdn_lossless_commit(desc, state, idx_sets[i % 4], acc_dev[i % 16], T, tu, tk, tg, None, status, stream)

    vbytes = B * w.HV * lossless_verify_head_bytes(w.K, w.V, G, T, 2, 2)
    cbytes = [w.HV * sum(lossless_commit_head_bytes(w.K, w.V, G, int(a)) for a in acc_h[j]) + 8 * B
              for j in range(16)]

    def timed(fn, n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    for i in range(warmup):
        verify(i)
        commit(i)
    win_s = timed(lambda i: (verify(i), commit(i)), K)
    ver_s = timed(verify, K)
    com_s = timed(commit, K)
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    com_bytes = float(np.mean([cbytes[i % 16] for i in range(K)]))
    pk = Bd.Step(pool[0].mixed_qkv[:B], pool[0].g[:B], pool[0].beta[:B], idx_sets[0],
                 torch.empty((B, w.HV, w.V), dtype=torch.bfloat16, device=dev))
    pk_s = timed(lambda i: Bd.gdn_packed_decode(desc, state, pk, None, stream), max(K // 4, 16))
    peak, _ = measured_hbm_peak()
    snap = B * w.HV * (4 * w.V * w.K * (1 + T))  # a snapshot verify: state read + T snapshots written
    return {"workload": w.name, "B": B, "T": T, "acceptance_rate_per_draft": rate, "windows": K,
            "mean_accepted": float(acc_h.mean()), "ms_per_window": win_s * 1e3,
            "verified_tokens_per_s": B * T / win_s,
            "verify_ms_per_launch": ver_s * 1e3, "verify_algorithmic_bytes": vbytes,
            "verify_hbm_gbs_algorithmic": vbytes / ver_s / 1e9, "verify_frac": vbytes / ver_s / 1e9 / peak,
            "commit_ms_per_launch": com_s * 1e3, "commit_algorithmic_bytes": com_bytes,
            "commit_hbm_gbs_algorithmic": com_bytes / com_s / 1e9, "commit_frac": com_bytes / com_s / 1e9 / peak,
            "snapshot_verify_bytes_over_lossless": snap / vbytes,
            "packed_decode_ms_per_step": pk_s * 1e3}


def measure_graph(B, n, warmup, dev, extra_flags=0):
    """One GDN layer's decode + advance at batch B (L=16, fp16 ring): n steps
    launched one by one, against the same n steps captured once in a CUDA graph
    and replayed (the library allocates nothing and never synchronises, so its
    calls capture).  Kernel-only, inputs resident."""
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import inputs as I

    w = I.sweep_point(B, 16, Bd.F16)
    gen = I.generator(w.seed, dev)
    wp = I.write_pos(gen, w, dev)
    c = I.cache(gen, w, wp, dev)
    cache = Bd.Cache(c.state, c.ring_d, c.ring_k, c.ring_g)
    idx = I.indices(gen, w.B, w.N, w.n_pad, dev)
    desc = Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, ring_dtype=w.ring_dtype)
    out = torch.empty((idx.shape[0], w.HV, w.V), dtype=torch.bfloat16, device=dev)
    steps_in = [Bd.Step(b.mixed_qkv, b.g, b.beta, idx, out, flags=extra_flags)
                for b in (I.step_inputs(gen, w, dev) for _ in range(4))]
    ws = Bd.decode_advance_workspace(dev)

    def seq(stream):
        for i in range(n):
            Bd.gdn_replayssm_decode_advance(desc, cache, wp, None, steps_in[i % 4], ws, Bd.RECON_TENSOR, None, None,
                                            stream)

    def timed(fn, stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    cur = torch.cuda.current_stream()
    for _ in range(max(1, warmup // n + 1)):
        seq(cur)
    eager_us = timed(lambda: seq(cur), cur)
    graph = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(cs):
        with torch.cuda.graph(graph, stream=cs):
            seq(cs)
    graph.replay()
    torch.cuda.synchronize()
    graph_us = timed(graph.replay, cur)
    kernel = Bd.gdn_replayssm_decode_kernel(desc, cache, steps_in[0], Bd.RECON_TENSOR)

    # the packed decode on the same batch, one by one and as a graph (its own state pool)
    pstate = I.state(gen, w.N, w.HV, w.V, w.K, dev)

    def pseq(stream):
        for i in range(n):
            Bd.gdn_packed_decode(desc, pstate, steps_in[i % 4], None, stream)

    for _ in range(max(1, warmup // n + 1)):
        pseq(cur)
    p_eager_us = timed(lambda: pseq(cur), cur)
    pgraph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cs):
        with torch.cuda.graph(pgraph, stream=cs):
            pseq(cs)
    pgraph.replay()
    torch.cuda.synchronize()
    p_graph_us = timed(pgraph.replay, cur)
    return {"workload": w.name, "B": B, "kernel": {0: "persistent_tc", 1: "per_head_tc", 3: "small_batch"}.get(kernel),
            "steps_per_graph": n, "eager_us_per_step": eager_us,
            "graph_us_per_step": graph_us, "graph_head_steps_per_s": B * w.HV / (graph_us * 1e-6),
            "graph_vs_eager": eager_us / graph_us,
            "packed_eager_us_per_step": p_eager_us, "packed_graph_us_per_step": p_graph_us,
            "eager_vs_packed": p_eager_us / eager_us, "graph_vs_packed_graph": p_graph_us / graph_us}


def measure_graph_stack(B, layers, n, warmup, dev):
    """A model's decode steps at batch B: `layers` GDN layers (L=16, fp16 ring,
    each with its own cache and one cursor array), one step = gdn_replayssm_decode
    on every layer but the last (every layer after the first with
    STEP_OVERLAP_PREVIOUS: the launch before it is another layer's decode) and
    gdn_replayssm_decode_advance on the last; against the packed decode on every
    layer (its own state pools).  n steps launched one by one (prepared calls on
    both sides) and as one captured CUDA graph; per-layer times.  Kernel-only,
    inputs resident."""
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import inputs as I

    w = I.with_(I.sweep_point(B, 16, Bd.F16), N=max(B, 16))
    gen = I.generator(w.seed, dev)
    wp = I.write_pos(gen, w, dev)
    caches, pstates = [], []
    for _ in range(layers):
        c = I.cache(gen, w, wp, dev)
        caches.append(Bd.Cache(c.state, c.ring_d, c.ring_k, c.ring_g))
        pstates.append(I.state(gen, w.N, w.HV, w.V, w.K, dev))
    idx = I.indices(gen, w.B, w.N, w.n_pad, dev)
    desc = Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, ring_dtype=w.ring_dtype)
    out = torch.empty((idx.shape[0], w.HV, w.V), dtype=torch.bfloat16, device=dev)
    ins = [I.step_inputs(gen, w, dev) for _ in range(2)]
    first = [Bd.Step(b.mixed_qkv, b.g, b.beta, idx, out) for b in ins]
    later = [Bd.Step(b.mixed_qkv, b.g, b.beta, idx, out, flags=Bd.STEP_OVERLAP_PREVIOUS) for b in ins]
    ws = Bd.decode_advance_workspace(dev)

    # every call prepared once (checked and packed), as a serving loop would,
    # on both sides, so the eager numbers compare launches, not marshalling
    rcalls = [[Bd.prepare_replayssm_decode(desc, caches[layer], wp, None, (first if layer == 0 else later)[k],
                                           Bd.RECON_TENSOR, ws if layer == layers - 1 else None)
               for layer in range(layers)] for k in range(2)]
    pcalls = [[Bd.prepare_packed_decode(desc, pstates[layer], first[k]) for layer in range(layers)]
              for k in range(2)]

    def seq(stream):
        h = stream.cuda_stream
        for i in range(n):
            for layer in range(layers):
                rcalls[(i + layer) % 2][layer].run(h)

    def pseq(stream):
        h = stream.cuda_stream
        for i in range(n):
            for layer in range(layers):
                pcalls[(i + layer) % 2][layer].run(h)

    def timed(fn, stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (n * layers)

    cur = torch.cuda.current_stream()
    res = {}
    for name, f in (("replay", seq), ("packed", pseq)):
        for _ in range(max(1, warmup // n + 1)):
            f(cur)
        eager = timed(lambda: f(cur), cur)
        graph = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(cs):
            with torch.cuda.graph(graph, stream=cs):
                f(cs)
        graph.replay()
        torch.cuda.synchronize()
        res[name] = (eager, timed(graph.replay, cur))
    kernel = Bd.gdn_replayssm_decode_kernel(desc, caches[0], later[0], Bd.RECON_TENSOR)
    return {"workload": f"{layers}-layer stack: N={w.N} B={B} HV={w.HV} HK={w.HK} K=V={w.K} L={w.L} fp16 ring bf16 qkv",
            "B": B, "layers": layers,
            "kernel": {0: "persistent_tc", 1: "per_head_tc", 3: "small_batch"}.get(kernel),
            "steps_per_graph": n, "eager_us_per_layer": res["replay"][0], "graph_us_per_layer": res["replay"][1],
            "packed_eager_us_per_layer": res["packed"][0], "packed_graph_us_per_layer": res["packed"][1],
            "eager_vs_packed": res["packed"][0] / res["replay"][0],
            "graph_vs_packed_graph": res["packed"][1] / res["replay"][1]}


def run_graph(args):
    """CUDA-graph replay against one-by-one launches: one JSON line per batch."""
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import build as cuda_build

    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    cuda_build.build()
    Bd.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    for B in [int(x) for x in args.graph_batches.split(",")]:
        if args.graph_layers > 1:
            print(json.dumps(measure_graph_stack(B, args.graph_layers, 8, args.warmup, dev)), flush=True)
        else:
            print(json.dumps(measure_graph(B, 64, args.warmup, dev,
                                           Bd.STEP_PERSISTENT_KERNEL if args.persistent_kernel else 0)), flush=True)
        torch.cuda.empty_cache()
    return 0


def run_lossless(args):
    """Lossless verify + commit sweep: one JSON line per (batch, window)."""
    import torch

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import build as cuda_build

    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    cuda_build.build()
    Bd.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    for B in [int(x) for x in args.spec_batches.split(",")]:
        for T in [int(x) for x in args.spec_windows.split(",")]:
            r = measure_lossless(B, T, max(args.steps, 32), args.warmup, dev, rate=args.spec_accept)
            print(json.dumps(r), flush=True)
            torch.cuda.empty_cache()
    return 0


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from linear_attention_decode_gb300 import binding as Bd
    from linear_attention_decode_gb300 import build as cuda_build
    from linear_attention_decode_gb300 import inputs as I

    ws, rank, local = dist_env()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    cuda_build.build()
    Bd.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = pick_workload(args.workload)
    if args.workload.startswith("stack30"):
        # the 30-layer forward: 30 launches a step, the last one also advancing
        if not args.kernel_only:
            raise SystemExit("--workload stack30 is measured with --kernel-only")
        r = measure_replay(w, args.steps, args.warmup, Bd.RECON_TENSOR, dev, layers=w.layers,
                           overlap=not args.no_overlap)
        if rank == 0:
            print(json.dumps(r))
        if ws > 1:
            dist.destroy_process_group()
        return 0
    recon = {"ffma": Bd.RECON_FFMA, "output": Bd.RECON_OUTPUT}.get(args.recon, Bd.RECON_TENSOR)
    rb = 4 if w.ring_dtype == Bd.F32 else 2
    gen = I.generator(w.seed + rank, dev)
    wp = I.write_pos(gen, w, dev)
    c = I.cache(gen, w, wp, dev)
    cache = Bd.Cache(c.state, c.ring_d, c.ring_k, c.ring_g)
    idx = I.indices(gen, w.B, w.N, w.n_pad, dev)
    rows = idx.shape[0]
    desc = Bd.layer_desc(w.N, w.HV, w.HK, w.K, w.V, w.L, gate=w.gate, ring_dtype=w.ring_dtype)
    POOL = 8
    batches = [I.step_inputs(gen, w, dev) for _ in range(POOL)]
    out = torch.empty((rows, w.HV, w.V), dtype=torch.bfloat16, device=dev)
    steps_in = [Bd.Step(b.mixed_qkv, b.g, b.beta, idx, out) for b in batches]
    stream = torch.cuda.current_stream()

    # host mirror of the cursors for the per-launch algorithmic bytes
    idx_h = idx.cpu().numpy()
    wp_h = wp.cpu().numpy().copy()

    def host_advance():
        live = idx_h[idx_h >= 0]
        p = wp_h[live]
        wp_h[live] = np.where(p == w.L - 1, 0, p + 1)

    def launch_bytes_now():
        live = idx_h[idx_h >= 0]
        p = wp_h[live]
        return launch_bytes(w, p, p == w.L - 1, 2, int((idx_h < 0).sum()))

    adv_ws = Bd.decode_advance_workspace(dev)

    def step(i):
        Bd.gdn_replayssm_decode_advance(desc, cache, wp, None, steps_in[i % POOL], adv_ws, recon, None, None, stream)

    # Untimed legs first (the packed decode beside it and the end-to-end run
    # through host buffers); the W warm-up steps then run right before the
    # timed region (below), so that it starts on a GPU that has not gone idle.
    K = args.steps
    if not args.kernel_only:
        # in-repo packed decode on the workload's shapes (baseline: reads and writes
        # the state; four disjoint slot sets in turn, so no launch hits L2)
        pk = measure_packed(w, max(64, K // 8), dev)
        packed_s = pk["ms_per_launch"] / 1e3
        pbytes = pk["hbm_gbs_algorithmic"] * 1e9 * packed_s
        torch.cuda.empty_cache()

        # end to end through the public API with host buffers: every step copies
        # its inputs from pinned host memory to the device, runs the decode +
        # advance, and copies its output back to pinned host memory.  As a serving
        # loop would, the copies run on their own streams with two device buffer
        # sets, so step i + 1's inputs and step i - 1's output move while step i
        # computes; events order every reuse of a buffer.
        hq = [b.mixed_qkv.cpu().pin_memory() for b in batches]
        hg = [b.g.cpu().pin_memory() for b in batches]
        hb = [b.beta.cpu().pin_memory() for b in batches]
        hi = idx.cpu().pin_memory()
        NBUF = 2
        houts = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(NBUF)]
        dbuf = [(torch.empty_like(batches[0].mixed_qkv), torch.empty_like(batches[0].g),
                 torch.empty_like(batches[0].beta), torch.empty_like(idx), torch.empty_like(out)) for _ in range(NBUF)]
        h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        in_ready = [torch.cuda.Event() for _ in range(NBUF)]  # step's inputs on the device
        used = [torch.cuda.Event() for _ in range(NBUF)]      # step's decode done with its buffers
        out_back = [torch.cuda.Event() for _ in range(NBUF)]  # step's output in host memory
        e2e_steps = max(64, K // 8)
        h2d = hq[0].numel() * hq[0].element_size() + hg[0].numel() * 4 + hb[0].numel() * 4 + hi.numel() * 4
        d2h = houts[0].numel() * houts[0].element_size()

        def e2e_run(n):
            for i in range(n):
                k, j = i % NBUF, i % POOL
                dq, dg, db, di, do = dbuf[k]
                if i >= NBUF:
                    h2d_s.wait_event(used[k])  # the decode of step i - 2 has read these inputs
                with torch.cuda.stream(h2d_s):
                    dq.copy_(hq[j], non_blocking=True)
                    dg.copy_(hg[j], non_blocking=True)
                    db.copy_(hb[j], non_blocking=True)
                    di.copy_(hi, non_blocking=True)
                in_ready[k].record(h2d_s)
                stream.wait_event(in_ready[k])
                if i >= NBUF:
                    stream.wait_event(out_back[k])  # step i - 2's output has left this buffer
                Bd.gdn_replayssm_decode_advance(desc, cache, wp, None, Bd.Step(dq, dg, db, di, do), adv_ws, recon,
                                                None, None, stream)
                used[k].record(stream)
                d2h_s.wait_event(used[k])
                with torch.cuda.stream(d2h_s):
                    houts[k].copy_(do, non_blocking=True)
                out_back[k].record(d2h_s)
            torch.cuda.synchronize()

        e2e_run(8)  # warm the streams and events
        t0 = time.perf_counter()
        e2e_run(e2e_steps)
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        for _ in range(8 + e2e_steps):  # the e2e steps advanced the cursors too
            host_advance()

    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The clock sampler starts before the warm-up: a GPU left idle for a few
    # hundred milliseconds (as while the sampler starts) pays over 100 us more
    # on its next launch, which would otherwise land in the timed region.
    with ClockSampler(local) as clocks:
        # the cursors follow the advance rule, so every timed launch's bytes
        # are known up front; the host does this bookkeeping before the warm-up
        # launches, which then run right before the timed region (no idle gap)
        for i in range(args.warmup):
            host_advance()
        total_bytes = 0.0
        for i in range(K):
            total_bytes += launch_bytes_now()
            host_advance()
        for i in range(args.warmup):
            step(i)
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        # one kernel per step and nothing else between launches, so the
        # kernel's average launch duration is the elapsed time over K (events
        # between launches would also cut the overlap of one launch's set-up
        # with the previous launch's tail)
        start.record(stream)
        for i in range(K):
            step(i)
        stop.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    elapsed_ms = start.elapsed_time(stop)
    mean_kern_s = elapsed_ms / K / 1e3  # this rank's average launch duration
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    # the device cursors must have followed the host mirror exactly
    assert np.array_equal(wp.cpu().numpy(), wp_h), "device cursors diverged from the advance rule"

    head_steps = w.B * w.HV * K
    value = job_throughput(head_steps, ws, elapsed_ms / 1e3)
    bytes_per_launch = total_bytes / K
    peak, peak_src = measured_hbm_peak()
    achieved = bytes_per_launch / mean_kern_s / 1e9
    traffic = profiled_traffic() if (args.workload == "headline" and recon == Bd.RECON_TENSOR) else None
    if args.kernel_only:
        if rank == 0:
            print(json.dumps({"workload": w.name, "recon": args.recon, "steps": K,
                              "kernel_ms": mean_kern_s * 1e3, "ms_per_step": elapsed_ms / K,
                              "head_steps_per_s": value, "algorithmic_bytes_per_launch": bytes_per_launch,
                              "hbm_gbs_algorithmic": achieved, "frac": achieved / peak}))
        if ws > 1:
            dist.destroy_process_group()
        return 0

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return 0
    cpu = cpu_baseline_report(w, seconds=args.ref_seconds, rows=args.ref_rows) if ws == 1 else None
    clk = clocks.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "global_batch": ws * w.B, "num_slots": w.N, "HV": w.HV, "HK": w.HK,
                   "K": w.K, "V": w.V, "L": w.L, "ring_dtype": "f16", "qkv_dtype": "bf16", "out_dtype": "bf16",
                   "tensor_core_operands": "f16 (fp32 accumulate)", "cursors": "staggered uniform [0,L)",
                   "l2": "inputs larger than L2: 512 MiB of checkpoint read per step, no flush",
                   "parallelism": f"replicas x{ws}"},
        "tokens_per_s_per_layer": ws * w.B * K / (elapsed_ms / 1e3),
        "hbm_gbs_algorithmic": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "tcp_decode_kernel (gdn_replayssm_decode_advance: persistent tcgen05 replay, TMA stream, cursor advance)",
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s", "frac_of_8tbs": achieved / 8000.0,
                     "algorithmic_bytes_per_launch": bytes_per_launch, "kernel_ms": mean_kern_s * 1e3},
        "packed_baseline": {"kernel": "gdn_packed_decode", "ms": packed_s * 1e3,
                            "head_steps_per_s": w.B * w.HV / packed_s,
                            "hbm_gbs_algorithmic": pbytes / packed_s / 1e9,
                            "frac": pbytes / packed_s / 1e9 / peak,
                            "replay_speedup": packed_s / mean_kern_s},
        "cpu_baseline": cpu,
        "e2e": {"value": w.B * w.HV / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3, "steps": e2e_steps,
                "copies": "pinned host buffers; H2D and D2H on their own streams, two device buffer sets"},
        "gpu_launches": K,
        "clocks": clk,
    }
    print(json.dumps(line))
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=32)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="headline")
    ap.add_argument("--recon", choices=["tensor", "ffma", "output"], default="tensor")
    ap.add_argument("--kernel-only", action="store_true")
    ap.add_argument("--packed", action="store_true",
                    help="time only the packed decode baseline on the workload (kernel-only, one JSON line)")
    ap.add_argument("--sweep", action="store_true",
                    help="batch x ring length x ring dtype sweep of one layer (one JSON line per point)")
    ap.add_argument("--sweep-batches", default="1,8,64,128,256,512")
    ap.add_argument("--sweep-lens", default="1,4,8,16,32")
    ap.add_argument("--sweep-rings", default="f16,f32")
    ap.add_argument("--sweep-layers", type=int, default=1,
                    help="layer buffers rotated per step (>= 4 keeps a layer's working set out of L2)")
    ap.add_argument("--persistent-kernel", action="store_true",
                    help="sweep: run every point on the persistent tensor-core kernel (no small-batch kernel)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="multi-layer modes: launch every layer without STEP_OVERLAP_PREVIOUS")
    ap.add_argument("--spec", action="store_true",
                    help="speculative verify window sweep (one JSON line per batch x window)")
    ap.add_argument("--graph", action="store_true",
                    help="CUDA-graph replay of 64 decode + advance steps against one-by-one launches")
    ap.add_argument("--graph-batches", default="1,8,64,256")
    ap.add_argument("--graph-layers", type=int, default=1,
                    help="with --graph: a stack of this many layers per step (overlap flag on all but the first)")
    ap.add_argument("--lossless", action="store_true",
                    help="lossless verify + exact-order commit sweep (one JSON line per batch x window)")
    ap.add_argument("--spec-batches", default="64,256")
    ap.add_argument("--spec-windows", default="2,4,8")
    ap.add_argument("--spec-accept", type=float, default=0.7,
                    help="probability that each draft token is accepted (until the first rejection)")
    ap.add_argument("--ref-seconds", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=16)
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds of oracle work the reference arm aims for")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.packed:
        return run_packed(args)
    if args.sweep:
        return run_sweep(args)
    if args.spec:
        return run_spec(args)
    if args.lossless:
        return run_lossless(args)
    if args.graph:
        return run_graph(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
