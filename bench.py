"""Benchmark of the Mamba2 selective-state-update decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extras] [--no-cpu-baseline]

One step is one pass of the decode hot path over one batch of seeded synthetic
inputs (resident in HBM): for the default workload (Mamba2-2.7B-shaped
decode: batch 256, 80 heads, headdim 64, dstate 128, fp32 state pool of 512
slots, 5% pad) that is one ssu_update launch; for the MTP workload one
ssu_update_varlen launch plus the ReplaySSM tracker update and commit.
With extras on, the line also carries the packed SSD prefill
(`ssd_prefill`: 16 sequences of 256..2048 tokens, Mamba2-2.7B layer shape,
one ssd_combined_fwd_varlen call per step); `--workload ssd-prefill-2.7b`
measures that call alone.

Prints ONE JSON line.  `value` is decode tokens/s (non-pad tokens of all ranks
/ max-over-ranks time); the line also carries achieved HBM GB/s of the SSU
kernel against the measured HBM peak (`roofline`), the end-to-end rate through
the public API with host buffers (`e2e`), the CPU oracle's rate (`cpu_baseline`)
and, with extras on, the other serving workloads (`workloads`).

Under torchrun (N > 1) every rank runs its own shard of sequences (its own
seed) on its own GPU: weak scaling, no data-path collective; ranks meet only
at the barriers around the timed region and the max-reduction of its time.
`--impl reference` times the CPU oracle (the reference arm) on
the same workload, on rank 0 only.
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
L2_BYTES = 129 * 2**20


# ---------------------------------------------------------------------------
# workload bookkeeping
# ---------------------------------------------------------------------------

def _workload(name, device, seed):
    from mamba2_ssm_decode_gb300 import workloads as W
    if name in W.WORKLOADS:
        return W.WORKLOADS[name](seed=seed, device=device)
    m = re.fullmatch(r"sweep-(single|mtp)-(float32|bfloat16)-b(\d+)(-nowrite)?(-sr)?", name)
    if m:
        return W.sweep_case(int(m.group(3)), getattr(torch, m.group(2)), m.group(1),
                            disable_state_update=bool(m.group(4)), seed=seed, device=device,
                            stochastic_rounding=bool(m.group(5)))
    raise SystemExit(f"unknown workload {name}")


def _esize(t):
    return 0 if t is None else t.element_size()


def replay_accounting(case):
    """(tokens, algorithmic bytes, 0) of a ReplaySSM checkpointing call.

    Per processed sequence (valid slot, trackers in range) and head: the
    checkpoint read, a checkpoint write when k + L > W, the k cached tokens' x
    and dt read from the ring and the L new ones written to it; per group the
    cached / new B; per row x, z, dt, B, C read and y written; the trackers (8
    bytes read, 8 more written with the update) and the slot vector.  With the
    tracker update in the call, k cycles through 1..W from call to call, so the
    count is the mean over one cycle of W calls (exact for a multiple of W
    timed calls)."""
    slots, H, P, N, G = case.dims
    sb = case.state.element_size()
    io = case.x.element_size()
    R, W = case.ring_buffer_len, case.logical_window
    sbi = case.state_batch_indices.cpu().long() if case.state_batch_indices is not None else None
    if case.cu_seqlens is not None:
        cu = case.cu_seqlens.cpu().long().tolist()
    else:
        cu = list(range(case.nseqs + 1))
    pna = case.prev_num_accepted.cpu().long().tolist()
    rs = case.ring_start.cpu().long().tolist()
    limit = min(slots, len(pna), len(rs))
    seqs = []
    for s in range(case.nseqs):
        L = cu[s + 1] - cu[s]
        slot = int(sbi[s]) if sbi is not None else s
        if L <= 0 or slot == case.pad_slot_id or not 0 <= slot < limit:
            continue
        k, st = pna[slot], rs[slot]
        if k < 0 or k + L > R or not 0 <= st < R:
            continue
        seqs.append((L, k))
    phases = W if case.update_trackers and W >= 1 else 1
    total = 0
    for _ in range(phases):
        for L, k in seqs:
            total += H * P * N * sb * (1 + (k + L > W))
            total += (k + L) * (H * P * io + H * 4 + G * N * io)
            total += 8 + (8 if case.update_trackers else 0)
        if phases > 1:
            seqs = [(L, 1 if k + 1 > W else k + 1) for L, k in seqs]
    per_row = H * P * io * (3 if case.z is not None else 2) + H * 4 + 2 * G * N * io
    meta = sum(t.numel() * t.element_size() for t in (case.state_batch_indices, case.cu_seqlens)
               if t is not None)
    tokens = sum(L for L, _ in seqs)
    return tokens, total // phases + case.rows * per_row + meta, 0


def accounting(case):
    """(non-pad tokens, algorithmic bytes of the SSU launch, tracker bytes).

    Algorithmic bytes per launch: every sequence with a valid read slot reads
    its H x P x N state block once and writes it once per valid destination
    write; every packed row reads x, z, dt, B, C and writes y; plus the index
    tables and metadata (read once).  Pad sequences move no state."""
    if case.kind == "replay":
        return replay_accounting(case)
    slots, H, P, N, G = case.dims
    sb = case.state.element_size()
    block = H * P * N * sb
    pad = case.pad_slot_id
    rows = case.rows
    sbi = case.state_batch_indices.cpu() if case.state_batch_indices is not None else None
    dsbi = (case.dst_state_batch_indices.cpu()
            if case.dst_state_batch_indices is not None else None)

    def ok(v):
        return v != pad and 0 <= v < slots

    reads = writes = tokens = 0
    if case.kind == "single":
        for b in range(case.nseqs):
            src = int(sbi[b]) if sbi is not None else b
            if not ok(src):
                continue
            reads += 1
            tokens += 1
            dst = int(dsbi[b]) if dsbi is not None else src
            if not case.disable_state_update and ok(dst):
                writes += 1
    else:
        if case.cu_seqlens is not None:
            cu = case.cu_seqlens.cpu().long().tolist()
        else:
            cu = [s * case.dense_steps for s in range(case.nseqs + 1)]
        na = (case.num_accepted_tokens.cpu().long().tolist()
              if case.num_accepted_tokens is not None else None)
        for s in range(case.nseqs):
            L = cu[s + 1] - cu[s]
            if L <= 0:
                continue
            if sbi is not None:
                col = (na[s] - 1) if na is not None else 0
                row = sbi[s] if sbi.dim() == 2 else sbi[s:]
                src = int(row[col]) if 0 <= col < row.numel() else pad
            else:
                src = s
            if not ok(src):
                continue
            reads += 1
            tokens += L
            if case.disable_state_update:
                continue
            tab = dsbi if dsbi is not None else sbi
            for t in range(L):
                if tab is None:
                    dst = s
                else:
                    row = tab[s] if tab.dim() == 2 else tab[s:]
                    dst = int(row[t]) if t < row.numel() else pad
                writes += ok(dst)
    io = case.x.element_size()
    per_row = H * P * io * (3 if case.z is not None else 2)           # x, (z), out
    per_row += (case.dt[0].numel()) * 4                               # dt
    per_row += 2 * G * N * io                                         # B, C
    meta = sum(t.numel() * t.element_size() for t in (sbi, dsbi, case.cu_seqlens,
                                                        case.num_accepted_tokens)
               if t is not None)
    ssu_bytes = (reads + writes) * block + rows * per_row + meta
    trk = 0
    if case.ring_start is not None:
        # update: slot + 2 loads + 2 stores; commit: slot, 3 loads, 3 stores, count, 2 starts
        trk = case.nseqs * (_esize(sbi) + 16) + case.nseqs * (_esize(sbi) + 24 + 12)
    return tokens, ssu_bytes, trk


# ---------------------------------------------------------------------------
# the step
# ---------------------------------------------------------------------------

class Step:
    """One pass of the hot path over a resident batch (all device tensors)."""

    def __init__(self, case, algorithm="auto"):
        import mamba2_ssm_decode_gb300 as ssu
        self.ssu = ssu
        self.case = case
        self.algorithm = algorithm
        self.out = torch.empty_like(case.x)
        self.replay = case.kind == "replay"
        # the replay call runs its tracker update itself (counters in scratch)
        self.launches = 1 + (2 if case.ring_start is not None and not self.replay else 0)
        self.scratch = (torch.zeros(max(1, case.nseqs), dtype=torch.int32, device=case.x.device)
                        if self.replay else None)
        self.seed = (torch.tensor([case.sr_seed], dtype=torch.int64, device=case.x.device)
                     if case.sr_seed is not None else None)
        if case.kind == "varlen" and case.cu_seqlens is None:
            S, T = case.nseqs, case.dense_steps

            def v4(t):   # the dense [batch, steps, ...] view; a per-head dt gets a unit dim
                if t is None:
                    return None
                if t.dim() == 2:
                    return t.view(S, T, t.shape[1], 1)
                return t.view(S, T, *t.shape[1:])

            self.v4 = v4
        else:
            self.v4 = None

    # the tensors a caller supplies anew every step (everything but the state
    # pool, the trackers and the per-head parameters)
    STEP_INPUTS = ("x", "z", "dt", "B", "C", "state_batch_indices", "dst_state_batch_indices",
                   "cu_seqlens", "num_accepted_tokens")

    def ssu_launch(self, out=None, **over):
        c = self.case
        t = {n: over[n] if over.get(n) is not None else getattr(c, n) for n in self.STEP_INPUTS}
        out = self.out if out is None else out
        if self.replay:
            self.ssu.ssu_replay_update(
                c.state, t["x"], t["dt"], c.A, t["B"], t["C"], c.x_cache, c.B_cache, c.dt_cache,
                c.ring_start, c.prev_num_accepted, c.logical_window, D=c.D, z=t["z"],
                dt_bias=c.dt_bias, dt_softplus=c.dt_softplus, cu_seqlens=t["cu_seqlens"],
                state_batch_indices=t["state_batch_indices"], pad_slot_id=c.pad_slot_id, out=out,
                update_trackers=c.update_trackers, scratch=self.scratch, rand_seed=self.seed)
            return
        kw = dict(D=c.D, z=t["z"], dt_bias=c.dt_bias, dt_softplus=c.dt_softplus,
                  pad_slot_id=c.pad_slot_id, disable_state_update=c.disable_state_update,
                  out=out, algorithm=self.algorithm, rand_seed=self.seed)
        if c.kind == "single":
            self.ssu.ssu_update(c.state, t["x"], t["dt"], c.A, t["B"], t["C"],
                                state_batch_indices=t["state_batch_indices"],
                                dst_state_batch_indices=t["dst_state_batch_indices"], **kw)
        elif self.v4 is not None:
            v = self.v4
            kw["z"], kw["out"] = v(t["z"]), v(out)
            self.ssu.ssu_update_varlen(c.state, v(t["x"]), v(t["dt"]), c.A, v(t["B"]),
                                       v(t["C"]), num_accepted_tokens=t["num_accepted_tokens"],
                                       state_batch_indices=t["state_batch_indices"],
                                       dst_state_batch_indices=t["dst_state_batch_indices"],
                                       **kw)
        else:
            self.ssu.ssu_update_varlen(c.state, t["x"], t["dt"], c.A, t["B"], t["C"],
                                       cu_seqlens=t["cu_seqlens"],
                                       num_accepted_tokens=t["num_accepted_tokens"],
                                       state_batch_indices=t["state_batch_indices"],
                                       dst_state_batch_indices=t["dst_state_batch_indices"],
                                       nseqs=c.nseqs, **kw)

    def trackers(self, **over):
        c = self.case
        if c.ring_start is None or self.replay:
            return
        t = {n: over[n] if over.get(n) is not None else getattr(c, n) for n in self.STEP_INPUTS}
        sbi = t["state_batch_indices"]
        tr = (c.ring_start, c.prev_num_accepted, c.prev_query_len)
        self.ssu.ssu_ring_update(*tr, sbi, c.logical_window, c.ring_buffer_len,
                                 pad_slot_id=c.pad_slot_id)
        self.ssu.ssu_ring_commit(*tr, sbi, t["num_accepted_tokens"], t["cu_seqlens"],
                                 c.logical_window, c.ring_buffer_len, pad_slot_id=c.pad_slot_id)

    def __call__(self):
        self.ssu_launch()
        self.trackers()


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

_REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40),
            ("sw_thermal_slowdown", 0x20), ("sw_power_cap", 0x4))


class _Nvml:
    """SM clock and clock-event reasons of one GPU read through NVML (ctypes on
    the driver's libnvidia-ml; read-only queries)."""

    def __init__(self, uuid):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        n = ctypes.c_uint(0)
        if lib.nvmlDeviceGetCount_v2(ctypes.byref(n)) != 0:
            raise OSError("nvmlDeviceGetCount failed")
        self.h = None
        buf = ctypes.create_string_buffer(96)
        for i in range(n.value):
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(h)) != 0:
                continue
            if lib.nvmlDeviceGetUUID(h, buf, 96) != 0:
                continue
            if buf.value.decode().lower().replace("gpu-", "") == uuid:
                self.h = h
                break
        if self.h is None:
            raise OSError("GPU not found by UUID")
        self.lib = lib
        try:
            self._reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))   # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)

    def read(self):
        ct = self.ct
        sm = ct.c_uint(0)
        r = ct.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(sm)) != 0:
            return None
        self._reasons(self.h, ct.byref(r))
        return float(sm.value), self.max_mhz, frozenset(n for n, b in _REASONS if r.value & b)


class ClockSampler:
    """SM clock and throttle reasons of this GPU, sampled every millisecond
    through NVML (so that even a few-millisecond timed region holds samples),
    or every 100 ms from nvidia-smi where NVML cannot be loaded."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        props = torch.cuda.get_device_properties(device)
        self.uuid = str(getattr(props, "uuid", "")).lower().replace("gpu-", "")
        self.samples = []      # (time, sm MHz, max MHz, reasons)
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.marks = {}
        self.source = None

    def start(self):
        try:
            nv = _Nvml(self.uuid)
            self.source = "nvml 1 ms"
            self.thread = threading.Thread(target=self._poll, args=(nv,), daemon=True)
            self.thread.start()
            return
        except (OSError, AttributeError):
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi 100 ms"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _poll(self, nv):
        while not self.stop_flag.is_set():
            v = nv.read()
            if v is not None:
                self.samples.append((time.perf_counter(), *v))
            time.sleep(0.001)

    def _read(self):
        names = [n for n, _ in _REASONS]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            uuid = parts[0].lower().replace("gpu-", "")
            if self.uuid and uuid != self.uuid:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = frozenset(n for n, v in zip(names, parts[3:7]) if v == "Active")
            self.samples.append((time.perf_counter(), sm, mx, reasons))

    def mark(self, name):
        self.marks[name] = time.perf_counter()

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        t0, t1 = self.marks.get("timed_start"), self.marks.get("timed_end")
        inside = [x for x in self.samples if t0 is not None and t0 <= x[0] <= t1]
        pool = inside or self.samples
        sm = [x[1] for x in pool]
        mx = [x[2] for x in pool]
        reasons = sorted({r for x in pool for r in x[3]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(pool), "samples_in_timed_region": len(inside),
                "source": self.source}


# ---------------------------------------------------------------------------
# measurement
# ---------------------------------------------------------------------------

def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


DATA = "synthetic (seeded random inputs of Mamba2 serving shapes)"


def _code_only(src):
    """C / CUDA source text without comments and with whitespace collapsed."""
    text = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return " ".join(text.split())


def kernel_source_hash(workload=None):
    """Hash of the CUDA sources a workload's kernels are built from: the SSD
    prefill's (ssd* and the three SSU headers it includes) or the SSU decode's
    (every other source), so that a change to one leaves the other's ncu
    traffic record valid.  Only the code is hashed: an edit to comments or
    whitespace leaves the records valid."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mamba2_ssm_decode_gb300", "csrc")
    ssd = workload == SSD_WORKLOAD
    for f in sorted(os.listdir(csrc)):
        if f.startswith("ssd") != ssd and not (ssd and f in ("ssu_headrun.cuh", "ssu_kernel.cuh",
                                                          "ssu_bulk.cuh")):
            continue
        with open(os.path.join(csrc, f), encoding="utf-8", errors="replace") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch (per call for the SSD prefill) from the committed
    ncu summary of this workload, valid only while the kernel sources hash to
    the value recorded with it."""
    prefix = "" if workload == SSD_WORKLOAD else "ssu_"
    path = os.path.join(ROOT, "profiles", f"{prefix}{workload}_dram.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"^kernel_source_hash:\s*(\w+)", text, re.M)
    m_val = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    if not (m_hash and m_val) or m_hash.group(1) != kernel_source_hash(workload):
        return None
    return float(m_val.group(1))


def time_steps(step, steps, stream, per_launch=True):
    """K steps on `stream`: total ms from CUDA events, and the mean duration of
    the SSU launch itself (events around it, on the same stream)."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if per_launch else []
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if per_launch else []
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for k in range(steps):
            if per_launch:
                starts[k].record(stream)
            step.ssu_launch()
            if per_launch:
                ends[k].record(stream)
            step.trackers()
        t_end.record(stream)
    t_end.synchronize()
    total = t_start.elapsed_time(t_end)
    launch = (sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps) if per_launch else None
    return total, launch


def e2e(step, steps, warmup, stream):
    """The same step through the public API with host buffers: every step copies
    every per-step input (x, z, dt, B, C, the slot tables, cu_seqlens and the
    acceptance counts) from pinned host memory, runs the call (and the tracker
    update / commit where the workload has them) and copies y back, then waits
    for it."""
    c = step.case
    host = {n: getattr(c, n).cpu().pin_memory() for n in step.STEP_INPUTS
            if getattr(c, n) is not None}
    dev = {n: torch.empty_like(getattr(c, n)) for n in host}
    y_host = torch.empty(c.x.shape, dtype=c.x.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = y_host.numel() * y_host.element_size()

    def one():
        with torch.cuda.stream(stream):
            for n, t in host.items():
                dev[n].copy_(t, non_blocking=True)
            step.ssu_launch(**dev)
            step.trackers(**dev)
            y_host.copy_(step.out, non_blocking=True)
        stream.synchronize()

    for _ in range(warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    return (time.perf_counter() - t0) * 1e3 / steps, h2d, d2h


STATE_TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2, torch.float16: 2e-2}
HALF_ULP = {torch.bfloat16: 2.0**-8, torch.float16: 2.0**-11, torch.float32: 0.0}


def _excess(got, ref, tol, half_ulp=0.0):
    """max |got - ref| / (tol + (tol + half_ulp) |ref|) (1.0 = at the tolerance)."""
    got, ref = got.double(), ref.double()
    if got.numel() == 0:
        return 0.0
    return float(((got - ref).abs() / (tol + (tol + half_ulp) * ref.abs())).max())


def _oracle_call(sub):
    import oracle
    kw = dict(D=sub.D, z=sub.z, dt_bias=sub.dt_bias, dt_softplus=sub.dt_softplus,
              pad_slot_id=sub.pad_slot_id, disable_state_update=sub.disable_state_update,
              state_batch_indices=sub.state_batch_indices,
              dst_state_batch_indices=sub.dst_state_batch_indices)
    if sub.kind == "single":
        return oracle.ssu_update(sub.state, sub.x, sub.dt, sub.A, sub.B, sub.C, **kw)
    return oracle.ssu_update_varlen(sub.state, sub.x, sub.dt, sub.A, sub.B, sub.C,
                                    cu_seqlens=sub.cu_seqlens, nseqs=sub.nseqs,
                                    dense_steps=sub.dense_steps,
                                    num_accepted_tokens=sub.num_accepted_tokens, **kw)


def _time_oracle(shards, threads, min_seconds, passes=None):
    """Oracle time per pass over `shards` (CPU sub-cases, disjoint slots) on
    `threads` host threads (the oracle is C called through ctypes, which runs
    with the interpreter lock released), repeated until `min_seconds` (or
    exactly `passes` times).  Each shard runs on its own copy of its pool, made
    before the clock starts; later passes continue from the state the previous
    pass left (the time does not depend on the values).  Returns (seconds per
    pass, passes, first pass's (y, pool) per shard)."""
    import concurrent.futures as cf
    import dataclasses
    work = [dataclasses.replace(sub, state=sub.state.clone()) for sub in shards]
    first = None
    reps, t0 = 0, time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while True:
            ys = list(ex.map(_oracle_call, work))
            if first is None:   # keep the first pass's results (not timed)
                tc = time.perf_counter()
                first = [(y, w.state.clone()) for y, w in zip(ys, work)]
                t0 += time.perf_counter() - tc
            reps += 1
            if passes is not None:
                if reps >= passes:
                    break
            elif time.perf_counter() - t0 >= min_seconds:
                break
    return (time.perf_counter() - t0) / reps, reps, first


def cpu_leg(step, max_seqs, min_seconds):
    """The CPU oracle (plain fp64 C) beside the GPU, on a bounded sample of the
    workload: the first `max_seqs` sequences.  Their slots are copied to the host,
    the GPU runs one more step of the whole batch, and the oracle runs the sample
    once on one host thread and once on all host cores (the sample split into
    contiguous shards, one per thread); both are timed.  The GPU step's outputs
    and written slots of the sample are compared with the oracle's at the
    stated tolerances."""
    from mamba2_ssm_decode_gb300 import workloads as W
    import oracle
    oracle.build()
    case = step.case
    seqs = list(range(min(max_seqs, case.nseqs)))
    sub, rows, remap = W.subset_case(case, seqs)
    tokens, _, _ = accounting(sub)
    # the GPU step whose sample is checked
    torch.cuda.synchronize()
    step.ssu_launch()
    torch.cuda.synchronize()
    y_gpu = step.out[torch.tensor(rows, dtype=torch.long, device=step.out.device)].cpu()
    old = list(remap.keys())
    pool_gpu = (case.state[torch.tensor(old, dtype=torch.long, device=case.state.device)].cpu()
                if old else None)
    # one thread over the whole sample, then all cores over contiguous shards
    t1, reps1, res1 = _time_oracle([sub], 1, min_seconds / 2)
    ncores = max(1, min(os.cpu_count() or 1, len(seqs)))
    bounds = [len(seqs) * k // ncores for k in range(ncores + 1)]
    shards = [W.subset_case(sub, list(range(bounds[k], bounds[k + 1])))[0]
              for k in range(ncores) if bounds[k + 1] > bounds[k]]
    tn, repsn, _ = _time_oracle(shards, len(shards), min_seconds / 2)
    # parity of the GPU step on the sample
    y_ref, st_ref = res1[0]
    sdt = case.state.dtype
    tol = STATE_TOL[sdt]
    covered = ~torch.isnan(y_ref.reshape(y_ref.shape[0], -1)).any(dim=1)
    y_err = _excess(y_gpu[covered].float(), y_ref[covered], tol, HALF_ULP[y_gpu.dtype])
    st_err = _excess(pool_gpu.float(), st_ref.float(), tol) if pool_gpu is not None else 0.0
    return {"value": tokens / tn, "unit": "tokens/s", "cores": len(shards), "kind": "oracle",
            "single_core_value": tokens / t1,
            "sample": f"the first {len(seqs)} of the {case.nseqs} sequences of {case.name} "
                      f"({tokens} tokens): {reps1} pass(es) on one host core, {repsn} on "
                      f"{len(shards)} threads (contiguous shards), fp64 C oracle",
            "parity": {"sequences": len(seqs), "rows": len(rows),
                       "y_err_over_tol": y_err, "state_err_over_tol": st_err,
                       "ok": bool(y_err <= 1.0 and st_err <= 1.0)}}


def measure(name, device, seed, steps, warmup, stream, algorithm="auto"):
    case = _workload(name, device, seed)
    tokens, ssu_bytes, trk_bytes = accounting(case)
    step = Step(case, algorithm)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step()
    torch.cuda.synchronize()
    total, launch = time_steps(step, steps, stream)
    ms = total / steps
    return case, step, {"tokens": tokens, "ssu_bytes": ssu_bytes, "ms_per_step": ms,
                        "launch_ms": launch, "tokens_per_s": tokens / (ms * 1e-3),
                        "gbs": ssu_bytes / (launch * 1e-3) / 1e9}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

DEFAULT_WORKLOAD = "mamba2-2.7b-decode"
EXTRAS = ["hybrid-grouped-decode", "mtp-varlen", "replay-decode", "replay-mtp",
          "mamba2-2.7b-decode-perchannel", "mtp-varlen-dtperdim",
          "sweep-single-float32-b1024", "sweep-single-bfloat16-b1024",
          "sweep-mtp-float32-b1024", "sweep-mtp-bfloat16-b1024",
          "sweep-single-bfloat16-b4096", "sweep-mtp-bfloat16-b4096",
          "sweep-single-float32-b1024-nowrite", "sweep-single-bfloat16-b1024-nowrite",
          "sweep-mtp-float32-b1024-nowrite", "sweep-mtp-bfloat16-b1024-nowrite",
          "sweep-single-bfloat16-b1024-sr", "sweep-mtp-bfloat16-b1024-sr"]
# the largest single-GPU points, measured like the headline (every timed step,
# end to end, oracle baseline and parity sample)
LARGE = ["sweep-single-float32-b4096", "sweep-mtp-float32-b4096"]


# ---------------------------------------------------------------------------
# packed SSD prefill
# ---------------------------------------------------------------------------

SSD_WORKLOAD = "ssd-prefill-2.7b"
SSD_TOL = 2e-2   # |gpu - oracle| <= SSD_TOL (|oracle| + rms of the oracle's row)


def ssd_accounting(c, state_dtype=None):
    """(tokens, algorithmic bytes, algorithmic flops) of one packed SSD call.

    Bytes: x, z, B, C, dt read and y written once per token, the initial
    states read and the final states written once per sequence, plus the
    chunk metadata; the chunk states the call keeps in its workspace are not
    algorithmic.  Flops (2 per multiply-add) of the contractions: the chunk
    states (P x N per token and head), C . h_enter (the same), the
    intra-chunk products (P per pair s <= t and head) and C . B^T (N per pair
    and group)."""
    T, H, P = c.x.shape
    G, N = c.B.shape[1], c.B.shape[2]
    io = c.x.element_size()
    batch = c.cu_seqlens.numel() - 1
    cuc = c.cu_chunk_seqlens.cpu().long().tolist()
    lens = [cuc[i + 1] - cuc[i] for i in range(len(cuc) - 1)]
    tokens = cuc[-1] - cuc[0]
    sdt = state_dtype or (c.initial_states.dtype if c.initial_states is not None else c.C.dtype)
    hpn = H * P * N
    nbytes = tokens * (H * P * io * (3 if c.z is not None else 2) + H * 4 + 2 * G * N * io)
    if c.initial_states is not None:
        nbytes += batch * hpn * c.initial_states.element_size()
    nbytes += batch * hpn * torch.empty((), dtype=sdt).element_size()
    nbytes += sum(t.numel() * t.element_size() for t in (c.cu_seqlens, c.cu_chunk_seqlens,
                                                         c.seq_idx, c.last_chunk_indices))
    flops = 4 * tokens * hpn + sum((H * P + G * N) * L * (L + 1) for L in lens)
    return tokens, nbytes, flops


class SSDStep:
    """One packed SSD prefill call through the public API, with out, states
    and workspace preallocated (the call itself allocates nothing)."""

    INPUTS = ("x", "dt", "B", "C", "z", "initial_states", "cu_seqlens", "cu_chunk_seqlens",
              "last_chunk_indices", "seq_idx")

    def __init__(self, case):
        import mamba2_ssm_decode_gb300 as ssu
        self.ssu, self.case = ssu, case
        c = case
        T, H, P = c.x.shape
        G, N = c.B.shape[1], c.B.shape[2]
        nch = c.cu_chunk_seqlens.numel() - 1
        batch = c.cu_seqlens.numel() - 1
        self.out = torch.empty_like(c.x)
        sdt = c.initial_states.dtype if c.initial_states is not None else c.C.dtype
        self.states = torch.empty((batch, H, P, N), dtype=sdt, device=c.x.device)
        self.workspace = torch.empty(ssu.ssd_workspace_bytes(nch, H, G, P, N, c.chunk_size),
                                     dtype=torch.uint8, device=c.x.device)
        self.launches = 3   # chunk states, state passing, scan

    def __call__(self, **over):
        c = self.case
        v = {n: over.get(n, getattr(c, n)) for n in self.INPUTS}
        return self.ssu.ssd_combined_fwd_varlen(
            v["x"], v["dt"], c.A, v["B"], v["C"], c.chunk_size, v["cu_seqlens"],
            v["cu_chunk_seqlens"], v["last_chunk_indices"], v["seq_idx"], out=self.out,
            D=c.D, z=v["z"], dt_bias=c.dt_bias, dt_softplus=c.dt_softplus, dt_limit=c.dt_limit,
            initial_states=v["initial_states"], states=self.states, workspace=self.workspace)


def _ssd_row_excess(got, ref):
    """max over elements of |got - ref| / (SSD_TOL (|ref| + rms of ref's row)),
    a row being the last axis, floored at 1e-3 of the global rms."""
    import numpy as np
    got = got.detach().cpu().double().numpy()
    if ref.size == 0:
        return 0.0
    if not np.isfinite(got).all():
        return float("inf")
    row = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    row = np.maximum(row, 1e-3 * float(np.sqrt(np.mean(ref * ref))))
    return float((np.abs(got - ref) / (SSD_TOL * (np.abs(ref) + row))).max())


def ssd_cpu_leg(step, nseqs=2):
    """The fp64 SSD oracle on the first `nseqs` sequences (a bounded sample:
    sequences are independent, so their tokens, chunks and states are a slice
    of the batch): its rate on one host core, and the GPU call's y and final
    states of those sequences against it."""
    from mamba2_ssm_decode_gb300 import workloads as W
    from oracle import ssd as ssd_oracle
    c = step.case
    torch.cuda.synchronize()
    step()
    torch.cuda.synchronize()
    cu = c.cu_seqlens.cpu().tolist()
    last = c.last_chunk_indices.cpu().tolist()
    nb = min(nseqs, len(last))
    T, nch = cu[nb], last[nb - 1] + 1
    sub = W.SSDCase(name="sample", x=c.x[:T], dt=c.dt[:T], A=c.A, B=c.B[:T], C=c.C[:T], D=c.D,
                    z=c.z[:T] if c.z is not None else None, dt_bias=c.dt_bias,
                    chunk_size=c.chunk_size, cu_seqlens=c.cu_seqlens[:nb + 1],
                    cu_chunk_seqlens=c.cu_chunk_seqlens[:nch + 1],
                    last_chunk_indices=c.last_chunk_indices[:nb], seq_idx=c.seq_idx[:nch],
                    initial_states=(c.initial_states[:nb] if c.initial_states is not None
                                    else None),
                    dt_softplus=c.dt_softplus, dt_limit=c.dt_limit).to("cpu")
    t0 = time.perf_counter()
    y_ref, s_ref = ssd_oracle.ssd_combined_fwd_varlen(
        sub.x, sub.dt, sub.A, sub.B, sub.C, sub.chunk_size, sub.cu_seqlens, sub.cu_chunk_seqlens,
        sub.last_chunk_indices, sub.seq_idx, D=sub.D, z=sub.z, dt_bias=sub.dt_bias,
        dt_softplus=sub.dt_softplus, dt_limit=sub.dt_limit, initial_states=sub.initial_states)
    secs = time.perf_counter() - t0
    y_err = _ssd_row_excess(step.out[:T], y_ref)
    s_err = _ssd_row_excess(step.states[:nb], s_ref)
    return {"value": T / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"the first {nb} of the {len(last)} sequences of {c.name} ({T} tokens, "
                      f"{nch} chunks): one pass of the fp64 numpy oracle on one host core",
            "parity": {"sequences": nb, "tokens": T, "y_err_over_tol": y_err,
                       "state_err_over_tol": s_err, "tol": SSD_TOL,
                       "ok": bool(y_err <= 1.0 and s_err <= 1.0)}}


def ssd_e2e(step, steps, warmup, stream):
    """The SSD call through the public API with host buffers: every step copies
    the call's inputs (x, z, dt, B, C, initial states, chunk metadata) from
    pinned host memory, runs the call and copies y and the final states back,
    then waits for them."""
    c = step.case
    host = {n: getattr(c, n).cpu().pin_memory() for n in step.INPUTS if getattr(c, n) is not None}
    dev = {n: torch.empty_like(getattr(c, n)) for n in host}
    y_host = torch.empty(c.x.shape, dtype=c.x.dtype).pin_memory()
    s_host = torch.empty(step.states.shape, dtype=step.states.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = y_host.numel() * y_host.element_size() + s_host.numel() * s_host.element_size()

    def one():
        with torch.cuda.stream(stream):
            for n, t in host.items():
                dev[n].copy_(t, non_blocking=True)
            step(**dev)
            y_host.copy_(step.out, non_blocking=True)
            s_host.copy_(step.states, non_blocking=True)
        stream.synchronize()

    for _ in range(warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    return (time.perf_counter() - t0) * 1e3 / steps, h2d, d2h


def ssd_leg(args, device, stream, peak, peak_kind, steps, cpu=True):
    """Every measurement of the packed SSD prefill: the timed calls (CUDA
    events around each call on its stream: the three launches of one call are
    one unit), the byte and flop rooflines of a call, the end-to-end rate and,
    on request, the oracle sample with its parity check."""
    from mamba2_ssm_decode_gb300 import workloads as W
    case = W.ssd_prefill(seed=args.seed, device=device)
    tokens, nbytes, flops = ssd_accounting(case)
    step = SSDStep(case)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    torch.cuda.synchronize()
    clocks = ClockSampler(device)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    clocks.mark("timed_start")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for k in range(steps):
            starts[k].record(stream)
            step()
            ends[k].record(stream)
    ends[-1].synchronize()
    clocks.mark("timed_end")
    time.sleep(0.15)
    clocks.stop()
    total = starts[0].elapsed_time(ends[-1])
    call_ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps
    device_error = step.ssu.ssu_device_error()
    tflops_peak = _tensor_peak()
    achieved = nbytes / (call_ms * 1e-3) / 1e9
    tflops = flops / (call_ms * 1e-3) / 1e12
    T, H, P = case.x.shape
    G, N = case.B.shape[1], case.B.shape[2]
    e2e_ms, h2d, d2h = ssd_e2e(step, max(3, min(steps, 50)), 3, stream)
    out = {
        "metric": "packed SSD prefill tokens/s (1 GPU)",
        "value": tokens * steps / (total * 1e-3), "unit": "tokens/s", "steps": steps,
        "ms_per_step": total / steps, "higher_is_better": True, "dtype": "bf16 io, f32 state",
        "config": {"workload": case.name, "batch": case.cu_seqlens.numel() - 1, "tokens": T,
                   "nchunks": case.cu_chunk_seqlens.numel() - 1, "chunk_size": case.chunk_size,
                   "nheads": H, "headdim": P, "dstate": N, "ngroups": G,
                   "io_dtype": str(case.x.dtype)[6:],
                   "state_dtype": str(step.states.dtype)[6:],
                   "l2": f"no flush: each call reads and writes {nbytes / 1e9:.2f} GB > 129 MB L2"},
        "roofline": {"bound": "hbm" if nbytes / (peak * 1e9) >= flops / (tflops_peak * 1e12)
                     else "tensor",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic(case.name),
                     "algorithmic_bytes_per_call": nbytes, "algorithmic_flops_per_call": flops,
                     "tflops": tflops, "tensor_peak_tflops": tflops_peak,
                     "tensor_frac": tflops / tflops_peak, "call_ms": call_ms,
                     "launches_per_call": step.launches,
                     "peak_source": f"{peak_kind} hbm_gbs; measured bf16_tflops (burst)"},
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": step.launches * steps,
        "device_error": device_error,
        "clocks": clocks.summary(),
    }
    if cpu and not args.no_cpu_baseline:
        out["cpu_baseline"] = ssd_cpu_leg(step)
    del step, case
    torch.cuda.empty_cache()
    return out


def _tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        return 1900.0


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def headline(name, args, world, device, stream, peak, peak_kind, cpu=True):
    """Every measurement of one workload: the timed steps (barrier, max over
    ranks), the SSU launch's roofline, the device error word, the end-to-end
    rate through the public API and, on rank 0, the oracle leg."""
    rank = int(os.environ.get("RANK", "0"))
    seed = args.seed + rank   # each rank: its own shard of sequences
    case = _workload(name, device, seed)
    tokens, ssu_bytes, _ = accounting(case)
    step = Step(case, args.algorithm)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    clocks = ClockSampler(device)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark("timed_start")
    total, launch = time_steps(step, args.steps, stream)
    torch.cuda.synchronize()
    clocks.mark("timed_end")
    barrier(world)
    time.sleep(0.15)
    clocks.stop()
    device_error = step.ssu.ssu_device_error()
    total_max = max_over_ranks(total, world, device)
    launch_max = max_over_ranks(launch, world, device)
    tokens_all = sum_over_ranks(tokens * args.steps, world, device)
    ms = total_max / args.steps
    e2e_ms, h2d, d2h = e2e(step, max(3, min(args.steps, 200)), 3, stream)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_value = sum_over_ranks(tokens, world, device) / (e2e_ms * 1e-3)
    achieved = ssu_bytes / (launch_max * 1e-3) / 1e9
    slots, H, P, N, G = case.dims
    out = {
        "value": tokens_all / (total_max * 1e-3), "ms_per_step": ms,
        "config": {"workload": case.name, "batch": case.nseqs, "nheads": H, "headdim": P,
                   "dstate": N, "ngroups": G, "state_dtype": str(case.state.dtype)[6:],
                   "io_dtype": str(case.x.dtype)[6:], "slots": slots, "non_pad_tokens": tokens,
                   "rows": case.rows, "kind": case.kind,
                   "disable_state_update": case.disable_state_update,
                   "algorithm": args.algorithm,
                   "l2": f"no flush: each step touches {ssu_bytes / 1e9:.2f} GB > 129 MB L2",
                   "parallelism": f"replicas x{world} (weak; independent sequence shards)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(name),
                     "algorithmic_bytes_per_launch": ssu_bytes,
                     "launch_ms": launch_max, "peak_source": f"{peak_kind} hbm_gbs"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": step.launches * args.steps,
        "device_error": device_error,
        "clocks": clocks.summary(),
    }
    if device_error:
        raise SystemExit(f"{case.name}: the device error word is {device_error:#x} after the "
                         "timed steps (a bounded wait gave up)")
    if cpu and rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_leg(step, 256 if name == DEFAULT_WORKLOAD else 48,
                                      args.cpu_seconds if name == DEFAULT_WORKLOAD
                                      else args.cpu_seconds / 2)
    del step, case
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    from mamba2_ssm_decode_gb300 import build as _b
    world, rank, local = dist_setup(args.gpus)
    if rank == 0 or world == 1:
        _b.build()
    barrier(world)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    peak, peak_kind = measured_peak()

    if args.workload == SSD_WORKLOAD:   # the packed SSD prefill on its own
        if world > 1:
            raise SystemExit("the SSD prefill leg runs on one GPU")
        line = ssd_leg(args, device, stream, peak, peak_kind, args.steps)
        line.update({"n_gpus": 1, "warmup": max(3, args.warmup), "scaling": "weak",
                     "vs_baseline": None, "data": DATA})
        print(json.dumps(line), flush=True)
        return
    h = headline(args.workload, args, world, device, stream, peak, peak_kind)
    line = {
        "metric": "SSU decode tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)",
        "value": h["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": h["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": DATA,
        "config": h["config"], "hbm_gbs": h["roofline"]["achieved"],
        "roofline": h["roofline"], "e2e": h["e2e"], "gpu_launches": h["gpu_launches"],
        "device_error": h["device_error"], "clocks": h["clocks"],
    }
    if "cpu_baseline" in h:
        line["cpu_baseline"] = h["cpu_baseline"]
    if not args.no_extras and world == 1:
        line["workloads"] = {}
        for name in EXTRAS:
            c2, s2, r = measure(name, device, args.seed, max(5, min(args.steps, 50)), 3, stream,
                                args.algorithm)
            r["frac"] = r["gbs"] / peak
            line["workloads"][c2.name] = {k: r[k] for k in ("tokens_per_s", "gbs", "frac",
                                                             "launch_ms", "ms_per_step")}
            del c2, s2
            torch.cuda.empty_cache()
        line["large_batch"] = {}
        for name in LARGE:
            r = headline(name, args, world, device, stream, peak, peak_kind)
            line["large_batch"][r["config"]["workload"]] = r
        line["ssd_prefill"] = ssd_leg(args, device, stream, peak, peak_kind,
                                      max(5, min(args.steps, 200)))
        line["device_error_after_extras"] = step_error = \
            __import__("mamba2_ssm_decode_gb300").ssu_device_error()
        if step_error:
            raise SystemExit(f"device error word {step_error:#x} after the extra workloads")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The reference arm: the CPU oracle on the same workload, rank 0 only; each
    step runs a bounded sample (the first 32 sequences) on all host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from mamba2_ssm_decode_gb300 import workloads as W
    oracle.build()
    case = _workload(args.workload, "cpu", args.seed)
    tokens_full, _, _ = accounting(case)
    nsample = min(32, case.nseqs)
    sample, _, _ = W.subset_case(case, list(range(nsample)))
    toks, _, _ = accounting(sample)
    ncores = max(1, min(os.cpu_count() or 1, nsample))
    bounds = [nsample * k // ncores for k in range(ncores + 1)]
    shards = [W.subset_case(sample, list(range(bounds[k], bounds[k + 1])))[0]
              for k in range(ncores) if bounds[k + 1] > bounds[k]]
    _time_oracle(shards, len(shards), 0.0, passes=args.warmup)
    per_pass, _, _ = _time_oracle(shards, len(shards), 0.0, passes=args.steps)
    secs = per_pass * args.steps
    value = toks * args.steps / secs
    slots, H, P, N, G = case.dims
    sample_desc = (f"first {nsample} of the {case.nseqs} sequences of {case.name} "
                   f"({toks} tokens) per step, fp64 C oracle on {len(shards)} host threads "
                   f"(contiguous shards)")
    line = {
        "impl": "reference",
        "metric": "SSU decode tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA,
        "config": {"workload": case.name, "batch": case.nseqs, "nheads": H, "headdim": P,
                   "dstate": N, "ngroups": G, "state_dtype": str(case.state.dtype)[6:],
                   "non_pad_tokens": tokens_full, "parallelism": "rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": len(shards),
                         "kind": "oracle", "sample": sample_desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 2000; 20 for --impl reference)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--algorithm", choices=["auto", "direct", "bulk"], default="auto")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    sys.path.insert(0, ROOT)
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 2000
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
