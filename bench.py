"""Benchmark of the Mamba2 selective-state-update decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-extras] [--no-cpu-baseline]

One step is one pass of the decode hot path over one batch of seeded synthetic
inputs (resident in HBM): for the default workload (Mamba2-2.7B-shaped
decode: batch 256, 80 heads, headdim 64, dstate 128, fp32 state pool of 512
slots, 5% pad) that is one ssu_update launch; for the MTP workload one
ssu_update_varlen launch plus the ReplaySSM tracker update and commit.

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
    m = re.fullmatch(r"sweep-(single|mtp)-(float32|bfloat16)-b(\d+)(-nowrite)?", name)
    if m:
        return W.sweep_case(int(m.group(3)), getattr(torch, m.group(2)), m.group(1),
                            disable_state_update=bool(m.group(4)), seed=seed, device=device)
    raise SystemExit(f"unknown workload {name}")


def _esize(t):
    return 0 if t is None else t.element_size()


def accounting(case):
    """(non-pad tokens, algorithmic bytes of the SSU launch, tracker bytes).

    Algorithmic bytes per launch: every sequence with a valid read slot reads
    its H x P x N state block once and writes it once per valid destination
    write; every packed row reads x, z, dt, B, C and writes y; plus the index
    tables and metadata (read once).  Pad sequences move no state."""
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
        self.launches = 1 + (2 if case.ring_start is not None else 0)
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

    def ssu_launch(self, x=None, z=None, dt=None, B=None, C=None, sbi=None, out=None):
        c = self.case
        x = c.x if x is None else x
        z = c.z if z is None else z
        dt = c.dt if dt is None else dt
        B = c.B if B is None else B
        C = c.C if C is None else C
        sbi = c.state_batch_indices if sbi is None else sbi
        out = self.out if out is None else out
        kw = dict(D=c.D, z=z, dt_bias=c.dt_bias, dt_softplus=c.dt_softplus,
                  pad_slot_id=c.pad_slot_id, disable_state_update=c.disable_state_update,
                  out=out, algorithm=self.algorithm)
        if c.kind == "single":
            self.ssu.ssu_update(c.state, x, dt, c.A, B, C, state_batch_indices=sbi,
                                dst_state_batch_indices=c.dst_state_batch_indices, **kw)
        elif self.v4 is not None:
            v = self.v4
            kw["z"], kw["out"] = v(z), v(out)
            self.ssu.ssu_update_varlen(c.state, v(x), v(dt), c.A, v(B), v(C),
                                       num_accepted_tokens=c.num_accepted_tokens,
                                       state_batch_indices=sbi,
                                       dst_state_batch_indices=c.dst_state_batch_indices, **kw)
        else:
            self.ssu.ssu_update_varlen(c.state, x, dt, c.A, B, C, cu_seqlens=c.cu_seqlens,
                                       num_accepted_tokens=c.num_accepted_tokens,
                                       state_batch_indices=sbi,
                                       dst_state_batch_indices=c.dst_state_batch_indices,
                                       nseqs=c.nseqs, **kw)

    def trackers(self, sbi=None):
        c = self.case
        if c.ring_start is None:
            return
        sbi = c.state_batch_indices if sbi is None else sbi
        tr = (c.ring_start, c.prev_num_accepted, c.prev_query_len)
        self.ssu.ssu_ring_update(*tr, sbi, c.logical_window, c.ring_buffer_len,
                                 pad_slot_id=c.pad_slot_id)
        self.ssu.ssu_ring_commit(*tr, sbi, c.num_accepted_tokens, c.cu_seqlens,
                                 c.logical_window, c.ring_buffer_len, pad_slot_id=c.pad_slot_id)

    def __call__(self):
        self.ssu_launch()
        self.trackers()


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons for this GPU."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        props = torch.cuda.get_device_properties(device)
        self.uuid = str(getattr(props, "uuid", "")).lower().replace("gpu-", "")
        self.samples = []
        self.proc = None
        self.thread = None
        self.marks = {}

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            uuid = parts[0].lower().replace("gpu-", "")
            if self.uuid and uuid != self.uuid:
                continue
            self.samples.append((time.perf_counter(), parts[1:]))

    def mark(self, name):
        self.marks[name] = time.perf_counter()

    def stop(self):
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
        inside = [s for t, s in self.samples if t0 is not None and t0 <= t <= t1]
        pool = inside or [s for _, s in self.samples]

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(s[0]) for s in pool if num(s[0]) is not None]
        mx = [num(s[1]) for s in pool if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in pool for n, v in zip(names, s[4:8]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(pool), "samples_in_timed_region": len(inside)}


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


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mamba2_ssm_decode_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    valid only while the kernel sources hash to the value recorded with it."""
    path = os.path.join(ROOT, "profiles", f"ssu_{workload}_dram.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"^kernel_source_hash:\s*(\w+)", text, re.M)
    m_val = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    if not (m_hash and m_val) or m_hash.group(1) != kernel_source_hash():
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
    its inputs (x, z, dt, B, C, slot table) from pinned host memory, runs the
    call and copies y back, then waits for it."""
    c = step.case
    names = ["x", "z", "dt", "B", "C", "state_batch_indices"]
    host = {n: getattr(c, n).cpu().pin_memory() for n in names if getattr(c, n) is not None}
    dev = {n: torch.empty_like(getattr(c, n)) for n in host}
    y_host = torch.empty(c.x.shape, dtype=c.x.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = y_host.numel() * y_host.element_size()

    def one():
        with torch.cuda.stream(stream):
            for n, t in host.items():
                dev[n].copy_(t, non_blocking=True)
            step.ssu_launch(x=dev["x"], z=dev.get("z"), dt=dev["dt"], B=dev["B"], C=dev["C"],
                            sbi=dev.get("state_batch_indices"))
            step.trackers(sbi=dev.get("state_batch_indices"))
            y_host.copy_(step.out, non_blocking=True)
        stream.synchronize()

    for _ in range(warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    return (time.perf_counter() - t0) * 1e3 / steps, h2d, d2h


def cpu_baseline(case, min_seconds=10.0):
    """The oracle (plain fp64 C, one thread) on host copies of the workload,
    repeated until about `min_seconds` of CPU work."""
    import oracle
    cpu = case.to("cpu")
    tokens, _, _ = accounting(cpu)
    reps = 0
    t0 = time.perf_counter()
    while True:
        state = cpu.state.clone()
        kw = dict(D=cpu.D, z=cpu.z, dt_bias=cpu.dt_bias, dt_softplus=cpu.dt_softplus,
                  pad_slot_id=cpu.pad_slot_id, disable_state_update=cpu.disable_state_update,
                  state_batch_indices=cpu.state_batch_indices,
                  dst_state_batch_indices=cpu.dst_state_batch_indices)
        t = time.perf_counter()
        if cpu.kind == "single":
            oracle.ssu_update(state, cpu.x, cpu.dt, cpu.A, cpu.B, cpu.C, **kw)
        else:
            oracle.ssu_update_varlen(state, cpu.x, cpu.dt, cpu.A, cpu.B, cpu.C,
                                     cu_seqlens=cpu.cu_seqlens, nseqs=cpu.nseqs,
                                     dense_steps=cpu.dense_steps,
                                     num_accepted_tokens=cpu.num_accepted_tokens, **kw)
        reps += 1
        if time.perf_counter() - t0 >= min_seconds:
            break
    secs = time.perf_counter() - t0
    return {"value": tokens * reps / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"the whole {case.name} batch ({tokens} tokens), {reps} repetitions, "
                      f"{secs:.1f} s on one host core (fp64 C oracle)"}


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
EXTRAS = ["hybrid-grouped-decode", "mtp-varlen",
          "sweep-single-float32-b1024", "sweep-single-bfloat16-b1024",
          "sweep-mtp-float32-b1024", "sweep-mtp-bfloat16-b1024",
          "sweep-single-float32-b4096", "sweep-single-bfloat16-b4096",
          "sweep-mtp-float32-b4096", "sweep-mtp-bfloat16-b4096",
          "sweep-single-float32-b1024-nowrite", "sweep-single-bfloat16-b1024-nowrite",
          "sweep-mtp-float32-b1024-nowrite", "sweep-mtp-bfloat16-b1024-nowrite"]


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


def run_ours(args):
    from mamba2_ssm_decode_gb300 import build as _b
    world, rank, local = dist_setup(args.gpus)
    if rank == 0 or world == 1:
        _b.build()
    barrier(world)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    seed = args.seed + rank   # each rank: its own shard of sequences

    case = _workload(args.workload, device, seed)
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
    total_max = max_over_ranks(total, world, device)
    launch_max = max_over_ranks(launch, world, device)
    tokens_all = sum_over_ranks(tokens * args.steps, world, device)
    ms = total_max / args.steps
    value = tokens_all / (total_max * 1e-3)

    # end to end through the public API with host buffers
    e2e_ms, h2d, d2h = e2e(step, max(3, min(args.steps, 200)), 3, stream)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_value = sum_over_ranks(tokens, world, device) / (e2e_ms * 1e-3)

    peak, peak_kind = measured_peak()
    achieved = ssu_bytes / (launch_max * 1e-3) / 1e9
    slots, H, P, N, G = case.dims
    line = {
        "metric": "SSU decode tokens/s and achieved HBM GB/s vs GB300 peak (1 GPU)",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": DATA,
        "config": {"workload": case.name, "batch": case.nseqs, "nheads": H, "headdim": P,
                   "dstate": N, "ngroups": G, "state_dtype": str(case.state.dtype)[6:],
                   "io_dtype": str(case.x.dtype)[6:], "slots": slots, "non_pad_tokens": tokens,
                   "algorithm": args.algorithm,
                   "l2": f"no flush: each step touches {ssu_bytes / 1e9:.2f} GB > 129 MB L2",
                   "parallelism": f"replicas x{world} (weak; independent sequence shards)"},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(args.workload),
                     "algorithmic_bytes_per_launch": ssu_bytes,
                     "launch_ms": launch_max, "peak_source": f"{peak_kind} hbm_gbs"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": step.launches * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_extras and world == 1:
        line["workloads"] = {}
        del case, step
        torch.cuda.empty_cache()
        for name in EXTRAS:
            c2, s2, r = measure(name, device, args.seed, max(5, min(args.steps, 50)), 3, stream,
                                args.algorithm)
            r["frac"] = r["gbs"] / peak
            line["workloads"][c2.name] = {k: r[k] for k in ("tokens_per_s", "gbs", "frac",
                                                             "launch_ms", "ms_per_step")}
            del c2, s2
            torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(_workload(args.workload, "cpu", args.seed),
                                            min_seconds=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The reference arm: the CPU oracle on the same workload, rank 0 only."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    case = _workload(args.workload, "cpu", args.seed)
    tokens_full, _, _ = accounting(case)
    # each step: the oracle on a 32-sequence sample of the batch
    from mamba2_ssm_decode_gb300 import workloads as W  # noqa: F401
    nsample = min(32, case.nseqs)
    sample = _sample_sequences(case, nsample)
    toks, _, _ = accounting(sample)

    def one():
        st = sample.state.clone()
        kw = dict(D=sample.D, z=sample.z, dt_bias=sample.dt_bias, dt_softplus=sample.dt_softplus,
                  pad_slot_id=sample.pad_slot_id,
                  disable_state_update=sample.disable_state_update,
                  state_batch_indices=sample.state_batch_indices,
                  dst_state_batch_indices=sample.dst_state_batch_indices)
        if sample.kind == "single":
            oracle.ssu_update(st, sample.x, sample.dt, sample.A, sample.B, sample.C, **kw)
        else:
            oracle.ssu_update_varlen(st, sample.x, sample.dt, sample.A, sample.B, sample.C,
                                     cu_seqlens=sample.cu_seqlens, nseqs=sample.nseqs,
                                     dense_steps=sample.dense_steps,
                                     num_accepted_tokens=sample.num_accepted_tokens, **kw)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    secs = time.perf_counter() - t0
    value = toks * args.steps / secs
    slots, H, P, N, G = case.dims
    sample_desc = (f"first {nsample} of the {case.nseqs} sequences of {case.name} "
                   f"({toks} tokens) per step, fp64 C oracle, one host core")
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
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample_desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _sample_sequences(case, n):
    """The first n sequences of a CPU case, as a case of their own (same slots)."""
    import dataclasses
    if case.kind == "single":
        rows = slice(0, n)
        return dataclasses.replace(
            case, x=case.x[rows], z=None if case.z is None else case.z[rows], dt=case.dt[rows],
            B=case.B[rows], C=case.C[rows],
            state_batch_indices=None if case.state_batch_indices is None
            else case.state_batch_indices[:n],
            dst_state_batch_indices=None if case.dst_state_batch_indices is None
            else case.dst_state_batch_indices[:n], nseqs=n)
    if case.cu_seqlens is not None:
        end = int(case.cu_seqlens[n])
        cu = case.cu_seqlens[: n + 1]
    else:
        end = n * case.dense_steps
        cu = None
    rows = slice(0, end)
    return dataclasses.replace(
        case, x=case.x[rows], z=None if case.z is None else case.z[rows], dt=case.dt[rows],
        B=case.B[rows], C=case.C[rows], cu_seqlens=cu,
        num_accepted_tokens=None if case.num_accepted_tokens is None
        else case.num_accepted_tokens[:n],
        state_batch_indices=None if case.state_batch_indices is None
        else case.state_batch_indices[:n],
        dst_state_batch_indices=None if case.dst_state_batch_indices is None
        else case.dst_state_batch_indices[:n], nseqs=n)


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
