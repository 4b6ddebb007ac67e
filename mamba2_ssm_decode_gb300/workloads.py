"""Seeded synthetic inputs shaped like Mamba2 serving decode.

This module only draws random tensors and slot tables; it holds none of the
selective-state-update arithmetic.  Both the CUDA path and the CPU oracle are
fed from it.  Value distributions (the same for every workload):

  state    ~ N(0, 0.1^2)            (std 0.1), in the state dtype
  x, z     ~ N(0, 1)                in the io dtype (bf16 unless stated)
  B, C     ~ N(0, 1)                [rows, groups, dstate], io dtype
  dt       ~ N(0, 1)                fp32, per head [rows, heads] unless dt_per_dim
  dt_bias  ~ U[-4, -1]              fp32 per head
  A        = -exp(U[0, ln 16])      fp32 per head, so A in [-16, -1]
  D        ~ U[0, 1]                fp32 per head

Slot tables are random subsets of the slot pool (distinct slots), with a
seeded choice of sequences whose slots are replaced by the pad id.
"""
from __future__ import annotations

import dataclasses
import math

import torch

PAD_SLOT_ID = -1


@dataclasses.dataclass
class SSUCase:
    """One call's inputs.  `kind` is "single" (one token per sequence) or "varlen"."""

    kind: str
    name: str
    state: torch.Tensor                 # [slots, H, P, N]
    x: torch.Tensor                     # [rows, H, P]
    dt: torch.Tensor                    # [rows, H] or [rows, H, P] fp32
    A: torch.Tensor                     # [H] fp32
    B: torch.Tensor                     # [rows, G, N]
    C: torch.Tensor                     # [rows, G, N]
    D: torch.Tensor | None              # [H] fp32
    dt_bias: torch.Tensor | None        # [H] fp32
    z: torch.Tensor | None              # [rows, H, P]
    state_batch_indices: torch.Tensor | None
    dst_state_batch_indices: torch.Tensor | None = None
    cu_seqlens: torch.Tensor | None = None
    num_accepted_tokens: torch.Tensor | None = None
    dense_steps: int = 1
    nseqs: int = 0
    pad_slot_id: int = PAD_SLOT_ID
    dt_softplus: bool = True
    disable_state_update: bool = False
    # ReplaySSM trackers (int32 [num_states]) and their parameters, when the
    # workload runs them
    ring_start: torch.Tensor | None = None
    prev_num_accepted: torch.Tensor | None = None
    prev_query_len: torch.Tensor | None = None
    logical_window: int = 0
    ring_buffer_len: int = 1
    # ReplaySSM checkpointing calls (kind "replay"): the ring caches, and whether
    # the call applies the one-token tracker update itself
    x_cache: torch.Tensor | None = None   # [slots, H, R, P]
    B_cache: torch.Tensor | None = None   # [slots, G, R, N]
    dt_cache: torch.Tensor | None = None  # [slots, H, R] fp32
    update_trackers: bool = False
    # stochastic rounding of 16-bit state: the call's random seed (None: off)
    sr_seed: int | None = None

    @property
    def rows(self) -> int:
        return self.x.shape[0]

    @property
    def dims(self):
        slots, H, P, N = self.state.shape
        return slots, H, P, N, self.B.shape[1]

    def tensors(self) -> dict:
        return {f.name: getattr(self, f.name) for f in dataclasses.fields(self)
                if isinstance(getattr(self, f.name), torch.Tensor)}

    def to(self, device) -> "SSUCase":
        kw = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            kw[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return SSUCase(**kw)

    def clone(self) -> "SSUCase":
        kw = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            kw[f.name] = v.clone() if isinstance(v, torch.Tensor) else v
        return SSUCase(**kw)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, dtype, g, device):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _uniform(shape, lo, hi, g, device):
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def _head_params(H, g, device):
    A = -torch.exp(_uniform((H,), 0.0, math.log(16.0), g, device))
    D = _uniform((H,), 0.0, 1.0, g, device)
    dt_bias = _uniform((H,), -4.0, -1.0, g, device)
    return A, D, dt_bias


def _channel_params(H, P, g, device):
    """A, D, dt_bias per (head, dim) channel [H, P], same distributions."""
    A = -torch.exp(_uniform((H, P), 0.0, math.log(16.0), g, device))
    D = _uniform((H, P), 0.0, 1.0, g, device)
    dt_bias = _uniform((H, P), -4.0, -1.0, g, device)
    return A, D, dt_bias


def _distinct_slots(count, slots, g, device):
    if count > slots:
        raise ValueError(f"need {count} distinct slots from a pool of {slots}")
    return torch.randperm(slots, generator=g, device=device)[:count]


def _pad_some(table, npad, pad, g, device):
    """Replace the slots of `npad` seeded sequences (whole rows) by the pad id."""
    if npad <= 0:
        return table
    who = torch.randperm(table.shape[0], generator=g, device=device)[:npad]
    table = table.clone()
    table[who] = pad
    return table


def single_token_case(*, batch, heads, headdim, dstate, groups, slots, state_dtype,
                      io_dtype=torch.bfloat16, pad_frac=0.0, with_z=True, dt_per_dim=False,
                      index_dtype=torch.int32, identity_slots=False, disable_state_update=False,
                      per_channel=False, seed=0, device="cpu", name="single") -> SSUCase:
    g = _gen(seed, device)
    state = _normal((slots, heads, headdim, dstate), 0.1, state_dtype, g, device)
    x = _normal((batch, heads, headdim), 1.0, io_dtype, g, device)
    dt_shape = (batch, heads, headdim) if dt_per_dim else (batch, heads)
    dt = _normal(dt_shape, 1.0, torch.float32, g, device)
    A, D, dt_bias = (_channel_params(heads, headdim, g, device) if per_channel
                     else _head_params(heads, g, device))
    B = _normal((batch, groups, dstate), 1.0, io_dtype, g, device)
    C = _normal((batch, groups, dstate), 1.0, io_dtype, g, device)
    z = _normal((batch, heads, headdim), 1.0, io_dtype, g, device) if with_z else None
    if identity_slots:
        sbi = torch.arange(batch, device=device)
    else:
        sbi = _distinct_slots(batch, slots, g, device)
    sbi = _pad_some(sbi, round(pad_frac * batch), PAD_SLOT_ID, g, device).to(index_dtype)
    return SSUCase(kind="single", name=name, state=state, x=x, dt=dt, A=A, B=B, C=C, D=D,
                   dt_bias=dt_bias, z=z, state_batch_indices=sbi, nseqs=batch,
                   disable_state_update=disable_state_update)


def varlen_case(*, nseqs, max_len, heads, headdim, dstate, groups, slots, state_dtype,
                io_dtype=torch.bfloat16, fixed_len=None, pad_frac=0.0, with_z=True,
                dt_per_dim=False, index_dtype=torch.int32, meta_dtype=torch.int32,
                same_tables=False, dense=False, with_trackers=False, logical_window=4,
                ring_buffer_len=8, disable_state_update=False, seed=0, device="cpu",
                name="varlen") -> SSUCase:
    """Packed varlen MTP call.  Lengths are U{1..max_len} (or `fixed_len`), the
    acceptance count of sequence s is U{1..len_s}; the read table and the write
    table are [nseqs, max_len] of distinct slots (one table when same_tables)."""
    g = _gen(seed, device)
    if fixed_len is not None:
        lens = torch.full((nseqs,), fixed_len, dtype=torch.int64, device=device)
    else:
        lens = torch.randint(1, max_len + 1, (nseqs,), generator=g, device=device)
    cu = torch.zeros(nseqs + 1, dtype=torch.int64, device=device)
    cu[1:] = torch.cumsum(lens, 0)
    rows = int(cu[-1].item())
    # acceptance count U{1..len}: floor(u * len) + 1
    u = torch.rand((nseqs,), generator=g, device=device)
    na = (torch.floor(u * lens.to(torch.float32)).to(torch.int64) + 1).clamp(max=lens)
    ntab = 1 if same_tables else 2
    perm = _distinct_slots(ntab * nseqs * max_len, slots, g, device)
    sbi = perm[: nseqs * max_len].reshape(nseqs, max_len)
    dsbi = sbi if same_tables else perm[nseqs * max_len:].reshape(nseqs, max_len)
    npad = round(pad_frac * nseqs)
    if npad:
        who = torch.randperm(nseqs, generator=g, device=device)[:npad]
        sbi = sbi.clone()
        sbi[who] = PAD_SLOT_ID
        dsbi = sbi if same_tables else dsbi.clone()
        if not same_tables:
            dsbi[who] = PAD_SLOT_ID
    state = _normal((slots, heads, headdim, dstate), 0.1, state_dtype, g, device)
    x = _normal((rows, heads, headdim), 1.0, io_dtype, g, device)
    dt_shape = (rows, heads, headdim) if dt_per_dim else (rows, heads)
    dt = _normal(dt_shape, 1.0, torch.float32, g, device)
    A, D, dt_bias = _head_params(heads, g, device)
    B = _normal((rows, groups, dstate), 1.0, io_dtype, g, device)
    C = _normal((rows, groups, dstate), 1.0, io_dtype, g, device)
    z = _normal((rows, heads, headdim), 1.0, io_dtype, g, device) if with_z else None
    case = SSUCase(kind="varlen", name=name, state=state, x=x, dt=dt, A=A, B=B, C=C, D=D,
                   dt_bias=dt_bias, z=z, state_batch_indices=sbi.to(index_dtype),
                   dst_state_batch_indices=None if same_tables else dsbi.to(index_dtype),
                   cu_seqlens=None if dense else cu.to(meta_dtype),
                   num_accepted_tokens=na.to(meta_dtype), dense_steps=fixed_len or 1,
                   nseqs=nseqs, disable_state_update=disable_state_update)
    if dense and fixed_len is None:
        raise ValueError("a dense call needs fixed_len")
    if with_trackers:
        case.ring_start = torch.randint(0, ring_buffer_len, (slots,), generator=g, device=device,
                                        dtype=torch.int64).to(torch.int32)
        case.prev_num_accepted = torch.randint(0, logical_window + 1, (slots,), generator=g,
                                               device=device, dtype=torch.int64).to(torch.int32)
        case.prev_query_len = torch.randint(0, max_len + 1, (slots,), generator=g, device=device,
                                            dtype=torch.int64).to(torch.int32)
        case.logical_window = logical_window
        case.ring_buffer_len = ring_buffer_len
    return case


def replay_case(*, nseqs, heads, headdim, dstate, groups, slots, state_dtype,
                io_dtype=torch.bfloat16, max_len=1, logical_window=4, ring_len=8,
                pad_frac=0.0, with_z=True, index_dtype=torch.int32, meta_dtype=torch.int32,
                update_trackers=None, seed=0, device="cpu", name="replay") -> SSUCase:
    """A ReplaySSM checkpointing call: checkpoints ~N(0, 0.1^2); ring caches
    holding earlier tokens (x, B ~N(0, 1) in the io dtype, dt ~N(0, 1)); int32
    trackers by slot with ring_start U{0..R-1} and, for each sequence's slot,
    k = prev_num_accepted U{1..W} for one-token calls (the values the update
    rule cycles through) or U{0..max(W, max_len)} after a commit, capped so the
    ring holds k + L tokens.  max_len 1: one row per sequence (no cu_seqlens);
    else lengths U{1..max_len} packed with cu_seqlens.  update_trackers
    defaults to on for one-token calls, off for packed ones (their trackers
    move by the commit)."""
    g = _gen(seed, device)
    one = max_len == 1
    if one:
        lens = torch.ones(nseqs, dtype=torch.int64, device=device)
    else:
        lens = torch.randint(1, max_len + 1, (nseqs,), generator=g, device=device)
    rows = int(lens.sum().item())
    state = _normal((slots, heads, headdim, dstate), 0.1, state_dtype, g, device)
    x = _normal((rows, heads, headdim), 1.0, io_dtype, g, device)
    dt = _normal((rows, heads), 1.0, torch.float32, g, device)
    A, D, dt_bias = _head_params(heads, g, device)
    B = _normal((rows, groups, dstate), 1.0, io_dtype, g, device)
    C = _normal((rows, groups, dstate), 1.0, io_dtype, g, device)
    z = _normal((rows, heads, headdim), 1.0, io_dtype, g, device) if with_z else None
    sbi = _distinct_slots(nseqs, slots, g, device)
    sbi = _pad_some(sbi, round(pad_frac * nseqs), PAD_SLOT_ID, g, device)
    xc = _normal((slots, heads, ring_len, headdim), 1.0, io_dtype, g, device)
    Bc = _normal((slots, groups, ring_len, dstate), 1.0, io_dtype, g, device)
    dc = _normal((slots, heads, ring_len), 1.0, torch.float32, g, device)
    rs = torch.randint(0, ring_len, (slots,), generator=g, device=device, dtype=torch.int64)
    lo, hi = (1, logical_window) if one else (0, max(logical_window, max_len))
    u = torch.rand((nseqs,), generator=g, device=device)
    cap = torch.clamp(ring_len - lens, min=0)
    k = torch.minimum(lo + torch.floor(u * (hi - lo + 1)).to(torch.int64), cap)
    pna = torch.zeros(slots, dtype=torch.int64, device=device)
    valid = sbi >= 0
    pna[sbi[valid]] = k[valid]
    cu = None
    if not one:
        cu = torch.zeros(nseqs + 1, dtype=torch.int64, device=device)
        cu[1:] = torch.cumsum(lens, 0)
        cu = cu.to(meta_dtype)
    return SSUCase(kind="replay", name=name, state=state, x=x, dt=dt, A=A, B=B, C=C, D=D,
                   dt_bias=dt_bias, z=z, state_batch_indices=sbi.to(index_dtype), cu_seqlens=cu,
                   nseqs=nseqs, ring_start=rs.to(torch.int32),
                   prev_num_accepted=pna.to(torch.int32),
                   prev_query_len=torch.zeros(slots, dtype=torch.int32, device=device),
                   logical_window=logical_window, ring_buffer_len=ring_len, x_cache=xc,
                   B_cache=Bc, dt_cache=dc,
                   update_trackers=one if update_trackers is None else update_trackers)


def replay_decode(seed=0, device="cpu") -> SSUCase:
    """ReplaySSM one-token decode shaped like the Mamba2-2.7B decode: batch 256,
    80 heads, headdim 64, dstate 128, 1 group, fp32 checkpoints in a pool of
    512 slots, 5% pad; window 4, ring 8; the tracker update in the call."""
    return replay_case(nseqs=256, heads=80, headdim=64, dstate=128, groups=1, slots=512,
                       state_dtype=torch.float32, pad_frac=0.05, logical_window=4, ring_len=8,
                       seed=seed, device=device, name="replay-decode-b256")


def replay_mtp(seed=0, device="cpu") -> SSUCase:
    """ReplaySSM speculative pass shaped like the packed MTP workload: 128
    sequences of U{1..4} rows, 80 heads, headdim 64, dstate 128, 1 group, fp32
    checkpoints in a pool of 1024 slots; window 4, ring 8; trackers as left by
    a commit (moved by ssu_ring_commit, not by the call)."""
    return replay_case(nseqs=128, heads=80, headdim=64, dstate=128, groups=1, slots=1024,
                       state_dtype=torch.float32, max_len=4, logical_window=4, ring_len=8,
                       seed=seed, device=device, name="replay-mtp-s128")


# ---------------------------------------------------------------------------
# the named serving workloads
# ---------------------------------------------------------------------------

def tiny(seed=0, device="cpu", dt_per_dim=False) -> SSUCase:
    """Tiny single-token decode: batch 4, 8 heads, headdim 64, dstate 16, 1 group,
    fp32 state [4, 8, 64, 16], identity slot map, no z."""
    return single_token_case(batch=4, heads=8, headdim=64, dstate=16, groups=1, slots=4,
                             state_dtype=torch.float32, with_z=False, dt_per_dim=dt_per_dim,
                             identity_slots=True, seed=seed, device=device, name="tiny")


def mamba2_2p7b_decode(seed=0, device="cpu") -> SSUCase:
    """Mamba2-2.7B-shaped decode: batch 256, 80 heads, headdim 64, dstate 128,
    1 group, fp32 state pool of 512 slots; int32 slot vector = a random subset
    with 5% (13) of its entries set to the pad id; z gating on."""
    return single_token_case(batch=256, heads=80, headdim=64, dstate=128, groups=1, slots=512,
                             state_dtype=torch.float32, pad_frac=0.05, seed=seed, device=device,
                             name="mamba2-2.7b-decode-b256")


def hybrid_grouped_decode(seed=0, device="cpu") -> SSUCase:
    """Hybrid-model decode: batch 1024, 128 heads, headdim 64, dstate 128,
    8 groups (16 heads per group), bf16 state pool of 2048 slots, z on."""
    return single_token_case(batch=1024, heads=128, headdim=64, dstate=128, groups=8,
                             slots=2048, state_dtype=torch.bfloat16, seed=seed, device=device,
                             name="hybrid-grouped-decode-b1024")


def mtp_varlen(seed=0, device="cpu") -> SSUCase:
    """Packed varlen MTP decode: 128 sequences of U{1..4} rows (int32
    cu_seqlens), 80 heads, headdim 64, dstate 128, 1 group, fp32 state pool of
    1024; acceptance counts U{1..len}; read and write tables [128, 4] int32 of
    distinct slots; ReplaySSM trackers int32 [1024] with window 4, ring 8."""
    return varlen_case(nseqs=128, max_len=4, heads=80, headdim=64, dstate=128, groups=1,
                       slots=1024, state_dtype=torch.float32, with_trackers=True,
                       logical_window=4, ring_buffer_len=8, seed=seed, device=device,
                       name="mtp-varlen-s128")


def mamba2_2p7b_decode_perchannel(seed=0, device="cpu") -> SSUCase:
    """The Mamba2-2.7B-shaped decode with A, D and dt_bias given per (head, dim)
    channel ([80, 64] fp32; "mate.mamba" _per_head's channel-wise form)."""
    return single_token_case(batch=256, heads=80, headdim=64, dstate=128, groups=1, slots=512,
                             state_dtype=torch.float32, pad_frac=0.05, per_channel=True,
                             seed=seed, device=device, name="mamba2-2.7b-decode-perchannel-b256")


def mtp_varlen_dt_per_dim(seed=0, device="cpu") -> SSUCase:
    """The packed varlen MTP workload with a full [rows, 80, 64] dt (one dt per
    head and dim) instead of one per head."""
    return varlen_case(nseqs=128, max_len=4, heads=80, headdim=64, dstate=128, groups=1,
                       slots=1024, state_dtype=torch.float32, dt_per_dim=True, seed=seed,
                       device=device, name="mtp-varlen-dtperdim-s128")


def sweep_case(batch, state_dtype, mode, disable_state_update=False, seed=0,
               device="cpu", stochastic_rounding=False) -> SSUCase:
    """Large-batch sweep point: 128 heads, headdim 64, dstate 128, 8 groups,
    int64 slot tables with 2% pad sequences, z on.  mode "single": pool 2*batch;
    mode "mtp": dense 4-step call, one [batch, 4] read/write table of distinct
    slots (pool 4*batch, the smallest that holds four write slots per sequence)."""
    name = f"sweep-{mode}-{str(state_dtype).split('.')[-1]}-b{batch}"
    if disable_state_update:
        name += "-nowrite"
    if stochastic_rounding:
        name += "-sr"
    if mode == "single":
        c = single_token_case(batch=batch, heads=128, headdim=64, dstate=128, groups=8,
                              slots=2 * batch, state_dtype=state_dtype, pad_frac=0.02,
                              index_dtype=torch.int64,
                              disable_state_update=disable_state_update, seed=seed,
                              device=device, name=name)
    elif mode == "mtp":
        c = varlen_case(nseqs=batch, max_len=4, fixed_len=4, heads=128, headdim=64,
                        dstate=128, groups=8, slots=4 * batch, state_dtype=state_dtype,
                        pad_frac=0.02, index_dtype=torch.int64, meta_dtype=torch.int64,
                        same_tables=True, dense=True,
                        disable_state_update=disable_state_update, seed=seed,
                        device=device, name=name)
    else:
        raise ValueError(mode)
    if stochastic_rounding:   # a fixed seed stands in for the per-call draw
        c.sr_seed = 0x2545F4914F6CDD1D ^ seed
    return c


WORKLOADS = {
    "tiny": tiny,
    "mamba2-2.7b-decode": mamba2_2p7b_decode,
    "hybrid-grouped-decode": hybrid_grouped_decode,
    "mtp-varlen": mtp_varlen,
    "mamba2-2.7b-decode-perchannel": mamba2_2p7b_decode_perchannel,
    "mtp-varlen-dtperdim": mtp_varlen_dt_per_dim,
    "replay-decode": replay_decode,
    "replay-mtp": replay_mtp,
}


# ---------------------------------------------------------------------------
# packed SSD prefill
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class SSDCase:
    """One packed SSD prefill call's inputs ("mate.mamba", ssd_combined_fwd_varlen)."""

    name: str
    x: torch.Tensor                     # [tokens, H, P]
    dt: torch.Tensor                    # [tokens, H] fp32
    A: torch.Tensor                     # [H] fp32
    B: torch.Tensor                     # [tokens, G, N]
    C: torch.Tensor                     # [tokens, G, N]
    D: torch.Tensor | None
    z: torch.Tensor | None
    dt_bias: torch.Tensor | None
    chunk_size: int
    cu_seqlens: torch.Tensor            # [batch + 1]
    cu_chunk_seqlens: torch.Tensor      # [nchunks + 1]
    last_chunk_indices: torch.Tensor    # [batch]
    seq_idx: torch.Tensor               # [nchunks]
    initial_states: torch.Tensor | None  # [batch, H, P, N]
    dt_softplus: bool = True
    dt_limit: tuple = (0.0, float("inf"))

    def to(self, device) -> "SSDCase":
        kw = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            kw[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return SSDCase(**kw)


def chunk_metadata(lengths, chunk_size, index_dtype=torch.int64, device="cpu"):
    """cu_seqlens, cu_chunk_seqlens, seq_idx, last_chunk_indices of a packed
    batch: every sequence is cut into chunks of chunk_size tokens (its last one
    shorter), as the pages' caller does."""
    cu, cuc, seq, last = [0], [0], [], []
    for b, L in enumerate(lengths):
        start, pos = cu[-1], 0
        while pos < L:
            n = min(chunk_size, L - pos)
            pos += n
            cuc.append(start + pos)
            seq.append(b)
        last.append(len(seq) - 1)
        cu.append(start + L)
    return [torch.tensor(v, dtype=index_dtype, device=device) for v in (cu, cuc, seq, last)]


def ssd_case(*, lengths, heads, headdim, dstate, groups, chunk_size=256,
             io_dtype=torch.bfloat16, init_dtype=torch.float32, with_init=True, with_z=True,
             D_per_dim=False, index_dtype=torch.int64, seed=0, device="cpu",
             name="ssd") -> SSDCase:
    """Seeded SSD prefill inputs: the decode distributions (x, z, B, C ~N(0, 1),
    dt ~N(0, 1), dt_bias U[-4, -1], A = -exp(U[0, ln 16]), D U[0, 1]),
    initial states ~N(0, 0.1^2)."""
    g = _gen(seed, device)
    T = int(sum(lengths))
    x = _normal((T, heads, headdim), 1.0, io_dtype, g, device)
    dt = _normal((T, heads), 1.0, torch.float32, g, device)
    A, D, dt_bias = _head_params(heads, g, device)
    if D_per_dim:
        D = _uniform((heads, headdim), 0.0, 1.0, g, device)
    B = _normal((T, groups, dstate), 1.0, io_dtype, g, device)
    C = _normal((T, groups, dstate), 1.0, io_dtype, g, device)
    z = _normal((T, heads, headdim), 1.0, io_dtype, g, device) if with_z else None
    init = (_normal((len(lengths), heads, headdim, dstate), 0.1, init_dtype, g, device)
            if with_init else None)
    cu, cuc, seq, last = chunk_metadata(lengths, chunk_size, index_dtype, device)
    return SSDCase(name=name, x=x, dt=dt, A=A, B=B, C=C, D=D, z=z, dt_bias=dt_bias,
                   chunk_size=chunk_size, cu_seqlens=cu, cu_chunk_seqlens=cuc,
                   last_chunk_indices=last, seq_idx=seq, initial_states=init)


def ssd_prefill(seed=0, device="cpu") -> SSDCase:
    """Packed SSD prefill shaped like the Mamba2-2.7B layer: 16 sequences of
    U{256..2048} tokens (seeded), 80 heads, headdim 64, dstate 128, 1 group,
    chunks of 256 tokens, bf16 x / B / C / z, fp32 initial states."""
    g = torch.Generator().manual_seed(1000 + seed)
    lengths = torch.randint(256, 2049, (16,), generator=g).tolist()
    return ssd_case(lengths=lengths, heads=80, headdim=64, dstate=128, groups=1,
                    chunk_size=256, seed=seed, device=device, name="ssd-prefill-2.7b")


# ---------------------------------------------------------------------------
# selecting sequences of a case (no arithmetic: rows, slots and tables only)
# ---------------------------------------------------------------------------

def _slot_list(t):
    return t.reshape(-1).tolist() if t is not None else []


def sequence_rows(case, seqs):
    """(packed rows, lengths) of the sequences `seqs` of a case."""
    if case.kind == "single":
        return list(seqs), [1] * len(seqs)
    if case.cu_seqlens is not None:
        cu = case.cu_seqlens.cpu().long().tolist()
    else:
        cu = [s * case.dense_steps for s in range(case.nseqs + 1)]
    rows, lens = [], []
    for s in seqs:
        rows += list(range(cu[s], cu[s + 1]))
        lens.append(cu[s + 1] - cu[s])
    return rows, lens


def subset_case(case, seqs):
    """A compact CPU case of the sequences `seqs` of `case` (any device): their
    rows, and their read / write slots copied into a small pool and renumbered.
    Returns (case, rows, slot map old -> new).  Trackers are dropped."""
    pad = case.pad_slot_id
    slots_total = case.state.shape[0]
    sbi = case.state_batch_indices.cpu() if case.state_batch_indices is not None else None
    dsbi = (case.dst_state_batch_indices.cpu()
            if case.dst_state_batch_indices is not None else None)
    rows, lens = sequence_rows(case, seqs)
    sel = torch.tensor(list(seqs), dtype=torch.long)
    sub_sbi = sbi[sel] if sbi is not None else None
    sub_dsbi = dsbi[sel] if dsbi is not None else None
    if sbi is None:   # no read table: sequence s uses slot s
        used_ids = list(seqs)
    else:
        used_ids = _slot_list(sub_sbi) + _slot_list(sub_dsbi)
    used = sorted({v for v in used_ids if v != pad and 0 <= v < slots_total})
    remap = {old: new for new, old in enumerate(used)}

    def mapped(t):
        if t is None:
            return None
        return t.clone().apply_(lambda v: remap.get(v, pad)).to(t.dtype)

    dev = case.state.device
    if used:
        pool = case.state[torch.tensor(used, dtype=torch.long, device=dev)].cpu().contiguous()
    else:   # a one-slot pool keeps the state tensor valid
        pool = torch.zeros((1, *case.state.shape[1:]), dtype=case.state.dtype)
    rws = torch.tensor(rows, dtype=torch.long, device=case.x.device)
    pick = (lambda t: None if t is None else t[rws].cpu())
    sub = dataclasses.replace(
        case, state=pool, x=pick(case.x), dt=pick(case.dt), B=pick(case.B), C=pick(case.C),
        z=pick(case.z), A=case.A.cpu(), D=None if case.D is None else case.D.cpu(),
        dt_bias=None if case.dt_bias is None else case.dt_bias.cpu(),
        state_batch_indices=mapped(sub_sbi) if sbi is not None else torch.tensor(
            [remap.get(s, pad) for s in seqs], dtype=torch.int64),
        dst_state_batch_indices=mapped(sub_dsbi), nseqs=len(seqs), ring_start=None,
        prev_num_accepted=None, prev_query_len=None)
    if case.kind == "varlen":
        cu_new = [0]
        for n in lens:
            cu_new.append(cu_new[-1] + n)
        sub.cu_seqlens = torch.tensor(cu_new, dtype=torch.int64)
        sub.dense_steps = 1
        sub.num_accepted_tokens = (None if case.num_accepted_tokens is None
                                   else case.num_accepted_tokens.cpu()[sel])
    return sub, rows, remap
