"""Pins of the ReplaySSM oracle (oracle.replay_update / oracle.replay_state).

The pages ("vllm.model_executor.layers.mamba.ops.ssu_dispatch":
selective_state_update_replayssm_flashinfer, the tracker kernels and the
commit_replayssm_ring_trackers docstring) fix the ring and where the trackers
move it, not the replay arithmetic.  Whatever the reading, a checkpointing
update must agree with the plain recurrence over the same token stream: with
an fp64 state pool (storing is then exact) every y and every logical state of
a replayed stream must equal the plain chain's BIT FOR BIT, one-token decode
with the tracker update after every token and speculative (MTP) passes with
the commit of the previous pass's accepted prefix alike.  Further pins: the
checkpoint is written exactly when k + L exceeds the window, new tokens land
at the ring positions the trackers name, the trackers follow the pinned update
rule, and sequences that cannot be replayed write nothing.
"""
from __future__ import annotations

import pytest
import torch

from mamba2_ssm_decode_gb300 import workloads as W

F64 = torch.float64


def _inputs(nseq, T, H=4, P=6, N=8, G=2, seed=0, io=torch.bfloat16):
    """Dense token streams: sequence i owns rows [i T, (i + 1) T)."""
    c = W.varlen_case(nseqs=nseq, max_len=T, fixed_len=T, heads=H, headdim=P, dstate=N,
                      groups=G, slots=2 * nseq * T, state_dtype=torch.float32, io_dtype=io,
                      same_tables=True, seed=seed)
    return c


def _caches(slots, H, P, N, G, R, io=torch.bfloat16):
    """Ring caches filled with NaN: a replay that reads a position nobody wrote
    turns its outputs into NaN."""
    xc = torch.full((slots, H, R, P), float("nan"), dtype=io)
    Bc = torch.full((slots, G, R, N), float("nan"), dtype=io)
    dc = torch.full((slots, H, R), float("nan"), dtype=torch.float32)
    return xc, Bc, dc


def _plain_chain(o, c, state0, seq_slots, rows_per_seq):
    """y of the plain chain over each sequence's rows (no state written) and the
    chain state after every row (an fp64 pool, one write slot per row)."""
    S = len(seq_slots)
    T = rows_per_seq
    slots = state0.shape[0]
    pool = torch.cat([state0, torch.zeros((S * T, *state0.shape[1:]), dtype=F64)])
    src = torch.tensor([[s] for s in seq_slots], dtype=torch.int64)
    dst = torch.arange(slots, slots + S * T, dtype=torch.int64).reshape(S, T)
    cu = torch.arange(0, (S + 1) * T, T, dtype=torch.int64)
    y = o.ssu_update_varlen(pool, c.x, c.dt, c.A, c.B, c.C, D=c.D, z=c.z, dt_bias=c.dt_bias,
                            dt_softplus=True, cu_seqlens=cu, state_batch_indices=src,
                            dst_state_batch_indices=dst)
    return y, pool[slots:].reshape(S, T, *state0.shape[1:])


# --------------------------------------------------------------------------
# one-token decode: update rule after every token
# --------------------------------------------------------------------------

@pytest.mark.parametrize("W_,R", [(1, 2), (1, 3), (2, 3), (2, 5), (3, 4), (3, 7), (4, 5),
                                  (4, 8), (5, 6), (5, 11)])
def test_one_token_replay_is_the_plain_chain_bit_for_bit(oracle_mod, W_, R):
    o = oracle_mod
    T, H, P, N, G = 23, 4, 6, 8, 2
    seq_slots = [2, 0]
    c = _inputs(len(seq_slots), T, H, P, N, G, seed=10 * W_ + R)
    g = torch.Generator().manual_seed(R)
    state0 = torch.randn((3, H, P, N), generator=g, dtype=F64) * 0.1
    y_ref, chain = _plain_chain(o, c, state0, seq_slots, T)
    state = state0.clone()
    xc, Bc, dc = _caches(3, H, P, N, G, R)
    rs = torch.zeros(3, dtype=torch.int32)
    pna = torch.zeros(3, dtype=torch.int32)
    sbi = torch.tensor(seq_slots, dtype=torch.int64)
    checkpoints = 0
    for t in range(T):
        rows = torch.tensor([i * T + t for i in range(len(seq_slots))])
        k_before = pna.clone()
        before = state.clone()
        y = o.replay_update(state, c.x[rows], c.dt[rows], c.A, c.B[rows], c.C[rows], xc, Bc, dc,
                            rs, pna, W_, D=c.D, z=c.z[rows], dt_bias=c.dt_bias, dt_softplus=True,
                            state_batch_indices=sbi, update_trackers=True)
        for i, slot in enumerate(seq_slots):
            assert torch.equal(y[i], y_ref[i * T + t]), f"y differs at token {t} of seq {i}"
            # the logical state after this token is the chain state after t + 1 tokens
            ls = o.replay_state(state, slot, c.A, xc, Bc, dc, rs, pna, dt_bias=c.dt_bias,
                                dt_softplus=True)
            assert torch.equal(ls, chain[i, t]), f"logical state differs after token {t}"
            # a checkpoint is written exactly when k + 1 exceeds the window
            must = int(k_before[slot]) + 1 > W_
            changed = not torch.equal(state[slot], before[slot])
            assert changed == must
            checkpoints += must
            assert int(pna[slot]) <= W_
        assert torch.equal(state[1], before[1])   # slot no sequence uses
    assert checkpoints >= 2 * ((T - 1) // W_) - 2


# --------------------------------------------------------------------------
# speculative passes: commit of the accepted prefix, then the pass
# --------------------------------------------------------------------------

@pytest.mark.parametrize("W_,R,Lmax", [(4, 8, 4), (2, 8, 4), (3, 5, 2), (1, 6, 3), (5, 10, 5),
                                       (3, 12, 6)])
def test_mtp_passes_with_commit_follow_the_accepted_chain(oracle_mod, W_, R, Lmax):
    """Each pass: ssu_ring_commit with the previous pass's acceptance count,
    then the checkpointing update of this pass's L rows without the tracker
    update.  Row t of a pass must equal the plain chain over every accepted
    token so far followed by rows 0..t of the pass, bit for bit.  (After a
    commit k <= max(W, Lmax), so a ring of max(W, Lmax) + Lmax positions holds
    every pass.)"""
    o = oracle_mod
    assert R >= max(W_, Lmax) + Lmax
    H, P, N, G = 4, 6, 8, 2
    passes = 14
    seq_slots = [1, 3, 0]
    S = len(seq_slots)
    g = torch.Generator().manual_seed(100 * W_ + R)
    lens = torch.randint(1, Lmax + 1, (passes, S), generator=g)
    acc = (torch.rand((passes, S), generator=g) * lens).floor().long() + 1   # U{1..L}
    total = int(lens.sum())
    c = _inputs(1, total, H, P, N, G, seed=W_ + R)   # a pool of rows, dealt out in order
    state0 = torch.randn((4, H, P, N), generator=g, dtype=F64) * 0.1
    state = state0.clone()
    truth = state0.clone()            # the chain over accepted tokens only
    xc, Bc, dc = _caches(4, H, P, N, G, R)
    rs = torch.zeros(4, dtype=torch.int32)
    pna = torch.zeros(4, dtype=torch.int32)
    pql = torch.zeros(4, dtype=torch.int32)
    sbi = torch.tensor(seq_slots, dtype=torch.int64)
    next_row = 0
    prev_acc = torch.zeros(S, dtype=torch.int64)
    for q in range(passes):
        L = lens[q]
        cu = torch.zeros(S + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(L, 0)
        rows = torch.arange(next_row, next_row + int(cu[-1]))
        next_row += int(cu[-1])
        o.ring_commit(rs, pna, pql, sbi, prev_acc, cu, W_, R)
        for i, slot in enumerate(seq_slots):   # the committed logical state is the truth
            ls = o.replay_state(state, slot, c.A, xc, Bc, dc, rs, pna, dt_bias=c.dt_bias,
                                dt_softplus=True)
            assert torch.equal(ls, truth[slot]), f"pass {q}: committed state of seq {i}"
        k_before = pna.clone()
        assert int(k_before.max()) <= max(W_, Lmax)
        before = state.clone()
        y = o.replay_update(state, c.x[rows], c.dt[rows], c.A, c.B[rows], c.C[rows], xc, Bc, dc,
                            rs, pna, W_, D=c.D, z=c.z[rows], dt_bias=c.dt_bias,
                            dt_softplus=True, cu_seqlens=cu, state_batch_indices=sbi,
                            update_trackers=False)
        # reference: the plain chain from the truth over this pass's rows
        tsel = torch.tensor([[s] for s in seq_slots])
        t2 = truth.clone()
        y_ref = o.ssu_update_varlen(t2, c.x[rows], c.dt[rows], c.A, c.B[rows], c.C[rows],
                                    D=c.D, z=c.z[rows], dt_bias=c.dt_bias, dt_softplus=True,
                                    cu_seqlens=cu, state_batch_indices=tsel,
                                    disable_state_update=True)
        assert torch.equal(y, y_ref), f"pass {q}: y differs from the accepted chain"
        for i, slot in enumerate(seq_slots):
            must = int(k_before[slot]) + int(L[i]) > W_
            assert (not torch.equal(state[slot], before[slot])) == (must and k_before[slot] > 0)
        # advance the truth by the accepted prefix of this pass
        a = acc[q]
        keep = torch.cat([torch.arange(int(cu[i]), int(cu[i]) + int(a[i])) for i in range(S)])
        cu_a = torch.zeros(S + 1, dtype=torch.int64)
        cu_a[1:] = torch.cumsum(a, 0)
        r_keep = rows[keep]
        # the chain's last accepted step goes back to the slot, no other step is stored
        dst = torch.full((S, Lmax), -1, dtype=torch.int64)
        for i, slot in enumerate(seq_slots):
            dst[i, int(a[i]) - 1] = slot
        o.ssu_update_varlen(truth, c.x[r_keep], c.dt[r_keep], c.A, c.B[r_keep], c.C[r_keep],
                            D=c.D, z=c.z[r_keep], dt_bias=c.dt_bias, dt_softplus=True,
                            cu_seqlens=cu_a, state_batch_indices=tsel,
                            dst_state_batch_indices=dst)
        prev_acc = a


# --------------------------------------------------------------------------
# one call in detail
# --------------------------------------------------------------------------

def _one_call(o, k, start, L, W_, R, seed=0, pad_slot=False, io=torch.bfloat16,
              state_dtype=F64, update_trackers=True):
    H, P, N, G = 4, 6, 8, 2
    c = _inputs(1, L, H, P, N, G, seed=seed, io=io)
    g = torch.Generator().manual_seed(seed + 1)
    slots = 5
    state = (torch.randn((slots, H, P, N), generator=g, dtype=F64) * 0.1).to(state_dtype)
    xc = torch.randn((slots, H, R, P), generator=g).to(io)
    Bc = torch.randn((slots, G, R, N), generator=g).to(io)
    dc = torch.randn((slots, H, R), generator=g)
    rs = torch.full((slots,), start, dtype=torch.int32)
    pna = torch.full((slots,), k, dtype=torch.int32)
    slot = -1 if pad_slot else 3
    return dict(c=c, state=state, xc=xc, Bc=Bc, dc=dc, rs=rs, pna=pna, slot=slot,
                cu=torch.tensor([0, L]), W_=W_, R=R, update_trackers=update_trackers)


def _run(o, d):
    c = d["c"]
    return o.replay_update(d["state"], c.x, c.dt, c.A, c.B, c.C, d["xc"], d["Bc"], d["dc"],
                           d["rs"], d["pna"], d["W_"], D=c.D, z=c.z, dt_bias=c.dt_bias,
                           dt_softplus=True, cu_seqlens=d["cu"],
                           state_batch_indices=torch.tensor([d["slot"]]),
                           update_trackers=d["update_trackers"])


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(
        torch.int32 if t.element_size() == 4 else torch.int64)


@pytest.mark.parametrize("k,start,L", [(0, 0, 1), (3, 5, 2), (5, 6, 3), (2, 7, 1), (4, 1, 4)])
def test_new_tokens_land_where_the_trackers_point(oracle_mod, k, start, L):
    o = oracle_mod
    d = _one_call(o, k, start, L, W_=4, R=8, seed=k + start)
    before = {n: d[n].clone() for n in ("xc", "Bc", "dc")}
    _run(o, d)
    c, s = d["c"], d["slot"]
    written = {(start + k + t) % 8: t for t in range(L)}
    for pos in range(8):
        for n in ("xc", "Bc", "dc"):
            new, old = d[n][s, :, pos], before[n][s, :, pos]
            if pos in written:
                t = written[pos]
                src = {"xc": c.x[t], "Bc": c.B[t], "dc": c.dt[t]}[n]
                assert torch.equal(_bits(new.contiguous()), _bits(src.contiguous())), (n, pos)
            else:
                assert torch.equal(_bits(new.contiguous()), _bits(old.contiguous())), (n, pos)
        for n in ("xc", "Bc", "dc"):   # other slots' rings untouched
            other = [i for i in range(5) if i != s]
            assert torch.equal(_bits(d[n][other]), _bits(before[n][other]))


@pytest.mark.parametrize("k,L,W_", [(0, 1, 1), (0, 2, 1), (1, 1, 1), (3, 1, 4), (4, 1, 4),
                                    (2, 3, 4), (2, 2, 4), (5, 3, 6)])
def test_checkpoint_is_the_state_after_the_replayed_tokens(oracle_mod, k, L, W_):
    o = oracle_mod
    d = _one_call(o, k, 2, L, W_=W_, R=8, seed=7 * k + L)
    s = d["slot"]
    c = d["c"]
    expect = o.replay_state(d["state"], s, c.A, d["xc"], d["Bc"], d["dc"], d["rs"], d["pna"],
                            dt_bias=c.dt_bias, dt_softplus=True)
    before = d["state"].clone()
    _run(o, d)
    if k + L > W_:
        assert torch.equal(d["state"][s], expect)
    else:
        assert torch.equal(d["state"][s], before[s])
    others = [i for i in range(5) if i != s]
    assert torch.equal(d["state"][others], before[others])


@pytest.mark.parametrize("k,start,L", [(0, 0, 1), (3, 5, 1), (4, 7, 1), (1, 2, 3)])
def test_update_trackers_apply_the_pinned_update_rule(oracle_mod, k, start, L):
    o = oracle_mod
    d = _one_call(o, k, start, L, W_=4, R=8, seed=3)
    rs_ref, pna_ref = d["rs"].clone(), d["pna"].clone()
    o.ring_update(rs_ref, pna_ref, torch.zeros(5, dtype=torch.int32), torch.tensor([3]), 4, 8)
    _run(o, d)
    assert torch.equal(d["rs"], rs_ref) and torch.equal(d["pna"], pna_ref)


@pytest.mark.parametrize("why", ["pad_slot", "ring_overflow", "start_out_of_range",
                                 "negative_count", "slot_beyond_trackers"])
def test_sequences_that_cannot_replay_write_nothing(oracle_mod, why):
    """A pad slot, a ring that cannot hold k + L tokens, a ring start outside
    [0, R), a negative count or a slot beyond the trackers: the rows run from
    a zero state (like a padded plain call) and nothing is written."""
    o = oracle_mod
    k, start, L = 2, 1, 3
    if why == "ring_overflow":
        k = 6
    if why == "negative_count":
        k = -1
    if why == "start_out_of_range":
        start = 8
    d = _one_call(o, k, start, L, W_=1, R=8, seed=11, pad_slot=why == "pad_slot")
    if why == "slot_beyond_trackers":
        d["rs"], d["pna"] = d["rs"][:3].clone(), d["pna"][:3].clone()   # slot 3 has none
    keep = {n: d[n].clone() for n in ("state", "xc", "Bc", "dc", "rs", "pna")}
    y = _run(o, d)
    for n, v in keep.items():
        assert torch.equal(_bits(d[n]), _bits(v)), f"{n} was written"
    c = d["c"]
    zero = torch.zeros((1, *d["state"].shape[1:]), dtype=F64)
    y_ref = o.ssu_update_varlen(zero, c.x, c.dt, c.A, c.B, c.C, D=c.D, z=c.z,
                                dt_bias=c.dt_bias, dt_softplus=True, cu_seqlens=d["cu"],
                                state_batch_indices=torch.tensor([[-1]]))
    assert torch.equal(y, y_ref)


@pytest.mark.parametrize("sdt,tol", [(torch.float32, 1e-5), (torch.bfloat16, 2e-2)])
def test_stored_checkpoints_round_once_per_checkpoint(oracle_mod, sdt, tol):
    """With an fp32 / bf16 pool only the checkpoints are rounded: the replayed
    stream stays within the state dtype's tolerance of the unrounded chain."""
    o = oracle_mod
    T, H, P, N, G, W_, R = 30, 4, 6, 8, 2, 3, 4
    c = _inputs(1, T, H, P, N, G, seed=5)
    g = torch.Generator().manual_seed(9)
    state0 = (torch.randn((1, H, P, N), generator=g, dtype=F64) * 0.1).to(sdt)
    y_ref, _ = _plain_chain(o, c, state0.to(F64), [0], T)
    state = state0.clone()
    xc, Bc, dc = _caches(1, H, P, N, G, R)
    rs = torch.zeros(1, dtype=torch.int32)
    pna = torch.zeros(1, dtype=torch.int32)
    worst = 0.0
    for t in range(T):
        y = o.replay_update(state, c.x[t:t + 1], c.dt[t:t + 1], c.A, c.B[t:t + 1], c.C[t:t + 1],
                            xc, Bc, dc, rs, pna, W_, D=c.D, z=c.z[t:t + 1], dt_bias=c.dt_bias,
                            dt_softplus=True, update_trackers=True)
        err = ((y[0] - y_ref[t]).abs() / (tol + tol * y_ref[t].abs())).max().item()
        worst = max(worst, err)
    assert worst <= 1.0
    if sdt == torch.bfloat16:
        assert worst > 1e-4   # the rounding is really there
