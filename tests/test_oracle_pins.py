"""Pins of the CPU oracle to things other than itself.

Each test ties an oracle function to a closed form, an invariant of the
recurrence, a library routine (numpy / scipy / torch CPU conversions) or a
brute-force search, so that a dropped term, a wrong sign, a wrong index or a
transposed operand in ssu_oracle.c fails at least one of them.

The recurrence (Mamba2 decode step; named on "vllm ... ssu_dispatch" and
"mate.mamba", stated in the oracle's header):
    dt' = softplus(dt + dt_bias); dA = exp(A dt'); h <- h dA + dt' x B;
    y = h.C + D x; y *= silu(z).
"""
from __future__ import annotations

import fractions
import math

import numpy as np
import pytest
import torch
from scipy.special import expit

from mamba2_ssm_decode_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

LN2 = 0.6931471805599453  # ln 2 to double precision


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def small_single(state_dtype=torch.float32, seed=1, **kw):
    args = dict(batch=5, heads=4, headdim=6, dstate=8, groups=2, slots=9,
                state_dtype=state_dtype, with_z=True, seed=seed)
    args.update(kw)
    return W.single_token_case(**args)


def small_varlen(state_dtype=torch.float32, seed=2, **kw):
    args = dict(nseqs=4, max_len=3, heads=4, headdim=6, dstate=8, groups=2, slots=40,
                state_dtype=state_dtype, with_z=True, seed=seed)
    args.update(kw)
    return W.varlen_case(**args)


def run_single(o, case, **over):
    kw = dict(D=case.D, z=case.z, dt_bias=case.dt_bias, dt_softplus=case.dt_softplus,
              state_batch_indices=case.state_batch_indices,
              dst_state_batch_indices=case.dst_state_batch_indices,
              pad_slot_id=case.pad_slot_id, disable_state_update=case.disable_state_update)
    kw.update(over)
    return o.ssu_update(case.state, case.x, case.dt, case.A, case.B, case.C, **kw)


def run_varlen(o, case, **over):
    kw = dict(D=case.D, z=case.z, dt_bias=case.dt_bias, dt_softplus=case.dt_softplus,
              cu_seqlens=case.cu_seqlens, nseqs=case.nseqs, dense_steps=case.dense_steps,
              num_accepted_tokens=case.num_accepted_tokens,
              state_batch_indices=case.state_batch_indices,
              dst_state_batch_indices=case.dst_state_batch_indices,
              pad_slot_id=case.pad_slot_id, disable_state_update=case.disable_state_update)
    kw.update(over)
    return o.ssu_update_varlen(case.state, case.x, case.dt, case.A, case.B, case.C, **kw)


def f64(t):
    return t.detach().to(torch.float64).numpy()


def group_of(H, G):
    return np.arange(H) // (H // G)


def softplus_np(v):
    return np.logaddexp(0.0, v)  # library routine: log(e^0 + e^v)


# --------------------------------------------------------------------------
# rounding and widening
# --------------------------------------------------------------------------

def _random_doubles(n, seed=0):
    rng = np.random.default_rng(seed)
    mant = rng.random(n) + 0.5
    exps = rng.integers(-150, 130, n)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    return sign * np.ldexp(mant, exps)


def test_round_f16_matches_numpy(oracle_mod):
    v = np.concatenate([_random_doubles(20000), np.ldexp(np.arange(1, 200) + 0.5, -24),
                        [65504.0, 65519.99, 65520.0, 1 + 2.0**-11, 1 + 3 * 2.0**-11, 0.0, -0.0]])
    v = v[np.abs(v) < 1e6]
    got = oracle_mod.round_to(torch.from_numpy(v), torch.float16).numpy()
    want = v.astype(np.float16)
    np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))


def test_round_f32_matches_numpy(oracle_mod):
    v = _random_doubles(20000, seed=3)
    got = oracle_mod.round_to(torch.from_numpy(v), torch.float32).numpy()
    np.testing.assert_array_equal(got.view(np.uint32), v.astype(np.float32).view(np.uint32))


def test_round_bf16_matches_torch_on_fp32_values(oracle_mod):
    # every fp32 value rounds once to bf16; torch's fp32 -> bf16 conversion is RNE
    v32 = _random_doubles(20000, seed=4).astype(np.float32)
    v32 = v32[np.isfinite(v32)]
    got = oracle_mod.round_to(torch.from_numpy(v32.astype(np.float64)), torch.bfloat16)
    want = torch.from_numpy(v32).to(torch.bfloat16)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def _bf16_values_near(v):
    """All bf16 values adjacent to v (brute force over the bit patterns around it)."""
    t = torch.tensor([v], dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
    b = int(t.view(torch.int16).item()) & 0xFFFF
    out = []
    for d in range(-2, 3):
        bb = (b + d) & 0xFFFF
        val = torch.tensor([bb], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
        f = float(val.to(torch.float64).item())
        if math.isfinite(f):
            out.append((f, bb))
    return out


def test_round_bf16_brute_force_on_doubles(oracle_mod):
    # doubles that are not fp32 values: nearest bf16 by exact rational comparison
    rng = np.random.default_rng(5)
    vals = list(_random_doubles(3000, seed=6)) + [1 + 2.0**-8, 1 + 3 * 2.0**-8,
                                                     1 + 2.0**-8 + 2.0**-40, -(1 + 2.0**-8)]
    for v in vals:
        if abs(v) > 3e38 or abs(v) < 1e-37:
            continue
        cands = _bf16_values_near(v)
        fv = fractions.Fraction(v)
        best = min(cands, key=lambda c: (abs(fractions.Fraction(c[0]) - fv), c[1] & 1))
        got = oracle_mod.round_scalar(v, torch.bfloat16)
        assert got == best[0], (v, got, best)
    del rng


def test_round_bf16_edges(oracle_mod):
    r = lambda v: oracle_mod.round_scalar(v, torch.bfloat16)  # noqa: E731
    bmax = (2 - 2.0**-7) * 2.0**127
    assert r(1 + 2.0**-8) == 1.0                      # tie -> even
    assert r(1 + 3 * 2.0**-8) == 1 + 2.0**-6          # tie -> even (up)
    assert r(bmax * (1 + 2.0**-10)) == bmax           # below half an ulp above max
    assert math.isinf(r(2.0**128))                    # overflow
    assert r(2.0**-134) == 0.0                        # half the smallest subnormal: tie -> 0
    assert r(3 * 2.0**-134) == 2.0**-132              # subnormal tie -> even


def test_widen_is_exact(oracle_mod):
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    for dt in (torch.bfloat16, torch.float16):
        vals = bits.view(dt)
        got = oracle_mod.widen(vals).numpy()
        want = vals.to(torch.float64).numpy()
        finite = np.isfinite(want)
        np.testing.assert_array_equal(got[finite], want[finite])
        assert np.all(np.isnan(got[np.isnan(want)]))


# --------------------------------------------------------------------------
# the recurrence: closed forms and invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("sdt", [torch.float32, torch.bfloat16, torch.float16])
def test_dt_zero_leaves_state_and_y_is_h_dot_C(oracle_mod, sdt):
    """dt = 0, no bias, no softplus: dA = 1 and the input term vanishes, so the
    state is unchanged bit for bit and y = h0 . C + D x (times silu z)."""
    case = small_single(sdt)
    case.dt.zero_()
    before = case.state.clone()
    y = run_single(oracle_mod, case, dt_bias=None, dt_softplus=False)
    assert torch.equal(case.state.view(torch.uint8), before.view(torch.uint8))
    slots, H, P, N, G = case.dims
    h0 = f64(before)[case.state_batch_indices.long().numpy()]           # [b, H, P, N]
    Cg = f64(case.C)[:, group_of(H, G), :]                                # [b, H, N]
    want = np.einsum("bhpn,bhn->bhp", h0, Cg) + f64(case.D)[None, :, None] * f64(case.x)
    want = want * f64(case.z) * expit(f64(case.z))
    np.testing.assert_allclose(y.numpy(), want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("A_val,factor", [(-1.0, 0.5), (-2.0, 0.25), (-3.0, 0.125)])
def test_B_zero_decays_by_power_of_two(oracle_mod, A_val, factor):
    """dt = -dt_bias with softplus gives dt' = softplus(0) = ln 2, so
    dA = exp(A ln 2) = 2^A; with B = 0 the fp32 state scales by exactly 2^A."""
    case = small_single(torch.float32)
    case.B.zero_()
    case.A.fill_(A_val)
    case.dt.copy_(-case.dt_bias[None, :].expand_as(case.dt))
    before = case.state.clone()
    run_single(oracle_mod, case)
    idx = case.state_batch_indices.long()
    assert torch.equal(case.state[idx], before[idx] * factor)
    untouched = torch.ones(case.state.shape[0], dtype=torch.bool)
    untouched[idx] = False
    assert torch.equal(case.state[untouched], before[untouched])


@pytest.mark.parametrize("arg,sp", [(0.0, LN2), (30.0, 30.000000000000092),
                                    (-30.0, 9.357622968840175e-14), (1.0, 1.3132616875182228)])
def test_softplus_values_through_the_step(oracle_mod, arg, sp):
    """Read dt' back through the step: B = 0, A = -1, D = 0, no z, one-hot C
    picks h'[p, n0] = h0[p, n0] exp(-dt') exactly in y (double)."""
    case = small_single(torch.float32, with_z=False)
    case.B.zero_()
    case.A.fill_(-1.0)
    case.D.zero_()
    case.C.zero_()
    case.C[:, :, 3] = 1.0
    case.dt.copy_(arg - case.dt_bias[None, :].expand_as(case.dt))
    h0 = f64(case.state)[case.state_batch_indices.long().numpy()][..., 3]
    y = run_single(oracle_mod, case).numpy()
    # dt + dt_bias is evaluated in double from the fp32 inputs: account exactly
    argd = f64(case.dt) + f64(case.dt_bias)[None, :]
    assert np.allclose(argd, arg, atol=1e-6)
    got_sp = -np.log(y / h0)
    # first-order correction for the fp32 representation of `arg`
    want = np.broadcast_to(sp + expit(arg) * (argd - arg)[:, :, None], got_sp.shape)
    np.testing.assert_allclose(got_sp, want, rtol=1e-9, atol=1e-15)


def test_zero_state_single_step_closed_form(oracle_mod):
    """From a zero state: h' = dt' x (outer) B, y = x (dt' B.C + D) silu(z).
    A does not enter at all."""
    case = small_single(torch.float32, dt_per_dim=True)
    case.state.zero_()
    case.A.fill_(-1e30)  # would blow up if A were (wrongly) applied to the input term
    y = run_single(oracle_mod, case).numpy()
    slots, H, P, N, G = case.dims
    dtp = softplus_np(f64(case.dt) + f64(case.dt_bias)[None, :, None])           # [b, H, P]
    Bg = f64(case.B)[:, group_of(H, G), :]
    Cg = f64(case.C)[:, group_of(H, G), :]
    x = f64(case.x)
    bc = np.einsum("bhn,bhn->bh", Bg, Cg)
    want = x * (dtp * bc[:, :, None] + f64(case.D)[None, :, None])
    want = want * f64(case.z) * expit(f64(case.z))
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)
    h_want = (dtp * x)[..., None] * Bg[:, :, None, :]                              # [b, H, P, N]
    idx = case.state_batch_indices.long().numpy()
    np.testing.assert_array_equal(f64(case.state)[idx], h_want.astype(np.float32))


def test_linear_in_state_and_input(oracle_mod):
    """For fixed dt, B, C, z: y(h0, x) = y(h0, 0) + y(0, x) (the step is linear)."""
    base = small_single(torch.float32, seed=11)

    def y_of(zero_state, zero_x):
        c = base.clone()
        if zero_state:
            c.state.zero_()
        if zero_x:
            c.x.zero_()
        return run_single(oracle_mod, c, disable_state_update=True).numpy()

    full, s_only, x_only = y_of(False, False), y_of(False, True), y_of(True, False)
    np.testing.assert_allclose(full, s_only + x_only, rtol=1e-12, atol=1e-12)


def _dual_form(case, s, rows, h0):
    """Unrolled (state-space dual) form of a chain over `rows` for every head:
    h_t = (prod_{u<=t} dA_u) h0 + sum_{j<=t} (prod_{j<u<=t} dA_u) dt'_j x_j (x) B_j."""
    slots, H, P, N, G = case.dims
    g = group_of(H, G)
    dt = f64(case.dt)
    if dt.ndim == 2:
        dt = np.repeat(dt[:, :, None], P, axis=2)
    dtp = softplus_np(dt + f64(case.dt_bias)[None, :, None])                  # [R, H, P]
    dA = np.exp(f64(case.A)[None, :, None] * dtp)
    X, Bg, Cg = f64(case.x), f64(case.B)[:, g, :], f64(case.C)[:, g, :]
    hs, ys = [], []
    for t_idx, r in enumerate(rows):
        decay_all = np.prod(dA[rows[: t_idx + 1]], axis=0)                    # [H, P]
        h = decay_all[..., None] * h0
        for j_idx in range(t_idx + 1):
            rj = rows[j_idx]
            later = rows[j_idx + 1: t_idx + 1]
            decay = np.prod(dA[later], axis=0) if later else np.ones((H, P))
            h = h + (decay * dtp[rj] * X[rj])[..., None] * Bg[rj][:, None, :]
        y = np.einsum("hpn,hn->hp", h, Cg[r]) + f64(case.D)[:, None] * X[r]
        y = y * f64(case.z)[r] * expit(f64(case.z)[r])
        hs.append(h)
        ys.append(y)
    return hs, ys


def test_chain_matches_unrolled_dual_form(oracle_mod):
    """A multi-token chain equals the unrolled sum form of the linear recurrence."""
    case = small_varlen(torch.float32, seed=21, dt_per_dim=True)
    before = case.state.clone()
    y = run_varlen(oracle_mod, case).numpy()
    cu = case.cu_seqlens.long().tolist()
    na = case.num_accepted_tokens.long().tolist()
    sbi = case.state_batch_indices.long()
    dsbi = case.dst_state_batch_indices.long()
    for s in range(case.nseqs):
        rows = list(range(cu[s], cu[s + 1]))
        h0 = f64(before)[sbi[s, na[s] - 1]]
        hs, ys = _dual_form(case, s, rows, h0)
        for t, r in enumerate(rows):
            np.testing.assert_allclose(y[r], ys[t], rtol=1e-10, atol=1e-10)
            np.testing.assert_allclose(f64(case.state)[dsbi[s, t]], hs[t], rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("sdt,tol", [(torch.float32, 1e-6), (torch.bfloat16, 2e-2)])
def test_chain_equals_single_token_calls(oracle_mod, sdt, tol):
    """k chained steps == k one-token calls, each reading the previous write
    (exact up to the state rounding the single calls add between steps)."""
    case = small_varlen(sdt, seed=31)
    chain = case.clone()
    y_chain = run_varlen(oracle_mod, chain).numpy()
    single = case.clone()
    cu = case.cu_seqlens.long().tolist()
    na = case.num_accepted_tokens.long()
    sbi = case.state_batch_indices.long()
    dsbi = case.dst_state_batch_indices.long()
    for s in range(case.nseqs):
        src = int(sbi[s, na[s] - 1])
        for t, r in enumerate(range(cu[s], cu[s + 1])):
            dst = int(dsbi[s, t])
            sl = slice(r, r + 1)
            y1 = oracle_mod.ssu_update(
                single.state, case.x[sl], case.dt[sl], case.A, case.B[sl], case.C[sl],
                D=case.D, z=case.z[sl], dt_bias=case.dt_bias, dt_softplus=True,
                state_batch_indices=torch.tensor([src]), dst_state_batch_indices=torch.tensor([dst]))
            np.testing.assert_allclose(y1.numpy()[0], y_chain[r], rtol=tol, atol=tol)
            src = dst
    np.testing.assert_allclose(f64(single.state), f64(chain.state), rtol=tol, atol=tol)


def test_groups_broadcast(oracle_mod):
    """(a) G = H with B/C tiled equal is G = 1 bit for bit; (b) from a zero state
    with B nonzero in group g only, exactly heads [g*hr, (g+1)*hr) move: heads of
    a group are contiguous (g = h // (H / G))."""
    one = small_single(torch.float32, groups=1, heads=4)
    many = one.clone()
    many.B = one.B.expand(-1, 4, -1).contiguous()
    many.C = one.C.expand(-1, 4, -1).contiguous()
    y1 = run_single(oracle_mod, one)
    y4 = run_single(oracle_mod, many)
    assert torch.equal(y1, y4) and torch.equal(one.state, many.state)

    case = small_single(torch.float32, groups=2, heads=6, seed=5)
    case.state.zero_()
    case.D.zero_()
    case.B[:, 0, :] = 0.0   # only group 1 (heads 3, 4, 5) gets input
    y = run_single(oracle_mod, case).numpy()
    assert np.all(y[:, :3, :] == 0.0)
    assert np.all(np.abs(y[:, 3:, :]).sum(axis=(0, 2)) > 0)
    idx = case.state_batch_indices.long()
    st = case.state[idx]
    assert torch.all(st[:, :3] == 0) and torch.all(st[:, 3:].abs().sum(dim=(0, 2, 3)) > 0)


@pytest.mark.parametrize("pad", [-1, 0])
def test_pad_and_out_of_range_slots(oracle_mod, pad):
    """A pad or out-of-range read slot writes nothing and runs from a zero state;
    a pad write slot skips only the write; disable_state_update writes nothing."""
    case = small_single(torch.float32, slots=12, seed=7)
    sbi = torch.tensor([3, pad, 12, -5, 7], dtype=torch.int32)  # 12 and -5 are out of range
    case.state_batch_indices = sbi
    before = case.state.clone()
    y = run_single(oracle_mod, case, pad_slot_id=pad).numpy()
    changed = [i for i in range(12) if not torch.equal(case.state[i], before[i])]
    assert changed == [3, 7]
    zero = case.clone()
    zero.state = torch.zeros_like(case.state)
    zero.state_batch_indices = torch.tensor([1, 1, 1, 1, 1], dtype=torch.int32)
    y0 = run_single(oracle_mod, zero, pad_slot_id=pad, disable_state_update=True).numpy()
    np.testing.assert_array_equal(y[1:4], y0[1:4])

    # pad write slot
    c2 = small_single(torch.float32, slots=12, seed=8)
    c2.state_batch_indices = torch.tensor([1, 2, 3, 4, 5], dtype=torch.int32)
    c2.dst_state_batch_indices = torch.tensor([6, pad, 8, 12, 10], dtype=torch.int32)
    b2 = c2.state.clone()
    run_single(oracle_mod, c2, pad_slot_id=pad)
    changed = [i for i in range(12) if not torch.equal(c2.state[i], b2[i])]
    assert changed == [6, 8, 10]

    # pad read slot with a valid write slot: the sequence writes nothing
    c4 = small_single(torch.float32, slots=12, seed=10)
    c4.state_batch_indices = torch.tensor([1, pad, 3, 13, 5], dtype=torch.int32)
    c4.dst_state_batch_indices = torch.tensor([6, 7, 8, 9, 10], dtype=torch.int32)
    b4 = c4.state.clone()
    run_single(oracle_mod, c4, pad_slot_id=pad)
    changed = [i for i in range(12) if not torch.equal(c4.state[i], b4[i])]
    assert changed == [6, 8, 10]
    # the same for a packed call whose read entry is pad
    v = small_varlen(torch.float32, seed=12, nseqs=2, max_len=2, fixed_len=2)
    v.num_accepted_tokens = None
    v.state_batch_indices = torch.tensor([[pad, 30], [31, 32]], dtype=torch.int32)
    v.dst_state_batch_indices = torch.tensor([[20, 21], [22, 23]], dtype=torch.int32)
    bv = v.state.clone()
    run_varlen(oracle_mod, v, pad_slot_id=pad)
    changed = [i for i in range(v.state.shape[0]) if not torch.equal(v.state[i], bv[i])]
    assert changed == [22, 23]

    # disable_state_update
    c3 = small_single(torch.float32, slots=12, seed=9)
    ref = c3.clone()
    y_ref = run_single(oracle_mod, ref).numpy()
    b3 = c3.state.clone()
    y3 = run_single(oracle_mod, c3, disable_state_update=True).numpy()
    assert torch.equal(c3.state, b3)
    np.testing.assert_array_equal(y3, y_ref)


def test_acceptance_count_reads_the_state_after_that_many_tokens(oracle_mod):
    """Reading column num_accepted - 1 of the previous call's write table gives
    the state after exactly num_accepted tokens: a second call seeded that way
    equals one chain over the accepted prefix plus the new tokens."""
    c1 = small_varlen(torch.float32, seed=41, nseqs=3, max_len=3, fixed_len=3)
    c1.num_accepted_tokens = None
    c1.state_batch_indices = torch.tensor([[0, 30, 31], [1, 32, 33], [2, 34, 35]], dtype=torch.int32)
    c1.dst_state_batch_indices = torch.tensor([[10, 11, 12], [13, 14, 15], [16, 17, 18]],
                                              dtype=torch.int32)
    pool0 = c1.state.clone()
    run_varlen(oracle_mod, c1)
    accepted = [1, 3, 2]
    # second call: one new token per sequence, read slot from the write table
    c2 = c1.clone()
    c2.cu_seqlens = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    c2.x, c2.dt, c2.B, c2.C, c2.z = (t[:3].flip(0).contiguous() for t in (c1.x, c1.dt, c1.B, c1.C, c1.z))
    c2.num_accepted_tokens = torch.tensor(accepted, dtype=torch.int32)
    c2.state_batch_indices = c1.dst_state_batch_indices
    c2.dst_state_batch_indices = torch.tensor([[20], [21], [22]], dtype=torch.int32)
    y2 = run_varlen(oracle_mod, c2).numpy()
    # reference: one chain per sequence over its accepted rows then the new row
    for s in range(3):
        rows1 = list(range(3 * s, 3 * s + accepted[s]))
        ref = c1.clone()
        ref.state = pool0.clone()
        ref.x = torch.cat([c1.x[rows1], c2.x[s:s + 1]])
        ref.dt = torch.cat([c1.dt[rows1], c2.dt[s:s + 1]])
        ref.B = torch.cat([c1.B[rows1], c2.B[s:s + 1]])
        ref.C = torch.cat([c1.C[rows1], c2.C[s:s + 1]])
        ref.z = torch.cat([c1.z[rows1], c2.z[s:s + 1]])
        L = len(rows1) + 1
        ref.cu_seqlens = torch.tensor([0, L], dtype=torch.int32)
        ref.num_accepted_tokens = None
        ref.nseqs = 1
        ref.state_batch_indices = torch.tensor([[s]], dtype=torch.int32)
        ref.dst_state_batch_indices = torch.tensor([[36 + i for i in range(L)]], dtype=torch.int32)
        yr = run_varlen(oracle_mod, ref).numpy()
        np.testing.assert_allclose(y2[s], yr[L - 1], rtol=1e-6, atol=1e-6)


def test_dense_equals_packed_and_flat_equals_2d(oracle_mod):
    case = small_varlen(torch.float32, seed=51, fixed_len=3, dense=True, nseqs=4, max_len=3)
    packed = case.clone()
    packed.cu_seqlens = torch.arange(0, 15, 3, dtype=torch.int32)
    y_dense = run_varlen(oracle_mod, case)
    y_packed = run_varlen(oracle_mod, packed)
    assert torch.equal(y_dense, y_packed) and torch.equal(case.state, packed.state)

    one = small_varlen(torch.float32, seed=52, fixed_len=3, nseqs=1, max_len=3)
    flat = one.clone()
    flat.state_batch_indices = one.state_batch_indices.reshape(-1)
    flat.dst_state_batch_indices = one.dst_state_batch_indices.reshape(-1)
    y2 = run_varlen(oracle_mod, one)
    yf = run_varlen(oracle_mod, flat)
    assert torch.equal(y2, yf) and torch.equal(one.state, flat.state)


def test_empty_sequences_and_per_dim_dt(oracle_mod):
    case = small_varlen(torch.float32, seed=61, nseqs=2, max_len=2, fixed_len=2)
    case.cu_seqlens = torch.tensor([0, 0, 2], dtype=torch.int32)
    before = case.state.clone()
    y = run_varlen(oracle_mod, case)
    # rows 0-1 belong to sequence 1; rows 2-3 belong to no sequence and stay unwritten
    assert torch.isfinite(y[:2]).all() and torch.isnan(y[2:]).all()
    s0_dst = case.dst_state_batch_indices[0].long()
    assert torch.equal(case.state[s0_dst], before[s0_dst])
    s1_dst = case.dst_state_batch_indices[1].long()
    assert not torch.equal(case.state[s1_dst], before[s1_dst])

    a = small_single(torch.float32, seed=62)
    b = a.clone()
    b.dt = a.dt[:, :, None].expand(-1, -1, a.x.shape[2]).contiguous()
    assert torch.equal(run_single(oracle_mod, a), run_single(oracle_mod, b))
    assert torch.equal(a.state, b.state)


@pytest.mark.parametrize("sdt", [torch.bfloat16, torch.float16])
def test_low_precision_state_is_rounded_once(oracle_mod, sdt):
    """The stored bf16/fp16 state is the RNE rounding of the double h' (read in
    double through a one-hot C), checked with torch/numpy conversions."""
    case = small_single(sdt, with_z=False, seed=71)
    case.D.zero_()
    N = case.state.shape[3]
    ys = []
    for n in range(N):
        c = case.clone()
        c.C.zero_()
        c.C[:, :, n] = 1.0
        ys.append(run_single(oracle_mod, c, disable_state_update=True).numpy())
    h_new = np.stack(ys, axis=-1)                                   # [b, H, P, N] double
    run_single(oracle_mod, case)
    got = case.state[case.state_batch_indices.long()]
    if sdt == torch.float16:
        want = torch.from_numpy(h_new.astype(np.float16))
    else:
        # the oracle's double -> bf16 rounding is pinned by the brute-force test above
        want = oracle_mod.round_to(torch.from_numpy(h_new), torch.bfloat16)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))


# --------------------------------------------------------------------------
# per-(head, dim) A / D / dt_bias ("mate.mamba", _per_head's channel-wise form)
# --------------------------------------------------------------------------

def test_per_channel_params_equal_per_head_when_constant(oracle_mod):
    a = small_single(torch.float32, seed=81)
    b = a.clone()
    P_ = a.x.shape[2]
    b.A = a.A[:, None].expand(-1, P_).contiguous()
    b.D = a.D[:, None].expand(-1, P_).contiguous()
    b.dt_bias = a.dt_bias[:, None, None].expand(-1, P_, 8)   # [H, P, N] view, zero dstate stride
    ya, yb = run_single(oracle_mod, a), run_single(oracle_mod, b)
    assert torch.equal(ya, yb) and torch.equal(a.state, b.state)


def test_per_channel_decay_is_exact_power_of_two(oracle_mod):
    """dt = -dt_bias[h, p] with softplus: dt' = ln 2 for every channel, so with
    B = 0 row p of head h scales by exactly 2^A[h, p]."""
    case = small_single(torch.float32, seed=82)
    H, P_ = case.x.shape[1], case.x.shape[2]
    exps = -(1 + (torch.arange(H * P_) % 3)).reshape(H, P_).to(torch.float32)   # -1, -2, -3
    case.A = exps
    case.dt_bias = torch.linspace(-4, -1, H * P_).reshape(H, P_)
    case.dt = -case.dt_bias[None].expand(case.x.shape[0], -1, -1).contiguous()
    case.B.zero_()
    before = case.state.clone()
    run_single(oracle_mod, case)
    idx = case.state_batch_indices.long()
    want = before[idx] * torch.pow(2.0, exps)[None, :, :, None]
    assert torch.equal(case.state[idx], want)


def test_per_channel_zero_state_closed_form(oracle_mod):
    case = small_single(torch.float32, seed=83)
    H, P_ = case.x.shape[1], case.x.shape[2]
    g = torch.Generator().manual_seed(7)
    case.D = torch.rand(H, P_, generator=g)
    case.dt_bias = -1 - 3 * torch.rand(H, P_, generator=g)
    case.state.zero_()
    y = run_single(oracle_mod, case).numpy()
    slots, H, P_, N, G = case.dims
    dtp = softplus_np(f64(case.dt)[:, :, None] + f64(case.dt_bias)[None])      # [b, H, P]
    Bg = f64(case.B)[:, group_of(H, G), :]
    Cg = f64(case.C)[:, group_of(H, G), :]
    bc = np.einsum("bhn,bhn->bh", Bg, Cg)
    x = f64(case.x)
    want = x * (dtp * bc[:, :, None] + f64(case.D)[None]) * f64(case.z) * expit(f64(case.z))
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)
