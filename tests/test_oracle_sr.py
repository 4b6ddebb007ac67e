"""Pins of the oracle's stochastic rounding of 16-bit state.

"vllm.model_executor.layers.mamba.ops.ssu_dispatch" (FlashInferSSUBackend.__call__,
selective_state_update_replayssm_flashinfer) draws a random seed per call and
passes philox_rounds (default 10); the reading stated in ssu_oracle.c: the
random bits come from Philox4x64 keyed by the seed with the element's index
in the state pool as counter, and a value rounds up with probability equal to
its fractional position between the two neighbours of the format (16-bit
resolution).  Pinned here against numpy's Philox generator, exact counts over
every 16-bit random value, and the plain round-to-nearest path."""
from __future__ import annotations

import fractions
import math
import random

import numpy as np
import pytest
import torch

from mamba2_ssm_decode_gb300 import workloads as W

M64 = (1 << 64) - 1


# --------------------------------------------------------------------------
# the generator
# --------------------------------------------------------------------------

def numpy_block(counter, key):
    """numpy's Philox4x64-10 advances its counter by one, then emits the block
    of that counter: ask for counter - 1 (with the borrow) to get `counter`'s."""
    c = list(counter)
    i = 0
    while True:
        c[i] = (c[i] - 1) & M64
        if c[i] != M64 or i == 3:
            break
        i += 1
    gen = np.random.Philox(counter=np.array(c, dtype=np.uint64),
                           key=np.array(list(key), dtype=np.uint64))
    return [int(v) for v in gen.random_raw(4)]


@pytest.mark.parametrize("seed", range(12))
def test_philox_is_numpys_philox4x64_10(oracle_mod, seed):
    rng = random.Random(seed)
    counter = [rng.getrandbits(64) for _ in range(4)]
    if seed == 0:
        counter = [0, 0, 0, 0]
    if seed == 1:
        counter = [0, 1, 0, 0]                    # the low word borrows in numpy's view
    key = [rng.getrandbits(64), rng.getrandbits(64)]
    assert oracle_mod.philox4x64(counter, key, 10) == numpy_block(counter, key)


def test_philox_rounds_and_stream_layout(oracle_mod):
    o = oracle_mod
    c, k = [5, 0, 0, 0], [77, 0]
    assert o.philox4x64(c, k, 0) == c                      # no round: the counter itself
    assert o.philox4x64(c, k, 7) != o.philox4x64(c, k, 10)
    # element e uses bits 16 (e % 4) of word (e / 4) % 4 of block e / 16
    for e in (0, 1, 5, 15, 16, 17, 1000003):
        blk = o.philox4x64([e >> 4, 0, 0, 0], [77, 0], 10)
        want = (blk[(e >> 2) & 3] >> (16 * (e & 3))) & 0xFFFF
        assert o.sr_bits(77, e, 10) == want
    assert o.sr_bits(77, 3, 10) != o.sr_bits(78, 3, 10) or o.sr_bits(77, 4, 10) != o.sr_bits(78, 4, 10)


# --------------------------------------------------------------------------
# the rounding
# --------------------------------------------------------------------------

def neighbours(v, dtype):
    """(lo, hi): the format's values around v, lo <= v <= hi, from numpy / torch."""
    if dtype == torch.float16:
        x = np.float16(v)
        xv = float(x)
        if xv == v:
            return xv, xv
        if xv < v:
            return xv, float(np.nextafter(x, np.float16(np.inf)))
        return float(np.nextafter(x, np.float16(-np.inf))), xv
    x = torch.tensor([v], dtype=torch.float64).to(torch.bfloat16)
    xv = float(x)
    if xv == v:
        return xv, xv
    bits = x.view(torch.int16)
    step = 1 if (xv < v) == (xv >= 0) else -1             # away from / toward zero in bits
    other = float((bits + step).view(torch.bfloat16))
    return (xv, other) if xv < v else (other, xv)


def _values(dtype):
    rng = random.Random(3 if dtype == torch.float16 else 4)
    vals = [0.1, -0.3, 1.0 + 2.0**-12, 3.14159, -2.718281828, 1e-3, 123.456]
    vals += [rng.uniform(-8, 8) for _ in range(6)]
    if dtype == torch.float16:
        vals += [3e-6, -1.7e-7, 6.1e-5, 65000.0]           # fp16 subnormals, near the top
    else:
        vals += [1e-39, -3e-40, 3e38]                      # bf16 subnormals, near the top
    return vals


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_rounding_goes_up_for_exactly_frac_of_the_random_values(oracle_mod, dtype):
    """Over all 2^16 random values the result is always one of the two
    neighbours, and the one farther from zero comes out exactly
    floor(2^16 frac) times, frac = (|v| - near) / (far - near) the magnitude's
    position between them, in exact rationals."""
    for v in _values(dtype):
        lo, hi = neighbours(v, dtype)
        near, far = sorted((abs(lo), abs(hi)))
        frac = fractions.Fraction(abs(v)) - fractions.Fraction(near)
        frac /= (fractions.Fraction(far) - fractions.Fraction(near))
        ups = 0
        for r in range(0, 1 << 16):
            out = oracle_mod.sr_round(v, dtype, r)
            assert out in (lo, hi), (v, r, out, lo, hi)
            ups += abs(out) == far
        assert ups == math.floor(frac * (1 << 16)), (v, ups, float(frac))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_representable_values_and_specials_are_unchanged(oracle_mod, dtype):
    for v in (0.0, -0.0, 1.0, -2.5, 0.15625, 2.0**-14, 2.0**-24 if dtype == torch.float16
              else 2.0**-133, math.inf, -math.inf):
        for r in (0, 1, 0x7FFF, 0xFFFF):
            out = oracle_mod.sr_round(v, dtype, r)
            assert out == v and math.copysign(1, out) == math.copysign(1, v)
    assert math.isnan(oracle_mod.sr_round(math.nan, dtype, 5))


def test_rounding_past_the_largest_value_overflows(oracle_mod):
    top = 65504.0
    v = top + 16.0                                         # half an fp16 ulp above the top
    outs = {oracle_mod.sr_round(v, torch.float16, r) for r in (0, 0x7FFF, 0x8000, 0xFFFF)}
    assert outs == {top, math.inf}


# --------------------------------------------------------------------------
# the state writes of the calls
# --------------------------------------------------------------------------

def _case(sdt, kind="single", seed=5):
    if kind == "single":
        return W.single_token_case(batch=5, heads=4, headdim=6, dstate=8, groups=2, slots=9,
                                   state_dtype=sdt, pad_frac=0.2, seed=seed)
    return W.varlen_case(nseqs=4, max_len=3, heads=4, headdim=6, dstate=8, groups=2, slots=40,
                         state_dtype=sdt, seed=seed)


def _run(o, c, **kw):
    args = dict(D=c.D, z=c.z, dt_bias=c.dt_bias, dt_softplus=True,
                state_batch_indices=c.state_batch_indices,
                dst_state_batch_indices=c.dst_state_batch_indices, pad_slot_id=c.pad_slot_id)
    args.update(kw)
    if c.kind == "single":
        return o.ssu_update(c.state, c.x, c.dt, c.A, c.B, c.C, **args)
    return o.ssu_update_varlen(c.state, c.x, c.dt, c.A, c.B, c.C, cu_seqlens=c.cu_seqlens,
                               num_accepted_tokens=c.num_accepted_tokens, **args)


@pytest.mark.parametrize("kind", ["single", "varlen"])
@pytest.mark.parametrize("sdt", [torch.bfloat16, torch.float16])
def test_each_stored_element_is_the_stochastic_rounding_of_the_exact_state(oracle_mod, sdt,
                                                                            kind):
    """The same call on an fp64 pool (stores exact) gives each element's
    unrounded value; the 16-bit call must store sr_round(value, bits of its
    index) in every written element and leave the rest alone."""
    o = oracle_mod
    c = _case(sdt, kind)
    before = c.state.clone()
    exact = c.clone()
    exact.state = c.state.to(torch.float64)
    _run(o, exact)
    seed, rounds = 0x1234_5678_9ABC, 10
    _run(o, c, rand_seed=seed, philox_rounds=rounds)
    flat_exact = exact.state.reshape(-1)
    flat_new = c.state.reshape(-1)
    flat_before = before.reshape(-1)
    changed = (flat_exact != flat_before.double()).nonzero().flatten().tolist()
    assert len(changed) > 100
    for e in changed:
        want = o.sr_round(float(flat_exact[e]), sdt, o.sr_bits(seed, e, rounds))
        assert float(flat_new[e]) == want, e
    untouched = torch.ones(flat_new.numel(), dtype=torch.bool)
    untouched[changed] = False
    bits = torch.int16
    assert torch.equal(flat_new[untouched].view(bits), flat_before[untouched].view(bits))


def test_seeds_decide_and_fp32_state_ignores_them(oracle_mod):
    o = oracle_mod
    base = _case(torch.bfloat16)
    a, b, c, rne = base.clone(), base.clone(), base.clone(), base.clone()
    _run(o, a, rand_seed=11)
    _run(o, b, rand_seed=11)
    _run(o, c, rand_seed=12)
    _run(o, rne)
    assert torch.equal(a.state, b.state)
    assert not torch.equal(a.state, c.state)
    # every stochastic result is within one bf16 ulp of the nearest-even one
    d = (a.state.double() - rne.state.double()).abs()
    ulp = rne.state.double().abs() * 2.0**-7 + 1e-40
    assert bool((d <= ulp).all())
    f = _case(torch.float32)
    g = f.clone()
    _run(o, f, rand_seed=99)
    _run(o, g)
    assert torch.equal(f.state, g.state)


def test_replay_checkpoints_round_stochastically_too(oracle_mod):
    o = oracle_mod
    c = W.replay_case(nseqs=6, heads=4, headdim=6, dstate=8, groups=2, slots=12,
                      state_dtype=torch.bfloat16, seed=9)
    exact = c.clone()
    exact.state = c.state.to(torch.float64)
    kw = lambda x: dict(D=x.D, z=x.z, dt_bias=x.dt_bias, dt_softplus=True,  # noqa: E731
                        state_batch_indices=x.state_batch_indices, update_trackers=True)
    o.replay_update(exact.state, c.x, c.dt, c.A, c.B, c.C, exact.x_cache, exact.B_cache,
                    exact.dt_cache, exact.ring_start, exact.prev_num_accepted,
                    c.logical_window, **kw(exact))
    before = c.state.clone()
    o.replay_update(c.state, c.x, c.dt, c.A, c.B, c.C, c.x_cache, c.B_cache, c.dt_cache,
                    c.ring_start, c.prev_num_accepted, c.logical_window, rand_seed=321,
                    **kw(c))
    flat_exact, flat_new = exact.state.reshape(-1), c.state.reshape(-1)
    changed = (flat_exact != before.reshape(-1).double()).nonzero().flatten().tolist()
    assert len(changed) > 50
    for e in changed:
        assert float(flat_new[e]) == o.sr_round(float(flat_exact[e]), torch.bfloat16,
                                                o.sr_bits(321, e, 10))
