"""GPU stochastic rounding of 16-bit state against the oracle.

Bit-exact: the kernels round their fp32 state.  The same call on an fp32 pool
stores those fp32 values exactly, so every element the 16-bit call with a seed
stores must be the oracle's stochastic rounding (ssu_oracle.c) of the fp32
value with the random bits of its index -- bit for bit, for every kernel that
stores state.  Against the fp64 oracle run with the same seed the call stays
within the 16-bit state tolerance, and untouched slots stay bit-identical."""
from __future__ import annotations

import pytest
import torch

import mamba2_ssm_decode_gb300 as ssu
from mamba2_ssm_decode_gb300 import workloads as W

from . import _parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"
SEED = 0x5EED_0F_C0FFEE


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssm_decode_gb300 import build
    build.build()


def _seed(v=SEED):
    return torch.tensor([v], dtype=torch.int64, device=DEV)


def _call(case, algorithm, rand_seed=None, rounds=10):
    kw = dict(D=case.D, z=case.z, dt_bias=case.dt_bias, dt_softplus=True,
              pad_slot_id=case.pad_slot_id, rand_seed=rand_seed, philox_rounds=rounds)
    if case.kind == "replay":
        return ssu.ssu_replay_update(case.state, case.x, case.dt, case.A, case.B, case.C,
                                     case.x_cache, case.B_cache, case.dt_cache, case.ring_start,
                                     case.prev_num_accepted, case.logical_window,
                                     cu_seqlens=case.cu_seqlens,
                                     state_batch_indices=case.state_batch_indices,
                                     update_trackers=False, **kw)
    if case.kind == "single":
        return ssu.ssu_update(case.state, case.x, case.dt, case.A, case.B, case.C,
                              state_batch_indices=case.state_batch_indices,
                              dst_state_batch_indices=case.dst_state_batch_indices,
                              algorithm=algorithm, **kw)
    return ssu.ssu_update_varlen(case.state, case.x, case.dt, case.A, case.B, case.C,
                                 cu_seqlens=case.cu_seqlens,
                                 num_accepted_tokens=case.num_accepted_tokens,
                                 state_batch_indices=case.state_batch_indices,
                                 dst_state_batch_indices=case.dst_state_batch_indices,
                                 nseqs=case.nseqs, algorithm=algorithm, **kw)


def _case(kind, sdt, seed):
    if kind == "single":
        return W.single_token_case(batch=33, heads=8, headdim=64, dstate=128, groups=2,
                                   slots=80, state_dtype=sdt, pad_frac=0.1, seed=seed,
                                   device=DEV)
    if kind == "varlen":
        return W.varlen_case(nseqs=17, max_len=4, heads=8, headdim=64, dstate=128, groups=2,
                             slots=160, state_dtype=sdt, pad_frac=0.1, seed=seed, device=DEV)
    return W.replay_case(nseqs=21, heads=8, headdim=64, dstate=128, groups=2, slots=48,
                         state_dtype=sdt, max_len=3, logical_window=2, pad_frac=0.1,
                         seed=seed, device=DEV)


CASES = [("single", "bulk"), ("single", "direct"), ("varlen", "direct"), ("varlen", "bulk"),
         ("replay", "auto")]


@pytest.mark.parametrize("sdt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("kind,algo", CASES)
def test_stochastic_rounding_is_the_oracles_rule_on_the_fp32_state(oracle_mod, kind, algo,
                                                                    sdt):
    o = oracle_mod
    case = _case(kind, sdt, seed=61)
    wide = case.clone()
    wide.state = case.state.to(torch.float32)
    before = case.state.clone()
    _call(wide, algo)
    _call(case, algo, _seed())
    torch.cuda.synchronize()
    f32 = wide.state.reshape(-1).cpu()
    got = case.state.reshape(-1).cpu()
    b0 = before.reshape(-1).cpu()
    written = (f32 != b0.float()).nonzero().flatten()
    assert written.numel() > 1000
    bits = torch.int16
    untouched = torch.ones_like(got, dtype=torch.bool)
    untouched[written] = False
    assert torch.equal(got[untouched].view(bits), b0[untouched].view(bits))
    sample = written[torch.randperm(written.numel(), generator=torch.Generator().manual_seed(1))
                     [:3000]].tolist()
    bad = []
    for e in sample:
        want = o.sr_round(float(f32[e]), sdt, o.sr_bits(SEED, e, 10))
        if float(got[e]) != want:
            bad.append((e, float(f32[e]), float(got[e]), want))
    assert not bad, bad[:5]
    # the rounding really is stochastic: some stored values are not the nearest
    nearest = f32[written].to(sdt)
    assert int((nearest.view(bits) != got[written].view(bits)).sum()) > 10


@pytest.mark.parametrize("sdt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("kind", ["single", "varlen", "replay"])
def test_stochastic_rounding_parity_with_the_fp64_oracle(oracle_mod, kind, sdt):
    o = oracle_mod
    case = _case(kind, sdt, seed=71)
    cpu = case.to("cpu")
    before = cpu.state.clone()
    kw = dict(D=cpu.D, z=cpu.z, dt_bias=cpu.dt_bias, dt_softplus=True,
              state_batch_indices=cpu.state_batch_indices, pad_slot_id=cpu.pad_slot_id,
              rand_seed=SEED, philox_rounds=10)
    if kind == "single":
        y_ref = o.ssu_update(cpu.state, cpu.x, cpu.dt, cpu.A, cpu.B, cpu.C,
                             dst_state_batch_indices=cpu.dst_state_batch_indices, **kw)
    elif kind == "varlen":
        y_ref = o.ssu_update_varlen(cpu.state, cpu.x, cpu.dt, cpu.A, cpu.B, cpu.C,
                                    cu_seqlens=cpu.cu_seqlens,
                                    num_accepted_tokens=cpu.num_accepted_tokens,
                                    dst_state_batch_indices=cpu.dst_state_batch_indices, **kw)
    else:
        y_ref = o.replay_update(cpu.state, cpu.x, cpu.dt, cpu.A, cpu.B, cpu.C, cpu.x_cache,
                                cpu.B_cache, cpu.dt_cache, cpu.ring_start, cpu.prev_num_accepted,
                                cpu.logical_window, cu_seqlens=cpu.cu_seqlens,
                                update_trackers=False, **kw)
    out = _call(case, "auto", _seed())
    torch.cuda.synchronize()
    covered = ~torch.isnan(y_ref.reshape(y_ref.shape[0], -1)).any(dim=1)
    P.compare_y(out, y_ref, sdt, rows=covered, label=f"{kind} {sdt}")
    P.compare_pool(case.state, cpu.state, before, label=f"{kind} {sdt}")


def test_seeds_decide_rounds_matter_and_fp32_ignores_the_seed():
    base = _case("single", torch.bfloat16, seed=81)
    a, b, c, d = base.clone(), base.clone(), base.clone(), base.clone()
    _call(a, "auto", _seed(5))
    _call(b, "auto", _seed(5))
    _call(c, "auto", _seed(6))
    _call(d, "auto", _seed(5), rounds=7)
    torch.cuda.synchronize()
    assert torch.equal(a.state, b.state)
    assert not torch.equal(a.state, c.state)
    assert not torch.equal(a.state, d.state)
    f = _case("single", torch.float32, seed=82)
    g = f.clone()
    _call(f, "auto", _seed(5))
    _call(g, "auto")
    torch.cuda.synchronize()
    assert torch.equal(f.state, g.state)
