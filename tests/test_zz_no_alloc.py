"""ssu_replay_update_static: the checkpointing update for callers that cannot
pass a scratch buffer (a plugin host that hands an operation only its own
tensors, or a runtime that forbids device allocations after start-up).  Its
tracker counters live in a fixed array inside the library.

Called through the C ABI, it must give what ssu_replay_update gives with
caller-provided scratch -- outputs and checkpoints within the state dtype's
tolerance, rings and trackers bit for bit -- on two calls in a row (the second
call finds the array as the first one left it), and it must refuse a batch
beyond its fixed size before anything runs.  This file is collected last, and
it passes on its own in a fresh process as well as after the other tests."""
from __future__ import annotations

import pytest
import torch

import mamba2_ssm_decode_gb300 as ssu
from mamba2_ssm_decode_gb300 import _abi
from mamba2_ssm_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2, torch.float16: 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssm_decode_gb300 import build
    build.build()


def _within(got, ref, tol, what):
    got, ref = got.double().cpu(), ref.double().cpu()
    excess = ((got - ref).abs() / (tol + tol * ref.abs())).max().item() if got.numel() else 0.0
    assert excess <= 1.0, f"{what}: {excess:.3g}x the tolerance"


def _args(c):
    return (c.state, c.x, c.dt, c.A, c.B, c.C, c.x_cache, c.B_cache, c.dt_cache, c.ring_start,
            c.prev_num_accepted, c.logical_window)


def _kw(c):
    return dict(D=c.D, z=c.z, dt_bias=c.dt_bias, dt_softplus=True, cu_seqlens=c.cu_seqlens,
                state_batch_indices=c.state_batch_indices, pad_slot_id=c.pad_slot_id,
                update_trackers=c.update_trackers)


@pytest.mark.parametrize("kind", ["one_token_fp32", "one_token_bf16", "mtp_fp32"])
def test_static_entry_matches_the_scratch_entry_on_two_calls_in_a_row(kind):
    sdt = torch.bfloat16 if kind.endswith("bf16") else torch.float32
    case = W.replay_case(nseqs=300, heads=16, headdim=64, dstate=128, groups=2, slots=640,
                         state_dtype=sdt, max_len=4 if kind.startswith("mtp") else 1,
                         pad_frac=0.05, seed=41, device=DEV)
    if kind.startswith("mtp"):
        case.update_trackers = True   # exercise the counters on the packed route too
    ref = case.clone()
    scratch = torch.zeros(case.nseqs, dtype=torch.int32, device=DEV)
    for call in range(2):
        out_ref = torch.empty_like(case.x)
        out = torch.empty_like(case.x)
        ssu.ssu_replay_update(*_args(ref), out=out_ref, scratch=scratch, **_kw(ref))
        ssu.ssu_replay_update_static(*_args(case), out=out, **_kw(case))
        torch.cuda.synchronize()
        tol = TOL[sdt]
        _within(out, out_ref, tol, f"{kind} call {call}: y")
        _within(case.state, ref.state, tol, f"{kind} call {call}: checkpoints")
        for n in ("x_cache", "B_cache", "dt_cache", "ring_start", "prev_num_accepted"):
            assert torch.equal(getattr(case, n), getattr(ref, n)), f"{kind} call {call}: {n}"
    assert ssu.ssu_device_error() == 0


def test_static_entry_refuses_more_sequences_than_its_array_holds():
    n = _abi.REPLAY_STATIC_MAX_SEQS + 1
    case = W.replay_case(nseqs=n, heads=1, headdim=16, dstate=16, groups=1, slots=n,
                         state_dtype=torch.float32, seed=43, device=DEV)
    before = case.clone()
    out = torch.zeros_like(case.x)
    with pytest.raises(ValueError, match="at most 65536 sequences"):
        ssu.ssu_replay_update_static(*_args(case), out=out, **_kw(case))
    torch.cuda.synchronize()
    for name in ("state", "x_cache", "ring_start", "prev_num_accepted"):
        assert torch.equal(getattr(case, name), getattr(before, name))
    assert int(out.abs().sum()) == 0
