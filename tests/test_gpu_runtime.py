"""GPU runtime properties of the library beyond parity: CUDA-graph capture of
decode steps on every kernel family, and the bounded-wait failure path of the
bulk-copy kernel."""
from __future__ import annotations

import pytest
import torch

from mamba2_ssm_decode_gb300 import workloads as W

from . import _parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssm_decode_gb300 import build
    build.build()


@pytest.mark.parametrize("algo", ["direct", "bulk"])
def test_decode_step_replays_in_a_cuda_graph(algo):
    """One captured MTP step (SSU + tracker update + commit), replayed three
    times, equals three eager steps bit for bit."""
    import mamba2_ssm_decode_gb300 as ssu
    case = W.mtp_varlen(device=DEV)
    case.dst_state_batch_indices = case.state_batch_indices   # replays chain in place
    eager = case.clone()
    out = torch.empty_like(case.x)

    def step(c, o):
        ssu.ssu_update_varlen(c.state, c.x, c.dt, c.A, c.B, c.C, D=c.D, z=c.z,
                              dt_bias=c.dt_bias, dt_softplus=True, cu_seqlens=c.cu_seqlens,
                              num_accepted_tokens=c.num_accepted_tokens,
                              state_batch_indices=c.state_batch_indices, out=o, algorithm=algo)
        tr = (c.ring_start, c.prev_num_accepted, c.prev_query_len)
        ssu.ssu_ring_update(*tr, c.state_batch_indices, 4, 8)
        ssu.ssu_ring_commit(*tr, c.state_batch_indices, c.num_accepted_tokens, c.cu_seqlens, 4, 8)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    warm = case.clone()
    with torch.cuda.stream(s):
        step(warm, torch.empty_like(out))          # set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(case, out)
    # capturing ran nothing: the state is untouched until the first replay
    assert torch.equal(case.state, eager.state)
    out_e = torch.empty_like(out)
    for _ in range(3):
        g.replay()
        step(eager, out_e)
    torch.cuda.synchronize()
    assert torch.equal(out, out_e)
    assert torch.equal(case.state, eager.state)
    for a, b in ((case.ring_start, eager.ring_start), (case.prev_num_accepted,
                                                      eager.prev_num_accepted),
                 (case.prev_query_len, eager.prev_query_len)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("kind", ["one_token_direct", "no_write_mtp_bf16"])
def test_head_run_calls_replay_in_a_cuda_graph(kind):
    """A one-token call on the head-run kernel (DIRECT) and a no-write MTP call
    (the tensor-core closed form) captured once and replayed three times give
    the bits of the same calls made eagerly."""
    import mamba2_ssm_decode_gb300 as ssu
    if kind == "one_token_direct":
        case = W.single_token_case(batch=96, heads=16, headdim=64, dstate=128, groups=2,
                                   slots=96, state_dtype=torch.float32, identity_slots=True,
                                   seed=21, device=DEV)

        def step(c, o):
            ssu.ssu_update(c.state, c.x, c.dt, c.A, c.B, c.C, D=c.D, z=c.z, dt_bias=c.dt_bias,
                           dt_softplus=True, state_batch_indices=c.state_batch_indices, out=o,
                           algorithm="direct")
    else:
        case = W.varlen_case(nseqs=64, max_len=4, heads=16, headdim=64, dstate=128, groups=2,
                             slots=512, state_dtype=torch.bfloat16, disable_state_update=True,
                             seed=22, device=DEV)

        def step(c, o):
            ssu.ssu_update_varlen(c.state, c.x, c.dt, c.A, c.B, c.C, D=c.D, z=c.z,
                                  dt_bias=c.dt_bias, dt_softplus=True, cu_seqlens=c.cu_seqlens,
                                  num_accepted_tokens=c.num_accepted_tokens,
                                  state_batch_indices=c.state_batch_indices,
                                  dst_state_batch_indices=c.dst_state_batch_indices,
                                  disable_state_update=True, out=o)
    eager = case.clone()
    out = torch.empty_like(case.x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(case.clone(), torch.empty_like(out))   # set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(case, out)
    assert torch.equal(case.state, eager.state)
    out_e = torch.empty_like(out)
    for _ in range(3):
        g.replay()
        step(eager, out_e)
    torch.cuda.synchronize()
    assert torch.equal(out, out_e)
    assert torch.equal(case.state, eager.state)


def test_bounded_wait_gives_up_and_the_context_stays_usable(oracle_mod):
    import mamba2_ssm_decode_gb300 as ssu
    ssu.ssu_device_error(reset=True)
    assert ssu.ssu_device_error() == 0
    waited = ssu.ssu_selftest_bounded_wait(2_000_000)        # 2 ms
    assert 2_000_000 <= waited < 500_000_000
    assert ssu.ssu_device_error() & 1                          # the timeout was recorded
    assert ssu.ssu_device_error(reset=True) & 1
    assert ssu.ssu_device_error() == 0
    # the device still runs the real kernels correctly
    P.parity(oracle_mod, W.tiny(device=DEV), label="after self-test", algorithm="bulk")
    with pytest.raises(ValueError):
        ssu.ssu_selftest_bounded_wait(0)
