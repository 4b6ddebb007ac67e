"""GPU runtime properties of the library beyond parity: CUDA-graph capture of
a decode step, and the bounded-wait failure path of the bulk-copy kernel."""
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
