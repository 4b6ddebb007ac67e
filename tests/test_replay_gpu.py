"""GPU parity of the ReplaySSM checkpointing update (C ABI ssu_replay_update)
against the CPU oracle on the same seeded inputs: y element by element at the
state dtype's tolerance, the checkpoint pool (written slots within tolerance,
every other slot bit-identical), the ring caches and the trackers bit-exact.
Plus: an fp32 replayed one-token stream reproduces the plain one-token
kernels' outputs bit for bit, graph capture and replay, one launch per call."""
from __future__ import annotations

import pytest
import torch

import mamba2_ssm_decode_gb300 as ssu
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


def run_gpu(c, out_dtype=None, scratch=None, stream=None):
    return ssu.ssu_replay_update(
        c.state, c.x, c.dt, c.A, c.B, c.C, c.x_cache, c.B_cache, c.dt_cache, c.ring_start,
        c.prev_num_accepted, c.logical_window, D=c.D, z=c.z, dt_bias=c.dt_bias,
        dt_softplus=c.dt_softplus, cu_seqlens=c.cu_seqlens, state_batch_indices=c.state_batch_indices,
        pad_slot_id=c.pad_slot_id, update_trackers=c.update_trackers, scratch=scratch,
        out_dtype=out_dtype, stream=stream)


def run_oracle(o, c):
    return o.replay_update(c.state, c.x, c.dt, c.A, c.B, c.C, c.x_cache, c.B_cache, c.dt_cache,
                           c.ring_start, c.prev_num_accepted, c.logical_window, D=c.D, z=c.z,
                           dt_bias=c.dt_bias, dt_softplus=c.dt_softplus, cu_seqlens=c.cu_seqlens,
                           state_batch_indices=c.state_batch_indices, pad_slot_id=c.pad_slot_id,
                           update_trackers=c.update_trackers, nseqs=c.nseqs)


def _bits(t):
    t = t.detach().cpu().contiguous()
    return t.view({2: torch.int16, 4: torch.int32, 8: torch.int64}[t.element_size()])


def replay_parity(o, case, out_dtype=None, label=""):
    cpu = case.to("cpu")
    before = cpu.state.clone()
    y_ref = run_oracle(o, cpu)
    out = run_gpu(case, out_dtype=out_dtype)
    torch.cuda.synchronize()
    covered = ~torch.isnan(y_ref.reshape(y_ref.shape[0], -1)).any(dim=1)
    ry = P.compare_y(out, y_ref, cpu.state.dtype, rows=covered, label=label)
    rs, nw = P.compare_pool(case.state, cpu.state, before, label=label)
    for n in ("x_cache", "B_cache", "dt_cache", "ring_start", "prev_num_accepted"):
        assert torch.equal(_bits(getattr(case, n)), _bits(getattr(cpu, n))), f"{label}: {n}"
    assert ssu.ssu_device_error() == 0
    return {"y_err": ry, "state_err": rs, "checkpoints": nw}


SDT = [torch.float32, torch.bfloat16, torch.float16]


@pytest.mark.parametrize("sdt", SDT)
@pytest.mark.parametrize("N", [16, 64, 128, 256])
@pytest.mark.parametrize("max_len", [1, 4])
def test_replay_dtypes_and_dstate(oracle_mod, sdt, N, max_len):
    case = W.replay_case(nseqs=9, heads=8, headdim=64, dstate=N, groups=2, slots=20,
                         state_dtype=sdt, max_len=max_len, pad_frac=0.2, seed=N + max_len,
                         device=DEV)
    r = replay_parity(oracle_mod, case, label=f"{sdt} N={N} L<={max_len}")
    assert r["checkpoints"] > 0


@pytest.mark.parametrize("variant", ["f16_io", "no_z", "no_D_bias", "dt_h1", "no_softplus",
                                     "int64", "table_2d", "out_f32", "P_ragged", "per_channel",
                                     "no_sbi", "window_1", "window_0", "long_chain",
                                     "long_chain_bf16", "invalid_trackers", "in_range_pad",
                                     "groups_per_head", "trackers_off", "empty_sequence"])
def test_replay_variants(oracle_mod, variant):
    kw = dict(nseqs=11, heads=8, headdim=64, dstate=128, groups=2, slots=24,
              state_dtype=torch.float32, max_len=3, pad_frac=0.2, seed=3, device=DEV)
    if variant == "f16_io":
        kw["io_dtype"] = torch.float16
    if variant == "no_z":
        kw["with_z"] = False
    if variant == "int64":
        kw.update(index_dtype=torch.int64, meta_dtype=torch.int64)
    if variant == "P_ragged":
        kw["headdim"] = 100
    if variant == "window_1":
        kw.update(logical_window=1, ring_len=6)
    if variant == "window_0":
        kw.update(logical_window=0, ring_len=4)
    if variant in ("long_chain", "long_chain_bf16"):   # k + L beyond one staged chunk
        kw.update(logical_window=12, ring_len=16, max_len=4)
        if variant == "long_chain_bf16":
            kw["state_dtype"] = torch.bfloat16
    if variant == "groups_per_head":
        kw["groups"] = 8
    if variant == "no_sbi":
        kw.update(pad_frac=0.0)
    case = W.replay_case(**kw)
    out_dtype = None
    if variant == "no_D_bias":
        case.D, case.dt_bias = None, None
    if variant == "dt_h1":
        case.dt = case.dt[:, :, None]
    if variant == "no_softplus":   # dt' = dt + dt_bias must stay positive over the chain
        case.dt_softplus = False
        case.dt = case.dt.abs() * 0.1
        case.dt_cache = case.dt_cache.abs() * 0.1
        case.dt_bias = case.dt_bias.abs() * 0.1
    if variant == "table_2d":
        t = case.state_batch_indices
        case.state_batch_indices = torch.stack([t, t.flip(0)], dim=1)   # column 0 is the slot
    if variant == "out_f32":
        out_dtype = torch.float32
    if variant == "per_channel":
        g = torch.Generator(device=DEV).manual_seed(5)
        case.A = -torch.exp(torch.rand(8, 64, generator=g, device=DEV) * 2.7)
        case.D = torch.rand(8, 64, generator=g, device=DEV)
        case.dt_bias = -1 - 3 * torch.rand(8, 64, generator=g, device=DEV)
    if variant == "no_sbi":
        case.state_batch_indices = None
    if variant == "long_chain" or variant == "long_chain_bf16":
        sl = case.state_batch_indices.long()
        ok = sl >= 0
        case.prev_num_accepted[sl[ok]] = 9          # 9 cached + up to 4 new: two chunks
    if variant == "invalid_trackers":
        sl = case.state_batch_indices.long()
        case.prev_num_accepted[sl[0]] = -1
        case.prev_num_accepted[sl[1]] = 8           # k + L > R
        case.ring_start[sl[2]] = 8                  # start outside [0, R)
    if variant == "in_range_pad":
        case.pad_slot_id = int(case.state_batch_indices[4])
    if variant == "trackers_off":
        case.update_trackers = False
    if variant == "empty_sequence":
        cu = case.cu_seqlens.clone()
        cu[3] = cu[2]                               # sequence 2 has no rows
        rows = int(cu[-1])
        case.cu_seqlens = cu
        for n in ("x", "dt", "B", "C", "z"):
            t = getattr(case, n)
            setattr(case, n, t[:rows].contiguous() if t.shape[0] >= rows else t)
        case.update_trackers = True
    replay_parity(oracle_mod, case, out_dtype=out_dtype, label=variant)


@pytest.mark.parametrize("name", ["replay-decode", "replay-mtp"])
def test_replay_serving_workloads_full_size(oracle_mod, name):
    case = W.WORKLOADS[name](device=DEV)
    r = replay_parity(oracle_mod, case, label=name)
    assert r["checkpoints"] > 10


@pytest.mark.parametrize("algo", ["direct", "bulk"])
def test_fp32_replay_stream_reproduces_the_plain_kernels_bit_for_bit(algo):
    """fp32 checkpoints store the fp32 chain exactly, and every replayed step is
    the plain kernels' arithmetic: a replayed one-token stream (tracker update
    in the call, window 4, ring 5) gives the plain one-token kernels' y bits,
    token after token."""
    T, S = 13, 37
    case = W.replay_case(nseqs=S, heads=16, headdim=64, dstate=128, groups=4, slots=40,
                         state_dtype=torch.float32, logical_window=4, ring_len=5, seed=17,
                         device=DEV)
    stream = W.single_token_case(batch=S * T, heads=16, headdim=64, dstate=128, groups=4,
                                 slots=S * T, state_dtype=torch.float32, seed=18, device=DEV)
    case.prev_num_accepted.zero_()
    case.ring_start.zero_()
    plain = case.state.clone()
    sbi = case.state_batch_indices
    scratch = torch.zeros(S, dtype=torch.int32, device=DEV)
    for t in range(T):
        rows = slice(t * S, (t + 1) * S)
        kw = dict(D=case.D, dt_bias=case.dt_bias, dt_softplus=True)
        y_r = ssu.ssu_replay_update(case.state, stream.x[rows], stream.dt[rows], case.A,
                                    stream.B[rows], stream.C[rows], case.x_cache, case.B_cache,
                                    case.dt_cache, case.ring_start, case.prev_num_accepted, 4,
                                    z=stream.z[rows], state_batch_indices=sbi,
                                    update_trackers=True, scratch=scratch, **kw)
        y_p = ssu.ssu_update(plain, stream.x[rows], stream.dt[rows], case.A, stream.B[rows],
                             stream.C[rows], z=stream.z[rows], state_batch_indices=sbi,
                             algorithm=algo, **kw)
        torch.cuda.synchronize()
        assert torch.equal(y_r, y_p), f"token {t}"
    assert int(scratch.abs().sum()) == 0


def test_replay_call_captures_and_replays_in_a_cuda_graph():
    """A captured one-token replay call (tracker update fused) replayed three
    times gives the bits of three eager calls: outputs, checkpoints, rings and
    trackers."""
    case = W.replay_case(nseqs=64, heads=16, headdim=64, dstate=128, groups=2, slots=96,
                         state_dtype=torch.bfloat16, pad_frac=0.1, seed=23, device=DEV)
    eager = case.clone()
    out = torch.empty_like(case.x)
    out_e = torch.empty_like(case.x)
    sc = torch.zeros(case.nseqs, dtype=torch.int32, device=DEV)
    sc_e = torch.zeros(case.nseqs, dtype=torch.int32, device=DEV)

    def call(c, o, scr):
        ssu.ssu_replay_update(c.state, c.x, c.dt, c.A, c.B, c.C, c.x_cache, c.B_cache,
                              c.dt_cache, c.ring_start, c.prev_num_accepted, c.logical_window,
                              D=c.D, z=c.z, dt_bias=c.dt_bias, dt_softplus=True,
                              state_batch_indices=c.state_batch_indices, out=o,
                              update_trackers=True, scratch=scr)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    warm = case.clone()
    with torch.cuda.stream(s):
        call(warm, torch.empty_like(out), torch.zeros_like(sc))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(case, out, sc)
    for _ in range(3):
        g.replay()
        call(eager, out_e, sc_e)
    torch.cuda.synchronize()
    assert torch.equal(out, out_e)
    for n in ("state", "x_cache", "B_cache", "dt_cache", "ring_start", "prev_num_accepted"):
        assert torch.equal(getattr(case, n), getattr(eager, n)), n
    assert int(sc.abs().sum()) == 0 and int(sc_e.abs().sum()) == 0


@pytest.mark.parametrize("update", [True, False])
def test_replay_call_is_one_launch(update):
    case = W.replay_case(nseqs=70001, heads=1, headdim=16, dstate=16, groups=1, slots=70010,
                         state_dtype=torch.float32, seed=29, device=DEV)
    case.update_trackers = update
    scratch = torch.zeros(case.nseqs, dtype=torch.int32, device=DEV)
    assert P.graph_kernel_nodes(lambda: run_gpu(case, scratch=scratch)) == 1


def test_replay_beyond_one_grid_dimension(oracle_mod):
    case = W.replay_case(nseqs=70001, heads=1, headdim=16, dstate=16, groups=1, slots=70010,
                         state_dtype=torch.float32, pad_frac=0.01, seed=31, device=DEV)
    replay_parity(oracle_mod, case, label="70001 sequences")


def test_replay_rejects_what_it_cannot_do():
    case = W.replay_case(nseqs=4, heads=2, headdim=16, dstate=16, groups=1, slots=8,
                         state_dtype=torch.float32, seed=1, device=DEV)
    with pytest.raises(NotImplementedError):   # a per-(head, dim) dt cannot be cached per head
        ssu.ssu_replay_update(case.state, case.x, case.dt[:, :, None].expand(4, 2, 16).contiguous(),
                              case.A, case.B, case.C, case.x_cache, case.B_cache, case.dt_cache,
                              case.ring_start, case.prev_num_accepted, 4)
    with pytest.raises(ValueError):            # the tracker update needs its counters
        ssu.ssu_replay_update(case.state, case.x, case.dt, case.A, case.B, case.C, case.x_cache,
                              case.B_cache, case.dt_cache, case.ring_start,
                              case.prev_num_accepted, 4,
                              scratch=torch.zeros(2, dtype=torch.int32, device=DEV))
