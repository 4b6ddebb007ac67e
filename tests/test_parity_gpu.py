"""GPU parity: the CUDA path (C ABI via the package binding) against the CPU
oracle on the same seeded inputs, element by element.

Small cases span several row tiles and a ragged tail (headdim not a multiple
of the 64-row CTA tile, odd sequence counts, empty sequences); the named
serving workloads run at full size (every element where the host can hold
the pool, sampled sequences for the large-batch sweep)."""
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


SDT = [torch.float32, torch.bfloat16, torch.float16]
IODT = [torch.bfloat16, torch.float16]
ALGOS = ["direct", "bulk"]


# ---------------------------------------------------------------------------
# one-token route
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("sdt", SDT)
@pytest.mark.parametrize("iodt", IODT)
@pytest.mark.parametrize("N", [16, 32, 64, 128, 256])
def test_one_token_dtypes_and_dstate(oracle_mod, sdt, iodt, N, algo):
    case = W.single_token_case(batch=7, heads=6, headdim=80, dstate=N, groups=3, slots=20,
                               state_dtype=sdt, io_dtype=iodt, pad_frac=0.3, seed=N,
                               device=DEV)
    P.parity(oracle_mod, case, label=f"{sdt} {iodt} N={N} {algo}", algorithm=algo)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("variant", ["no_z", "no_D_bias", "dt_per_dim", "dt_h1", "no_softplus",
                                     "dst_table", "in_range_pad", "out_f32", "int64",
                                     "identity", "disable", "P_ragged", "tied_A",
                                     "per_channel", "per_channel_view", "bc_unaligned"])
def test_one_token_variants(oracle_mod, variant, algo):
    kw = dict(batch=9, heads=4, headdim=64, dstate=128, groups=2, slots=24,
              state_dtype=torch.float32, pad_frac=0.2, seed=7, device=DEV)
    if variant == "no_z":
        kw["with_z"] = False
    if variant == "dt_per_dim":
        kw["dt_per_dim"] = True
    if variant == "int64":
        kw["index_dtype"] = torch.int64
    if variant == "identity":
        kw.update(identity_slots=True, pad_frac=0.0)
    if variant == "P_ragged":
        kw["headdim"] = 100   # one full 64-row tile and a ragged one
    case = W.single_token_case(**kw)
    out_dtype = None
    if variant == "no_D_bias":
        case.D, case.dt_bias = None, None
    if variant == "dt_h1":
        case.dt = case.dt[:, :, None]
    if variant == "no_softplus":
        case.dt_softplus = False
        case.dt = case.dt.abs() * 0.1
    if variant == "dst_table":
        # write slots no sequence reads (a slot read by one sequence and written by
        # another is undefined: the kernels run sequences in parallel)
        used = set(case.state_batch_indices.tolist())
        free = [s for s in range(24) if s not in used]
        case.dst_state_batch_indices = torch.tensor(free[:9], dtype=torch.int32, device=DEV)
        case.dst_state_batch_indices[2] = -1
    if variant == "in_range_pad":
        case.pad_slot_id = 0
        case.state_batch_indices[3] = 0
    if variant == "out_f32":
        out_dtype = torch.float32
    if variant == "disable":
        case.disable_state_update = True
    if variant == "identity":
        case.state_batch_indices = None
    if variant == "tied_A":
        case.A = case.A[:, None, None].expand(4, 64, 128)
    if variant in ("per_channel", "per_channel_view"):
        g = torch.Generator(device=DEV).manual_seed(5)
        case.A = -torch.exp(torch.rand(4, 64, generator=g, device=DEV) * 2.7)
        case.D = torch.rand(4, 64, generator=g, device=DEV)
        case.dt_bias = -1 - 3 * torch.rand(4, 64, generator=g, device=DEV)
        if variant == "per_channel_view":   # [H, dim, dstate] with zero dstate stride
            case.A = case.A[:, :, None].expand(4, 64, 128)
            case.dt_bias = case.dt_bias[:, :, None].expand(4, 64, 128)
    if variant == "bc_unaligned":
        unaligned_bc(case)
    P.parity(oracle_mod, case, out_dtype=out_dtype, label=variant, algorithm=algo)


def unaligned_xz(case):
    """Move x and z to odd element offsets (rows not 16-byte aligned)."""
    for name in ("x", "z"):
        t = getattr(case, name)
        R = t.shape[0]
        big = torch.zeros(R, t[0].numel() + 1, dtype=t.dtype, device=t.device)
        v = big[:, 1:].view(t.shape)
        v.copy_(t)
        setattr(case, name, v)


def unaligned_bc(case):
    """Move B and C into one buffer at odd element offsets (rows not 16-byte aligned)."""
    R, G, N = case.B.shape
    big = torch.zeros(R, 2 * G * N + 3, dtype=case.B.dtype, device=case.B.device)
    Bv = big[:, 1:1 + G * N].view(R, G, N)
    Cv = big[:, 2 + G * N:2 + 2 * G * N].view(R, G, N)
    Bv.copy_(case.B)
    Cv.copy_(case.C)
    case.B, case.C = Bv, Cv


def test_one_token_strided_operands_bit_exact():
    """x/z/out/B/C/dt as strided views of larger buffers give the same bits as
    contiguous operands."""
    case = W.single_token_case(batch=5, heads=4, headdim=64, dstate=128, groups=2, slots=10,
                               state_dtype=torch.float32, seed=3, device=DEV)
    ref = case.clone()
    y_ref = P.run_gpu(ref)
    big = torch.zeros(5, 4 * 64 * 3, dtype=torch.bfloat16, device=DEV)
    xv = big[:, 7: 7 + 256].view(5, 4, 64)
    xv.copy_(case.x)
    bigbc = torch.zeros(5, 2 * 128 * 3, dtype=torch.bfloat16, device=DEV)
    Bv = bigbc[:, 0:256].view(5, 2, 128)
    Cv = bigbc[:, 384:640].view(5, 2, 128)
    Bv.copy_(case.B)
    Cv.copy_(case.C)
    dtbig = torch.zeros(5, 12, device=DEV)
    dtv = dtbig[:, ::3]
    dtv.copy_(case.dt)
    case.x, case.B, case.C, case.dt = xv, Bv, Cv, dtv
    y = P.run_gpu(case)
    assert torch.equal(y, y_ref) and torch.equal(case.state, ref.state)


# ---------------------------------------------------------------------------
# calls that write no state (disable_state_update): the register kernel takes
# the closed form of the chain, so every lane layout is checked here too
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("sdt", SDT)
@pytest.mark.parametrize("N", [16, 64, 128, 256])
@pytest.mark.parametrize("kind", ["single", "varlen"])
def test_no_write_dtypes(oracle_mod, kind, sdt, N, algo):
    if kind == "single":
        case = W.single_token_case(batch=7, heads=6, headdim=80, dstate=N, groups=3, slots=20,
                                   state_dtype=sdt, pad_frac=0.3, seed=40 + N,
                                   disable_state_update=True, device=DEV)
    else:
        case = W.varlen_case(nseqs=9, max_len=6, heads=4, headdim=80, dstate=N, groups=2,
                             slots=160, state_dtype=sdt, pad_frac=0.25, seed=50 + N,
                             disable_state_update=True, device=DEV)
    r = P.parity(oracle_mod, case, label=f"no-write {kind} {sdt} N={N} {algo}", algorithm=algo)
    assert r["slots_written"] == 0


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("variant", ["bc_unaligned", "dt_per_dim", "per_channel", "no_z",
                                     "out_f32", "heads_per_group_odd", "f16_state_f16_io",
                                     "dstate64", "ragged_rows", "xz_unaligned"])
@pytest.mark.parametrize("kind", ["single", "varlen"])
def test_no_write_variants(oracle_mod, kind, variant, algo):
    """No-write calls through every staging path: element loads of B / C rows
    off 16-byte alignment, per-row dt' (dt, A, dt_bias per channel), no gate,
    fp32 y, a head count per group that CTAs cannot split in 2 or 4, the
    fp16 tensor-core path, dstate 64 and a headdim that leaves a ragged tile."""
    kw = dict(heads=4, headdim=64, dstate=128, groups=2, state_dtype=torch.bfloat16,
              disable_state_update=True, device=DEV)
    if variant == "dt_per_dim":
        kw["dt_per_dim"] = True
    if variant == "no_z":
        kw["with_z"] = False
    if variant == "heads_per_group_odd":
        kw.update(heads=6, groups=2)   # 3 heads per group
    if variant == "f16_state_f16_io":
        kw.update(state_dtype=torch.float16, io_dtype=torch.float16)
    if variant == "dstate64":
        kw["dstate"] = 64
    if variant == "ragged_rows":
        kw.update(headdim=80, heads=16, groups=2)  # 8 heads per group, a 16-row tail tile
    if kind == "single":
        case = W.single_token_case(batch=9, slots=24, pad_frac=0.2, seed=61, **kw)
    else:
        case = W.varlen_case(nseqs=7, max_len=4, slots=80, pad_frac=0.15, seed=62, **kw)
    if variant == "bc_unaligned":
        unaligned_bc(case)
    if variant == "xz_unaligned":
        unaligned_xz(case)
    if variant == "per_channel":
        g = torch.Generator(device=DEV).manual_seed(8)
        H, Pd = case.A.shape[0], case.x.shape[-1]
        case.A = -torch.exp(torch.rand(H, Pd, generator=g, device=DEV) * 2.7)
        case.D = torch.rand(H, Pd, generator=g, device=DEV)
        case.dt_bias = -1 - 3 * torch.rand(H, Pd, generator=g, device=DEV)
    out_dtype = torch.float32 if variant == "out_f32" else None
    r = P.parity(oracle_mod, case, out_dtype=out_dtype, label=f"no-write {kind} {variant} {algo}",
                 algorithm=algo)
    assert r["slots_written"] == 0


# ---------------------------------------------------------------------------
# packed varlen / MTP route
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("sdt", SDT)
@pytest.mark.parametrize("N", [16, 64, 128, 256])
def test_varlen_dtypes(oracle_mod, sdt, N, algo):
    case = W.varlen_case(nseqs=9, max_len=6, heads=4, headdim=80, dstate=N, groups=2, slots=160,
                         state_dtype=sdt, pad_frac=0.25, seed=11 + N, device=DEV)
    P.parity(oracle_mod, case, label=f"varlen {sdt} N={N} {algo}", algorithm=algo)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("variant", ["empty_seqs", "no_counts", "flat_tables", "dense",
                                     "same_table", "int64", "disable", "no_dst_no_src",
                                     "count_out_of_table", "long_chain", "out_f32",
                                     "dt_per_dim", "f16_io", "per_channel", "bc_unaligned",
                                     "disable_long_chain", "disable_dt_per_dim"])
def test_varlen_variants(oracle_mod, variant, algo):
    kw = dict(nseqs=7, max_len=4, heads=4, headdim=64, dstate=128, groups=2, slots=80,
              state_dtype=torch.float32, pad_frac=0.15, seed=23, device=DEV)
    if variant == "dense":
        kw.update(fixed_len=4, dense=True)
    if variant == "same_table":
        kw["same_tables"] = True
    if variant == "int64":
        kw.update(index_dtype=torch.int64, meta_dtype=torch.int64)
    if variant in ("long_chain", "disable_long_chain"):
        kw.update(max_len=11, slots=200)   # more steps than one staged group of 4
    if variant in ("disable_long_chain", "disable_dt_per_dim"):
        kw["disable_state_update"] = True
    if variant in ("dt_per_dim", "disable_dt_per_dim"):
        kw["dt_per_dim"] = True
    if variant == "f16_io":
        kw["io_dtype"] = torch.float16
    case = W.varlen_case(**kw)
    out_dtype = None
    if variant == "empty_seqs":
        cu = case.cu_seqlens.clone()
        cu[3] = cu[2]            # sequence 2 becomes empty
        cu[5] = cu[4]            # sequence 4 becomes empty
        case.cu_seqlens = cu
        case.num_accepted_tokens = torch.ones_like(case.num_accepted_tokens)
    if variant == "no_counts":
        case.num_accepted_tokens = None
    if variant == "flat_tables":
        # one sequence per call: the flat [rows] table names the same entries
        case = W.varlen_case(nseqs=1, max_len=4, fixed_len=4, heads=4, headdim=64, dstate=128,
                             groups=2, slots=16, state_dtype=torch.float32, seed=5, device=DEV)
        case.state_batch_indices = case.state_batch_indices.reshape(-1)
        case.dst_state_batch_indices = case.dst_state_batch_indices.reshape(-1)
    if variant == "disable":
        case.disable_state_update = True
    if variant == "no_dst_no_src":
        case = W.varlen_case(nseqs=5, max_len=3, heads=4, headdim=64, dstate=128, groups=2,
                             slots=40, state_dtype=torch.float32, seed=9, device=DEV)
        case.state_batch_indices = None
        case.dst_state_batch_indices = None
        case.num_accepted_tokens = None
    if variant == "count_out_of_table":
        na = case.num_accepted_tokens.clone()
        na[0] = 0                                   # position -1: no read slot
        na[1] = case.state_batch_indices.shape[1] + 1  # beyond the table
        case.num_accepted_tokens = na
    if variant == "out_f32":
        out_dtype = torch.float32
    if variant == "bc_unaligned":
        unaligned_bc(case)
    if variant == "per_channel":
        g = torch.Generator(device=DEV).manual_seed(6)
        case.A = -torch.exp(torch.rand(4, 64, generator=g, device=DEV) * 2.7)
        case.D = torch.rand(4, 64, generator=g, device=DEV)
        case.dt_bias = -1 - 3 * torch.rand(4, 64, generator=g, device=DEV)
    P.parity(oracle_mod, case, out_dtype=out_dtype, label=variant, algorithm=algo)


@pytest.mark.parametrize("make", ["mamba2_2p7b_decode", "hybrid_grouped_decode", "mtp_varlen"])
def test_algorithms_bit_identical(make):
    """The register kernel and the bulk-copy pipeline give the same bits."""
    a = getattr(W, make)(device=DEV)
    b = a.clone()
    ya = P.run_gpu(a, algorithm="direct")
    yb = P.run_gpu(b, algorithm="bulk")
    assert torch.equal(ya, yb)
    assert torch.equal(a.state, b.state)
    import mamba2_ssm_decode_gb300 as ssu
    assert ssu.ssu_device_error() == 0


def test_varlen_with_length_one_equals_one_token_bit_exact():
    """The packed route with one row per sequence computes what the one-token
    route computes, bit for bit ("mate.mamba": the one-token fast path is the
    packed call with cu_seqlens = arange(rows + 1))."""
    case = W.single_token_case(batch=11, heads=4, headdim=64, dstate=128, groups=2, slots=30,
                               state_dtype=torch.bfloat16, pad_frac=0.2, seed=13, device=DEV)
    other = case.clone()
    y1 = P.run_gpu(case)
    import mamba2_ssm_decode_gb300 as ssu
    y2 = ssu.ssu_update_varlen(
        other.state, other.x, other.dt, other.A, other.B, other.C, D=other.D, z=other.z,
        dt_bias=other.dt_bias, dt_softplus=True,
        cu_seqlens=torch.arange(12, dtype=torch.int32, device=DEV),
        state_batch_indices=other.state_batch_indices[:, None].contiguous(),
        pad_slot_id=other.pad_slot_id)
    assert torch.equal(y1, y2) and torch.equal(case.state, other.state)


def test_dense_equals_packed_bit_exact():
    case = W.varlen_case(nseqs=6, max_len=4, fixed_len=4, dense=True, heads=4, headdim=64,
                         dstate=128, groups=2, slots=64, state_dtype=torch.float32,
                         same_tables=True, seed=17, device=DEV)
    packed = case.clone()
    packed.cu_seqlens = torch.arange(0, 28, 4, dtype=torch.int32, device=DEV)
    packed.num_accepted_tokens = packed.num_accepted_tokens.to(torch.int32)
    y_dense = P.run_gpu(case)
    y_packed = P.run_gpu(packed)
    assert torch.equal(y_dense, y_packed) and torch.equal(case.state, packed.state)


@pytest.mark.parametrize("sdt,tol", [(torch.float32, 1e-5), (torch.bfloat16, 2e-2)])
def test_chain_equals_single_token_calls(sdt, tol):
    """A k-step chain equals k one-token calls that each read the previous
    write (the single calls round the state between steps)."""
    import mamba2_ssm_decode_gb300 as ssu
    case = W.varlen_case(nseqs=5, max_len=4, fixed_len=4, heads=4, headdim=64, dstate=128,
                         groups=2, slots=64, state_dtype=sdt, seed=29, device=DEV)
    case.num_accepted_tokens = None
    single = case.clone()
    y_chain = P.run_gpu(case).float()
    src = single.state_batch_indices[:, 0].contiguous()
    for t in range(4):
        rows = torch.arange(5, device=DEV) * 4 + t
        dst = single.dst_state_batch_indices[:, t].contiguous()
        y = ssu.ssu_update(single.state, single.x[rows], single.dt[rows], single.A,
                           single.B[rows], single.C[rows], D=single.D, z=single.z[rows],
                           dt_bias=single.dt_bias, dt_softplus=True, state_batch_indices=src,
                           dst_state_batch_indices=dst)
        torch.testing.assert_close(y.float(), y_chain[rows], rtol=tol + 2**-8, atol=tol)
        src = dst
    torch.testing.assert_close(single.state.float(), case.state.float(), rtol=tol, atol=tol)


# ---------------------------------------------------------------------------
# ReplaySSM trackers: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("idx", [torch.int32, torch.int64])
@pytest.mark.parametrize("pad", [-1, 5])
def test_trackers_bit_exact(oracle_mod, idx, pad):
    import mamba2_ssm_decode_gb300 as ssu
    g = torch.Generator().manual_seed(3)
    n_states = 700
    nseqs = 300                       # several 128-thread blocks and a ragged tail
    slots = torch.randperm(n_states + 100, generator=g)[:nseqs]   # some >= num_states
    table = torch.stack([slots, torch.randperm(n_states, generator=g)[:nseqs]], dim=1)
    table[::17, 0] = pad
    table[::23, 0] = -3
    table = table.to(idx)
    rs = torch.randint(0, 8, (n_states + 3,), generator=g, dtype=torch.int64).to(torch.int32)
    pna = torch.randint(0, 6, (n_states,), generator=g, dtype=torch.int64).to(torch.int32)
    pql = torch.randint(0, 5, (n_states + 1,), generator=g, dtype=torch.int64).to(torch.int32)
    lens = torch.randint(0, 5, (nseqs,), generator=g)
    qsl = torch.zeros(nseqs + 1, dtype=torch.int64)
    qsl[1:] = torch.cumsum(lens, 0)
    na = torch.randint(1, 5, (nseqs,), generator=g)
    for meta in (torch.int32, torch.int64):
        cpu = [t.clone() for t in (rs, pna, pql)]
        gpu = [t.clone().to(DEV) for t in (rs, pna, pql)]
        oracle_mod.ring_update(*cpu, table, 4, 8, pad_slot_id=pad)
        ssu.ssu_ring_update(*gpu, table.to(DEV), 4, 8, pad_slot_id=pad)
        oracle_mod.ring_commit(*cpu, table, na, qsl, 4, 8, pad_slot_id=pad)
        ssu.ssu_ring_commit(*gpu, table.to(DEV), na.to(meta).to(DEV), qsl.to(meta).to(DEV), 4, 8,
                            pad_slot_id=pad)
        oracle_mod.ring_update(*cpu, table[:50], pad_slot_id=pad)        # reset
        ssu.ssu_ring_update(*gpu, table[:50].to(DEV), pad_slot_id=pad)
        for c, gg in zip(cpu, gpu):
            assert torch.equal(c, gg.cpu())


def test_trackers_int32_wraparound(oracle_mod):
    import mamba2_ssm_decode_gb300 as ssu
    big = 2**31 - 1
    vals = [(big, 1, 1), (0, big, 0), (big - 3, 7, 9), (-5, 3, 2)]
    for rs0, pna0, pql0 in vals:
        for kind in ("update", "commit"):
            cpu = [torch.tensor([v], dtype=torch.int32) for v in (rs0, pna0, pql0)]
            gpu = [t.clone().to(DEV) for t in cpu]
            sbi = torch.tensor([0])
            if kind == "update":
                oracle_mod.ring_update(*cpu, sbi, 0, 7)
                ssu.ssu_ring_update(*gpu, sbi.to(DEV), 0, 7)
            else:
                na, qsl = torch.tensor([big]), torch.tensor([0, 3])
                oracle_mod.ring_commit(*cpu, sbi, na, qsl, 0, 7)
                ssu.ssu_ring_commit(*gpu, sbi.to(DEV), na.to(DEV), qsl.to(DEV), 0, 7)
            for c, gg in zip(cpu, gpu):
                assert torch.equal(c, gg.cpu()), (kind, rs0, pna0, pql0)


# ---------------------------------------------------------------------------
# the named serving workloads at full size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dt_per_dim", [False, True])
def test_workload_tiny(oracle_mod, dt_per_dim):
    case = W.tiny(device=DEV, dt_per_dim=dt_per_dim)
    P.parity(oracle_mod, case, label="tiny")
    case = W.tiny(device=DEV, dt_per_dim=dt_per_dim)
    P.parity(oracle_mod, case, out_dtype=torch.float32, label="tiny f32 out")


@pytest.mark.parametrize("out_dtype", [None, torch.float32])
def test_workload_mamba2_2p7b_decode(oracle_mod, out_dtype):
    P.parity(oracle_mod, W.mamba2_2p7b_decode(device=DEV), out_dtype=out_dtype,
             label="mamba2-2.7b")


def test_workload_hybrid_grouped_decode(oracle_mod):
    P.parity(oracle_mod, W.hybrid_grouped_decode(device=DEV), label="hybrid")


def test_workload_mtp_varlen_with_trackers(oracle_mod):
    import mamba2_ssm_decode_gb300 as ssu
    case = W.mtp_varlen(device=DEV)
    cpu_tr = [t.cpu().clone() for t in (case.ring_start, case.prev_num_accepted,
                                        case.prev_query_len)]
    P.parity(oracle_mod, case, label="mtp")
    sbi_cpu = case.state_batch_indices.cpu()
    oracle_mod.ring_update(*cpu_tr, sbi_cpu, case.logical_window, case.ring_buffer_len,
                           pad_slot_id=case.pad_slot_id)
    oracle_mod.ring_commit(*cpu_tr, sbi_cpu, case.num_accepted_tokens.cpu(),
                           case.cu_seqlens.cpu(), case.logical_window, case.ring_buffer_len,
                           pad_slot_id=case.pad_slot_id)
    gpu_tr = (case.ring_start, case.prev_num_accepted, case.prev_query_len)
    ssu.ssu_ring_update(*gpu_tr, case.state_batch_indices, case.logical_window,
                        case.ring_buffer_len, pad_slot_id=case.pad_slot_id)
    ssu.ssu_ring_commit(*gpu_tr, case.state_batch_indices, case.num_accepted_tokens,
                        case.cu_seqlens, case.logical_window, case.ring_buffer_len,
                        pad_slot_id=case.pad_slot_id)
    for c, g in zip(cpu_tr, gpu_tr):
        assert torch.equal(c, g.cpu())


SWEEP = [(b, sdt, mode, False) for b in (64, 256, 1024, 4096)
         for sdt in (torch.float32, torch.bfloat16) for mode in ("single", "mtp")]
SWEEP += [(1024, torch.float32, "single", True), (1024, torch.bfloat16, "mtp", True)]


@pytest.mark.parametrize("b,sdt,mode,disable", SWEEP)
def test_workload_sweep_sampled(oracle_mod, b, sdt, mode, disable):
    """Large-batch sweep at full size; the oracle checks 24 seeded sequences
    (pad sequences included) of each call."""
    case = W.sweep_case(b, sdt, mode, disable_state_update=disable, device=DEV)
    g = torch.Generator().manual_seed(b)
    seqs = sorted(set(torch.randperm(b, generator=g)[:22].tolist() + [0, b - 1]))
    sbi = case.state_batch_indices
    pads = torch.nonzero((sbi.reshape(b, -1)[:, 0] == case.pad_slot_id)).flatten().tolist()
    seqs = sorted(set(seqs + pads[:2]))
    res = P.sampled_parity(oracle_mod, case, seqs, label=case.name)
    assert res["rows"] >= len(seqs)
    del case
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# batches beyond the 65535 extent of one grid dimension
# ---------------------------------------------------------------------------

def _big_case(kind, disable, seed_offset=0):
    kw = dict(heads=1, headdim=16, dstate=16, groups=1, state_dtype=torch.float32,
              pad_frac=0.01, disable_state_update=disable, device=DEV)
    if kind == "single":
        return W.single_token_case(batch=70001, slots=70010, seed=71 + seed_offset, **kw)
    return W.varlen_case(nseqs=66000, max_len=2, slots=132010, same_tables=True,
                         seed=72 + seed_offset, **kw)


@pytest.mark.parametrize("disable", [False, True])
@pytest.mark.parametrize("kind", ["single", "varlen"])
def test_more_sequences_than_one_grid_dimension(oracle_mod, kind, disable):
    """The head-run kernels spread sequences over two grid dimensions: every
    element on both sides of the 65535-sequence boundary matches the oracle."""
    case = _big_case(kind, disable)
    r = P.parity(oracle_mod, case, label=f"{kind} disable={disable} beyond 65535 sequences",
                 algorithm="direct")
    if not disable:
        assert r["slots_written"] > 65535


@pytest.mark.parametrize("algo", ["auto", "direct", "bulk"])
@pytest.mark.parametrize("disable", [False, True])
@pytest.mark.parametrize("kind", ["single", "varlen"])
def test_every_call_is_one_launch(kind, disable, algo):
    """Each SSU call issues exactly one kernel launch, whatever the batch: the
    call captured in a CUDA graph holds one kernel node (70001 one-token
    sequences, 66000 packed sequences)."""
    case = _big_case(kind, disable, seed_offset=100)
    assert P.graph_kernel_nodes(lambda: P.run_gpu(case, algorithm=algo)) == 1
