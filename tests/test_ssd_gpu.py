"""GPU parity of the packed SSD prefill (C ABI ssd_combined_fwd_varlen) with
the fp64 oracle (oracle/ssd.py) on the same seeded inputs.

The contractions run on the tensor cores with 16-bit operands (x scaled by
its decay weight, C . B^T scaled by the decays, the entering state) and fp32
accumulation, so each product carries a relative error of about 2^-8; over
sums with mixed signs the bound is stated against the scale of each output
row (one token and head of y, one row of a state): |gpu - ref| <= 2e-2
(|ref| + rms of the row), element by element."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import mamba2_ssm_decode_gb300 as ssu
from mamba2_ssm_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba2_ssm_decode_gb300 import build
    build.build()


@pytest.fixture(scope="module")
def ssd_oracle():
    from oracle import ssd
    return ssd


def run_gpu(c, **kw):
    out = torch.full_like(c.x, float("nan"))
    states = ssu.ssd_combined_fwd_varlen(
        c.x, c.dt, c.A, c.B, c.C, c.chunk_size, c.cu_seqlens, c.cu_chunk_seqlens,
        c.last_chunk_indices, c.seq_idx, out=out, D=c.D, z=c.z, dt_bias=c.dt_bias,
        dt_softplus=c.dt_softplus, dt_limit=c.dt_limit, initial_states=c.initial_states, **kw)
    torch.cuda.synchronize()
    return out, states


def run_oracle(o, c, **kw):
    kw.pop("state_dtype", None)   # the oracle's states are fp64
    return o.ssd_combined_fwd_varlen(
        c.x, c.dt, c.A, c.B, c.C, c.chunk_size, c.cu_seqlens, c.cu_chunk_seqlens,
        c.last_chunk_indices, c.seq_idx, D=c.D, z=c.z, dt_bias=c.dt_bias,
        dt_softplus=c.dt_softplus, dt_limit=c.dt_limit, initial_states=c.initial_states, **kw)


def close(got, ref, label):
    """|got - ref| <= TOL (|ref| + rms of ref's row), a row being the last axis
    (one token and head of y, one state row of a head), floored at 1e-3 of the
    global rms."""
    got = got.detach().cpu().double().numpy()
    assert np.isfinite(got).all(), f"{label}: non-finite values"
    if ref.size == 0:
        return 0.0
    row = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    row = np.maximum(row, 1e-3 * math.sqrt(float(np.mean(ref * ref))))
    excess = np.abs(got - ref) / (TOL * (np.abs(ref) + row))
    worst = float(excess.max())
    print(f"SSDERR {label}: worst {worst:.3f} of tol; p99.9 {np.quantile(excess, 0.999):.3f}")
    assert worst <= 1.0, f"{label}: {worst:.3g}x the tolerance"
    return worst


def parity(o, c, label, **kw):
    out, states = run_gpu(c, **kw)
    assert ssu.ssu_device_error() == 0, "a tensor-core wait gave up"
    y_ref, s_ref = run_oracle(o, c.to("cpu"), **kw)
    covered = int(c.cu_chunk_seqlens[-1])
    ry = close(out[:covered], y_ref[:covered], f"{label}: y")
    rs = close(states, s_ref, f"{label}: states")
    return ry, rs


LENGTHS = [37, 256, 300, 1, 129, 64]


@pytest.mark.parametrize("io", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("N", [64, 128])
@pytest.mark.parametrize("chunk", [64, 128, 256])
def test_ssd_dtypes_dstate_chunks(ssd_oracle, io, N, chunk):
    c = W.ssd_case(lengths=LENGTHS, heads=8, headdim=64, dstate=N, groups=2, chunk_size=chunk,
                   io_dtype=io, seed=chunk + N, device=DEV)
    parity(ssd_oracle, c, f"{io} N={N} chunk={chunk}")


@pytest.mark.parametrize("variant", ["no_init", "no_z", "D_per_dim", "no_D_bias", "dt_limit",
                                     "no_softplus", "intermediate", "state_bf16", "init_bf16",
                                     "int32_meta", "groups_per_head", "one_group", "chunk_16",
                                     "chunk_48"])
def test_ssd_variants(ssd_oracle, variant):
    kw = dict(lengths=LENGTHS, heads=8, headdim=64, dstate=128, groups=2, chunk_size=128,
              seed=5, device=DEV)
    call = {}
    if variant == "no_init":
        kw["with_init"] = False
    if variant == "no_z":
        kw["with_z"] = False
    if variant == "D_per_dim":
        kw["D_per_dim"] = True
    if variant == "init_bf16":
        kw["init_dtype"] = torch.bfloat16
    if variant == "int32_meta":
        kw["index_dtype"] = torch.int32
    if variant == "groups_per_head":
        kw["groups"] = 8
    if variant == "one_group":
        kw["groups"] = 1
    if variant == "chunk_16":
        kw["chunk_size"] = 16
    if variant == "chunk_48":
        kw["chunk_size"] = 48
    c = W.ssd_case(**kw)
    if variant == "no_D_bias":
        c.D, c.dt_bias = None, None
    if variant == "dt_limit":
        c.dt_limit = (0.05, 0.4)
    if variant == "no_softplus":
        c.dt_softplus = False
        c.dt = c.dt.abs() * 0.1
    if variant == "intermediate":
        call["return_intermediate_states"] = True
    if variant == "state_bf16":
        call["state_dtype"] = torch.bfloat16
    if variant == "init_bf16":
        call["state_dtype"] = torch.float32
    parity(ssd_oracle, c, variant, **call)


def test_ssd_prefill_workload_sampled(ssd_oracle):
    """The full Mamba2-2.7B-shaped prefill on the GPU; the oracle on the first
    two sequences (sequences are independent: their chunks, tokens and states
    are a slice of the batch)."""
    c = W.ssd_prefill(device=DEV)
    out, states = run_gpu(c)
    cu = c.cu_seqlens.cpu().tolist()
    last = c.last_chunk_indices.cpu().tolist()
    nb = 2
    T = cu[nb]
    nch = last[nb - 1] + 1
    sub = W.SSDCase(name="sub", x=c.x[:T], dt=c.dt[:T], A=c.A, B=c.B[:T], C=c.C[:T], D=c.D,
                    z=c.z[:T], dt_bias=c.dt_bias, chunk_size=c.chunk_size,
                    cu_seqlens=c.cu_seqlens[:nb + 1], cu_chunk_seqlens=c.cu_chunk_seqlens[:nch + 1],
                    last_chunk_indices=c.last_chunk_indices[:nb], seq_idx=c.seq_idx[:nch],
                    initial_states=c.initial_states[:nb]).to("cpu")
    y_ref, s_ref = run_oracle(ssd_oracle, sub)
    close(out[:T], y_ref, "prefill y")
    close(states[:nb], s_ref, "prefill states")


def test_ssd_out_in_place_and_untouched_tokens():
    """Tokens no chunk covers keep what out held; the returned states are the
    last chunks' (one per sequence)."""
    c = W.ssd_case(lengths=[100, 50], heads=4, headdim=64, dstate=64, groups=1, chunk_size=64,
                   seed=3, device=DEV)
    c.cu_chunk_seqlens = c.cu_chunk_seqlens.clone()
    T = c.x.shape[0]
    out = torch.full_like(c.x, 7.0)
    cuc = c.cu_chunk_seqlens.clone()
    cuc[-1] = T - 10                      # the last 10 tokens belong to no chunk
    st = ssu.ssd_combined_fwd_varlen(c.x, c.dt, c.A, c.B, c.C, c.chunk_size, c.cu_seqlens, cuc,
                                     c.last_chunk_indices, c.seq_idx, out=out, D=c.D, z=c.z,
                                     dt_bias=c.dt_bias, dt_softplus=True,
                                     initial_states=c.initial_states)
    torch.cuda.synchronize()
    assert bool((out[T - 10:] == 7.0).all())
    assert bool(torch.isfinite(out[:T - 10].float()).all())
    assert tuple(st.shape) == (2, 4, 64, 64)


def test_ssd_call_is_three_launches():
    """Chunk states, state passing and the scan (which forms C . B^T itself):
    three kernels per call, whatever the batch, and no allocation with out,
    states and workspace given."""
    from ._parity import graph_kernel_nodes
    c = W.ssd_case(lengths=[300, 17, 256], heads=8, headdim=64, dstate=128, groups=2,
                   chunk_size=128, seed=11, device=DEV)
    out = torch.empty_like(c.x)
    nch = c.cu_chunk_seqlens.numel() - 1
    states = torch.empty((3, 8, 64, 128), dtype=torch.float32, device=DEV)
    ws = torch.empty(ssu.ssd_workspace_bytes(nch, 8, 2, 64, 128, 128), dtype=torch.uint8,
                     device=DEV)

    def call():
        ssu.ssd_combined_fwd_varlen(c.x, c.dt, c.A, c.B, c.C, c.chunk_size, c.cu_seqlens,
                                    c.cu_chunk_seqlens, c.last_chunk_indices, c.seq_idx, out=out,
                                    D=c.D, z=c.z, dt_bias=c.dt_bias, dt_softplus=True,
                                    initial_states=c.initial_states, states=states, workspace=ws)
    assert graph_kernel_nodes(call) == 3


def test_ssd_empty_chunks_and_chunks_shorter_than_a_tile(ssd_oracle):
    """Chunks of no tokens (a sequence's state passes through unchanged and is
    still reported for the chunk) and chunk boundaries that cut sequences into
    pieces of 1..200 tokens, as the chunk metadata allows."""
    c = W.ssd_case(lengths=[150, 90, 3], heads=8, headdim=64, dstate=128, groups=2,
                   chunk_size=256, seed=17, device=DEV)
    # sequence 0: [0, 40) [40, 40) [40, 150); sequence 1: [150, 151) [151, 240);
    # sequence 2: [240, 240) [240, 243)
    dev = c.cu_chunk_seqlens.device
    c.cu_chunk_seqlens = torch.tensor([0, 40, 40, 150, 151, 240, 240, 243], dtype=torch.int64,
                                      device=dev)
    c.seq_idx = torch.tensor([0, 0, 0, 1, 1, 2, 2], dtype=torch.int64, device=dev)
    c.last_chunk_indices = torch.tensor([2, 4, 6], dtype=torch.int64, device=dev)
    parity(ssd_oracle, c, "empty chunks")
    parity(ssd_oracle, c, "empty chunks, every chunk's state", return_intermediate_states=True)
