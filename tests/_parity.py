"""Helpers of the GPU parity tests: run one case through the CUDA path (the
C ABI via the package binding) and through the CPU oracle on identical inputs,
then compare element by element.

Tolerances (the stated acceptance criteria, made concrete):
  * fp32 state: state and an fp32 y within |d| <= 1e-5 + 1e-5 |ref|.
  * bf16 / fp16 state: state and y within |d| <= 2e-2 + 2e-2 |ref|.
  * y stored in a 16-bit out dtype cannot meet 1e-5; it must lie within half
    an ulp of that dtype of the exact value (2^-8 |ref| for bf16, 2^-11 |ref|
    for fp16) plus the state tolerance above.
  * Slots the oracle leaves untouched must be bit-identical on the GPU.
  * Indices and trackers: bit-exact.
"""
from __future__ import annotations

import torch

import mamba2_ssm_decode_gb300 as ssu

STATE_TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-2, torch.float16: 2e-2}
HALF_ULP_REL = {torch.bfloat16: 2.0**-8, torch.float16: 2.0**-11, torch.float32: 0.0}


def run_gpu(case, out_dtype=None, algorithm="auto"):
    """Call the CUDA path for a case whose tensors live on the GPU; returns out."""
    kw = dict(D=case.D, z=case.z, dt_bias=case.dt_bias, dt_softplus=case.dt_softplus,
              pad_slot_id=case.pad_slot_id, disable_state_update=case.disable_state_update,
              out_dtype=out_dtype, algorithm=algorithm)
    if case.kind == "single":
        return ssu.ssu_update(case.state, case.x, case.dt, case.A, case.B, case.C,
                              state_batch_indices=case.state_batch_indices,
                              dst_state_batch_indices=case.dst_state_batch_indices, **kw)
    if case.cu_seqlens is None:  # dense [batch, steps, ...] form
        S, T = case.nseqs, case.dense_steps

        def d4(t):
            if t is None:
                return None
            if t.dim() == 2:   # per-head dt: [rows, H] -> [S, T, H, 1]
                return t.view(S, T, t.shape[1], 1)
            return t.view(S, T, *t.shape[1:])

        out = ssu.ssu_update_varlen(case.state, d4(case.x), d4(case.dt), case.A, d4(case.B),
                                    d4(case.C), num_accepted_tokens=case.num_accepted_tokens,
                                    state_batch_indices=case.state_batch_indices,
                                    dst_state_batch_indices=case.dst_state_batch_indices,
                                    **{**kw, "z": d4(case.z)})
        return out.view(S * T, *out.shape[2:])
    return ssu.ssu_update_varlen(case.state, case.x, case.dt, case.A, case.B, case.C,
                                 cu_seqlens=case.cu_seqlens,
                                 num_accepted_tokens=case.num_accepted_tokens,
                                 state_batch_indices=case.state_batch_indices,
                                 dst_state_batch_indices=case.dst_state_batch_indices,
                                 nseqs=case.nseqs, **kw)


def run_oracle(oracle, case):
    """Run the oracle on a CPU case (state updated in place); returns y float64."""
    kw = dict(D=case.D, z=case.z, dt_bias=case.dt_bias, dt_softplus=case.dt_softplus,
              pad_slot_id=case.pad_slot_id, disable_state_update=case.disable_state_update,
              state_batch_indices=case.state_batch_indices,
              dst_state_batch_indices=case.dst_state_batch_indices)
    if case.kind == "single":
        return oracle.ssu_update(case.state, case.x, case.dt, case.A, case.B, case.C, **kw)
    return oracle.ssu_update_varlen(case.state, case.x, case.dt, case.A, case.B, case.C,
                                    cu_seqlens=case.cu_seqlens, nseqs=case.nseqs,
                                    dense_steps=case.dense_steps,
                                    num_accepted_tokens=case.num_accepted_tokens, **kw)


def _excess(got, ref, atol, rtol, half_ulp=0.0):
    """max over elements of |got - ref| / (atol + (rtol + half_ulp) |ref|)."""
    got = got.to(torch.float64)
    ref = ref.to(torch.float64)
    bound = atol + (rtol + half_ulp) * ref.abs()
    return float(((got - ref).abs() / bound).max()) if got.numel() else 0.0


def compare_y(y_gpu, y_ref, state_dtype, rows=None, label=""):
    """y_gpu: out tensor (any device), y_ref: float64 oracle values."""
    y_gpu = y_gpu.detach().cpu()
    if rows is not None:
        y_gpu, y_ref = y_gpu[rows], y_ref[rows]
    tol = STATE_TOL[state_dtype]
    ratio = _excess(y_gpu, y_ref, tol, tol, HALF_ULP_REL[y_gpu.dtype])
    assert torch.isfinite(y_gpu.to(torch.float32)).all(), f"{label}: non-finite y"
    assert ratio <= 1.0, f"{label}: y error {ratio:.3g}x the tolerance"
    return ratio


def compare_pool(pool_gpu, pool_ref, pool_before, label=""):
    """Whole-pool check: slots the oracle changed within tolerance, the rest bit-identical."""
    g = pool_gpu.detach().cpu()
    r, b = pool_ref, pool_before
    sdt = r.dtype
    S = r.shape[0]
    bits = torch.int32 if sdt == torch.float32 else torch.int16
    changed = (r.view(bits).reshape(S, -1) != b.view(bits).reshape(S, -1)).any(dim=1)
    untouched = ~changed
    same = (g.view(bits).reshape(S, -1) == b.view(bits).reshape(S, -1)).all(dim=1)
    bad = torch.nonzero(untouched & ~same).flatten().tolist()
    assert not bad, f"{label}: slots {bad[:10]} changed on the GPU but not in the oracle"
    tol = STATE_TOL[sdt]
    ratio = _excess(g[changed], r[changed], tol, tol)
    assert ratio <= 1.0, f"{label}: state error {ratio:.3g}x the tolerance"
    return ratio, int(changed.sum())


def parity(oracle, case_gpu, out_dtype=None, label="", algorithm="auto"):
    """Full-size parity of every element: GPU call vs oracle on host copies."""
    cpu = case_gpu.to("cpu")
    before = cpu.state.clone()
    y_ref = run_oracle(oracle, cpu)
    out = run_gpu(case_gpu, out_dtype, algorithm)
    torch.cuda.synchronize()
    covered = ~torch.isnan(y_ref.reshape(y_ref.shape[0], -1)).any(dim=1)
    ry = compare_y(out, y_ref, cpu.state.dtype, rows=covered, label=label)
    rs, nchanged = compare_pool(case_gpu.state, cpu.state, before, label=label)
    assert ssu.ssu_device_error() == 0, f"{label}: device error word set"
    return {"y_err": ry, "state_err": rs, "slots_written": nchanged}


def graph_kernel_nodes(fn):
    """Kernel launches `fn` makes: capture it in a CUDA graph (nothing runs) and
    count the graph's kernel nodes through the driver API."""
    import ctypes
    import pytest
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        pytest.skip("this torch cannot keep the captured graph")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                      # set-up (attributes, lazy loading) outside the capture
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        fn()
    cu = ctypes.CDLL("libcuda.so.1")
    h = ctypes.c_void_p(g.raw_cuda_graph())
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(h, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * max(1, n.value))()
    assert cu.cuGraphGetNodes(h, nodes, ctypes.byref(n)) == 0
    kernels = 0
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kernels += t.value == 0   # CU_GRAPH_NODE_TYPE_KERNEL
    del g
    return kernels


# ---------------------------------------------------------------------------
# sampled parity for workloads too large to copy whole to the host
# ---------------------------------------------------------------------------

def subset(case_gpu, seqs):
    """A small CPU case holding only sequences `seqs` of a GPU case (their rows,
    their slots copied into a compact pool); (cpu_case, rows, slot_map)."""
    from mamba2_ssm_decode_gb300 import workloads as W
    return W.subset_case(case_gpu, seqs)


def sampled_parity(oracle, case_gpu, seqs, out_dtype=None, label="", algorithm="auto"):
    """Parity of the sequences `seqs` of a full-size call made on the GPU: the
    oracle runs on their rows and slots only (copied before the call)."""
    sub, rows, remap = subset(case_gpu, seqs)
    before = sub.state.clone()
    out = run_gpu(case_gpu, out_dtype, algorithm)
    torch.cuda.synchronize()
    y_ref = run_oracle(oracle, sub)
    ry = compare_y(out[torch.tensor(rows, device=out.device)], y_ref, sub.state.dtype,
                   label=label)
    if remap:
        old = torch.tensor(list(remap.keys()), dtype=torch.long, device=case_gpu.state.device)
        new = torch.tensor(list(remap.values()), dtype=torch.long)
        rs, n = compare_pool(case_gpu.state[old], sub.state[new], before[new], label=label)
    else:
        rs, n = 0.0, 0
    return {"y_err": ry, "state_err": rs, "slots_written": n, "rows": len(rows)}
