"""Python binding of the C ABI (include/ssu.h): argument marshalling only.

Each function takes CUDA torch tensors, checks that they describe the layout
the ABI expects (no hidden copies, no compute), and calls the library on the
current torch stream of the tensors' device.  Every step of the operation runs
in libssu_gb300.so; there is no CPU or torch fallback.

Exceptions follow the pages' conventions ("mate.mamba"): ValueError for a
rejected argument, NotImplementedError for a capability the library does not
implement, RuntimeError for a failed launch.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi

_FLOAT_DT = {torch.float32: _abi.SSU_F32, torch.bfloat16: _abi.SSU_BF16,
             torch.float16: _abi.SSU_F16}
_INT_DT = {torch.int32: _abi.SSU_I32, torch.int64: _abi.SSU_I64}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _require_cuda(*tensors):
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libssu_gb300 works on CUDA tensors only (there is no CPU path)")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"all tensors must be on one device, got {dev} and {t.device}")
    return dev


def _float_dtype(t, name):
    if t.dtype not in _FLOAT_DT:
        raise NotImplementedError(f"{name} dtype {t.dtype} is not supported")
    return _FLOAT_DT[t.dtype]


def _int_dtype(t, name):
    if t.dtype not in _INT_DT:
        raise ValueError(f"{name} must be int32 or int64, got {t.dtype}")
    return _INT_DT[t.dtype]


def _rows3(t, name, rows, heads, dim):
    """(row stride, head stride) of a [rows, heads, dim] operand with unit dim stride."""
    if t.dim() != 3 or tuple(t.shape) != (rows, heads, dim):
        raise ValueError(f"{name} must be [{rows}, {heads}, {dim}], got {tuple(t.shape)}")
    if dim > 1 and t.stride(2) != 1:
        raise ValueError(f"{name} must be contiguous along dim (stride 1), got {t.stride()}")
    return t.stride(0), t.stride(1)


def _per_head(t, heads, dim, name):
    """(head stride, dim stride) of an fp32 A / D / dt_bias ("mate.mamba",
    _per_head): per head [H], [H, 1] or a tied [H, dim, dstate] view with zero
    inner strides (dim stride 0); per (head, dim) channel [H, dim] or a
    [H, dim, dstate] view with zero dstate stride."""
    if t is None:
        return 0, 0
    if t.dtype != torch.float32:
        raise NotImplementedError(f"{name} must be fp32, got {t.dtype}")
    if t.shape[0] != heads:
        raise ValueError(f"{name} must have one entry per head ({heads}), got {tuple(t.shape)}")
    if t.dim() == 1:
        return t.stride(0), 0
    if t.dim() == 2 and t.shape[1] == 1:
        return t.stride(0), 0
    if t.dim() == 2 and t.shape[1] == dim:
        return t.stride(0), t.stride(1)
    if t.dim() == 3 and t.stride(1) == 0 and t.stride(2) == 0:
        return t.stride(0), 0
    if t.dim() == 3 and t.shape[1] == dim and t.stride(2) == 0:
        return t.stride(0), t.stride(1)
    raise NotImplementedError(
        f"{name}: per-head or per-(head, dim) values only; got shape {tuple(t.shape)} "
        f"with strides {t.stride()}")


def _seed_ptr(rand_seed, dev):
    """Device address of the call's 64-bit seed (a CUDA int64 / uint64 tensor of
    one element, as the pages draw it), or None."""
    if rand_seed is None:
        return None
    if not rand_seed.is_cuda or rand_seed.device != dev:
        raise ValueError("rand_seed must be a one-element tensor on the call's device")
    if rand_seed.dtype not in (torch.int64, torch.uint64) or rand_seed.numel() != 1:
        raise ValueError("rand_seed must be one 64-bit integer")
    return rand_seed.data_ptr()


def _params(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out,
            disable_state_update, rows, algorithm="auto", rand_seed=None, philox_rounds=10):
    if state.dim() != 4:
        raise ValueError(f"state must be [slots, heads, dim, dstate], got {tuple(state.shape)}")
    if not state.is_contiguous():
        raise ValueError("state must be contiguous")
    slots, H, P, N = state.shape
    sdt = _float_dtype(state, "state")
    if x.dtype not in (torch.bfloat16, torch.float16):
        raise NotImplementedError(f"x must be bf16 or fp16, got {x.dtype}")
    io = _FLOAT_DT[x.dtype]
    xs = _rows3(x, "x", rows, H, P)
    zs = (0, 0) if z is None else _rows3(z, "z", rows, H, P)
    if z is not None and z.dtype != x.dtype:
        raise ValueError("z must match x in shape and dtype")
    os_ = _rows3(out, "out", rows, H, P)
    if out.dtype not in (x.dtype, torch.float32):
        raise ValueError(f"out must be {x.dtype} (or fp32), got {out.dtype}")
    if dt.dtype != torch.float32:
        raise NotImplementedError(f"dt must be fp32, got {dt.dtype}")
    if dt.dim() == 2 and tuple(dt.shape) == (rows, H):
        dts = (dt.stride(0), dt.stride(1), 0)
    elif dt.dim() == 3 and tuple(dt.shape[:2]) == (rows, H) and dt.shape[2] in (1, P):
        dts = (dt.stride(0), dt.stride(1), 0 if dt.shape[2] == 1 else dt.stride(2))
    else:
        raise ValueError(f"dt must be [{rows}, {H}], [{rows}, {H}, 1] or [{rows}, {H}, {P}], "
                         f"got {tuple(dt.shape)}")
    if B.dim() != 3 or C.shape != B.shape or B.shape[0] != rows or B.shape[2] != N:
        raise ValueError(f"B/C must be [rows, groups, dstate]; got B={tuple(B.shape)}, "
                         f"C={tuple(C.shape)}")
    if B.dtype != x.dtype or C.dtype != x.dtype:
        raise ValueError("B and C must share the x dtype")
    if (N > 1 and (B.stride(2) != 1 or C.stride(2) != 1)):
        raise ValueError("B and C must be contiguous along dstate")
    G = B.shape[1]
    p = _abi.SSUParams()
    p.state, p.state_dtype = state.data_ptr(), sdt
    p.slots, p.nheads, p.headdim, p.dstate, p.ngroups = slots, H, P, N, G
    p.io_dtype = io
    p.x, (p.x_row_stride, p.x_head_stride) = x.data_ptr(), xs
    p.z, (p.z_row_stride, p.z_head_stride) = (z.data_ptr() if z is not None else None), zs
    p.out, p.out_dtype = out.data_ptr(), _FLOAT_DT[out.dtype]
    p.out_row_stride, p.out_head_stride = os_
    p.dt = dt.data_ptr()
    p.dt_row_stride, p.dt_head_stride, p.dt_dim_stride = dts
    p.B, p.B_row_stride, p.B_group_stride = B.data_ptr(), B.stride(0), B.stride(1)
    p.C, p.C_row_stride, p.C_group_stride = C.data_ptr(), C.stride(0), C.stride(1)
    p.A = A.data_ptr()
    p.A_stride, p.A_dim_stride = _per_head(A, H, P, "A")
    p.D = D.data_ptr() if D is not None else None
    p.D_stride, p.D_dim_stride = _per_head(D, H, P, "D")
    p.dt_bias = dt_bias.data_ptr() if dt_bias is not None else None
    p.dt_bias_stride, p.dt_bias_dim_stride = _per_head(dt_bias, H, P, "dt_bias")
    p.dt_softplus = int(bool(dt_softplus))
    p.disable_state_update = int(bool(disable_state_update))
    p.pad_slot_id = int(pad_slot_id)
    if algorithm not in _abi.ALGORITHMS:
        raise ValueError(f"algorithm must be one of {sorted(_abi.ALGORITHMS)}, got {algorithm!r}")
    p.algorithm = _abi.ALGORITHMS[algorithm]
    p.rand_seed = _seed_ptr(rand_seed, state.device)
    p.philox_rounds = int(philox_rounds or 10)
    return p


def ssu_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=False,
               state_batch_indices=None, dst_state_batch_indices=None, pad_slot_id=-1,
               out=None, disable_state_update=False, out_dtype=None, algorithm="auto",
               stream=None, rand_seed=None, philox_rounds=10):
    """One-token selective state update (C ABI ``ssu_update``).

    state [slots, H, P, N] (updated in place); x, z [batch, H, P]; dt [batch, H]
    or [batch, H, P] fp32; B, C [batch, G, N]; A, D, dt_bias per head fp32;
    slot vectors [batch] int32/int64.  Returns ``out`` [batch, H, P] (x dtype,
    or ``out_dtype=torch.float32``).  ``algorithm``: "auto", "direct" or "bulk"
    (the two kernels of the library; identical results).  ``rand_seed``: a
    one-element int64 CUDA tensor turns on stochastic rounding of a 16-bit
    state pool (``philox_rounds`` Philox rounds)."""
    dev = _require_cuda(state, x, dt, A, B, C, D, z, dt_bias, state_batch_indices,
                        dst_state_batch_indices, out, rand_seed)
    batch = x.shape[0]
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=dev)
    p = _params(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out,
                disable_state_update, batch, algorithm, rand_seed, philox_rounds)
    idx_dt = 0
    for name, t in (("state_batch_indices", state_batch_indices),
                    ("dst_state_batch_indices", dst_state_batch_indices)):
        if t is not None:
            if t.dim() != 1 or t.shape[0] != batch:
                raise ValueError(f"{name} must be [sequences] ({batch}) on the one-token path; "
                                 f"got {tuple(t.shape)}")
            if t.stride(0) != 1 and batch > 1:
                raise ValueError(f"{name} must be contiguous")
            d = _int_dtype(t, name)
            if idx_dt and d != idx_dt:
                raise ValueError("state_batch_indices and dst_state_batch_indices must share a dtype")
            idx_dt = d
    _abi.check(_abi.lib().ssu_update(
        ctypes.byref(p), batch, _ptr(state_batch_indices), _ptr(dst_state_batch_indices),
        idx_dt or _abi.SSU_I32, _stream(dev, stream)))
    return out


def _table(t, name):
    if t is None:
        return _abi.SlotTable(None, 0, 0, 0, 0), 0
    d = _int_dtype(t, name)
    if t.dim() == 1:   # flat [rows]: entry (s, t) = s + t ("mate.mamba", _slot_table)
        return _abi.SlotTable(t.data_ptr(), t.numel(), t.stride(0), t.stride(0), t.numel()), d
    if t.dim() == 2:   # [sequences, steps]
        numel = (t.shape[0] - 1) * t.stride(0) + (t.shape[1] - 1) * t.stride(1) + 1
        return _abi.SlotTable(t.data_ptr(), numel if t.numel() else 0, t.stride(0), t.stride(1),
                              t.shape[1]), d
    raise ValueError(f"{name} must be the flat [rows] or the 2-D [sequences, steps] slot "
                     f"table; got {tuple(t.shape)}")


def ssu_update_varlen(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=False,
                      cu_seqlens=None, num_accepted_tokens=None, state_batch_indices=None,
                      dst_state_batch_indices=None, pad_slot_id=-1, out=None,
                      disable_state_update=False, nseqs=None, out_dtype=None, algorithm="auto",
                      stream=None, rand_seed=None, philox_rounds=10):
    """Packed varlen / MTP selective state update (C ABI ``ssu_update_varlen``).

    x is packed [rows, H, P] with ``cu_seqlens`` [S + 1], or dense
    [batch, steps, H, P] (then dt/B/C/z are 4-D as well and equal-length
    sequences are implied).  Slot tables are [S, T] or flat [rows];
    ``num_accepted_tokens`` [S] picks the read position (count - 1).
    ``rand_seed`` / ``philox_rounds``: stochastic rounding, as for ssu_update."""
    dev = _require_cuda(state, x, dt, A, B, C, D, z, dt_bias, cu_seqlens, num_accepted_tokens,
                        state_batch_indices, dst_state_batch_indices, out, rand_seed)
    dense_steps = 1
    dense_out = None
    dense_shape = None
    if x.dim() == 4:
        dense_shape = tuple(x.shape)
        batch, steps = x.shape[:2]
        rows = batch * steps

        def flat(t, name):
            if t is None:
                return None
            if t.dim() != 4:
                raise ValueError(f"a dense (4-D) x requires a 4-D {name} as well, got "
                                 f"{tuple(t.shape)}")
            return t.view(rows, *t.shape[2:])  # a view, never a copy

        x, dt, B, C, z = flat(x, "x"), flat(dt, "dt"), flat(B, "B"), flat(C, "C"), flat(z, "z")
        if out is not None:
            dense_out = out
            out = out.view(rows, *out.shape[2:])
        if cu_seqlens is None:
            dense_steps = steps
            nseqs = batch
    rows = x.shape[0]
    if nseqs is None:
        if cu_seqlens is not None:
            nseqs = cu_seqlens.numel() - 1
        elif num_accepted_tokens is not None:
            nseqs = num_accepted_tokens.numel()
        elif state_batch_indices is not None:
            nseqs = state_batch_indices.shape[0]
        elif dst_state_batch_indices is not None:
            nseqs = dst_state_batch_indices.shape[0]
        else:
            raise ValueError("a packed multi-token call must carry per-sequence metadata: "
                             "state_batch_indices, dst_state_batch_indices, "
                             "num_accepted_tokens or cu_seqlens")
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=dev)
    p = _params(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out,
                disable_state_update, rows, algorithm, rand_seed, philox_rounds)
    meta_dt = 0
    if cu_seqlens is not None:
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() != nseqs + 1:
            raise ValueError(f"cu_seqlens must hold {nseqs + 1} entries, got "
                             f"{tuple(cu_seqlens.shape)}")
        if cu_seqlens.stride(0) != 1 and cu_seqlens.numel() > 1:
            raise ValueError("cu_seqlens must be contiguous")
        meta_dt = _int_dtype(cu_seqlens, "cu_seqlens")
    if num_accepted_tokens is not None:
        if num_accepted_tokens.dim() != 1 or num_accepted_tokens.numel() != nseqs:
            raise ValueError(f"num_accepted_tokens must be [sequences] ({nseqs}), got "
                             f"{tuple(num_accepted_tokens.shape)}")
        if num_accepted_tokens.stride(0) != 1 and nseqs > 1:
            raise ValueError("num_accepted_tokens must be contiguous")
        d = _int_dtype(num_accepted_tokens, "num_accepted_tokens")
        if meta_dt and d != meta_dt:
            raise ValueError("cu_seqlens and num_accepted_tokens must share a dtype")
        meta_dt = d
    src, sd = _table(state_batch_indices, "state_batch_indices")
    dst, dd = _table(dst_state_batch_indices, "dst_state_batch_indices")
    if sd and dd and sd != dd:
        raise ValueError("state_batch_indices and dst_state_batch_indices must share a dtype")
    _abi.check(_abi.lib().ssu_update_varlen(
        ctypes.byref(p), nseqs, rows, _ptr(cu_seqlens), dense_steps, _ptr(num_accepted_tokens),
        meta_dt or _abi.SSU_I32, ctypes.byref(src), ctypes.byref(dst), sd or dd or _abi.SSU_I32,
        _stream(dev, stream)))
    if dense_out is not None:
        return dense_out
    if dense_shape is not None:    # a dense call gets its rank back ("mate.mamba")
        return out.view(dense_shape[:2] + tuple(out.shape[1:]))
    return out


def ssu_replay_update(state, x, dt, A, B, C, x_cache, B_cache, dt_cache, ring_start,
                      prev_num_accepted, logical_window, D=None, z=None, dt_bias=None,
                      dt_softplus=False, cu_seqlens=None, state_batch_indices=None,
                      pad_slot_id=-1, out=None, update_trackers=True, scratch=None,
                      out_dtype=None, stream=None, rand_seed=None, philox_rounds=10):
    """ReplaySSM checkpointing update (C ABI ``ssu_replay_update``).

    state [slots, H, P, N] holds checkpoints; x_cache [slots, H, R, P] and
    B_cache [slots, G, R, N] (x dtype), dt_cache [slots, H, R] fp32 are the
    rings; ring_start / prev_num_accepted int32 trackers by slot.  x, z
    [rows, H, P], dt [rows, H] (per head), B, C [rows, G, N]; ``cu_seqlens``
    [S + 1] packs several rows per sequence (None: one row per sequence).
    ``state_batch_indices`` [S] (or [S, T]: column 0) gives each sequence's
    slot.  With ``update_trackers`` the one-token tracker rule runs in the
    same launch; it needs ``scratch``, S int32 counters that are zero before
    the first call (every call leaves them zero) -- a zeroed tensor is
    allocated when none is given.  ``rand_seed`` / ``philox_rounds``:
    stochastic rounding of 16-bit checkpoints, as for ssu_update.  Returns
    ``out``."""
    dev = _require_cuda(state, x, dt, A, B, C, D, z, dt_bias, x_cache, B_cache, dt_cache,
                        ring_start, prev_num_accepted, cu_seqlens, state_batch_indices, out,
                        scratch, rand_seed)
    rows = x.shape[0]
    if dt.dim() == 3 and dt.shape[2] == 1:
        dt = dt[:, :, 0]
    if cu_seqlens is not None:
        if cu_seqlens.dim() != 1 or (cu_seqlens.numel() > 1 and cu_seqlens.stride(0) != 1):
            raise ValueError("cu_seqlens must be a contiguous vector")
        nseqs = cu_seqlens.numel() - 1
        meta = _int_dtype(cu_seqlens, "cu_seqlens")
    else:
        nseqs = rows
        meta = _abi.SSU_I32
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=dev)
    p = _params(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out, False, rows,
                "auto", rand_seed, philox_rounds)
    slots, H, P, N = state.shape
    G = B.shape[1]
    if x_cache.dim() != 4 or tuple(x_cache.shape[:2]) != (slots, H) or x_cache.shape[3] != P:
        raise ValueError(f"x_cache must be [{slots}, {H}, R, {P}], got {tuple(x_cache.shape)}")
    R = x_cache.shape[2]
    if tuple(B_cache.shape) != (slots, G, R, N):
        raise ValueError(f"B_cache must be [{slots}, {G}, {R}, {N}], got {tuple(B_cache.shape)}")
    if tuple(dt_cache.shape) != (slots, H, R):
        raise ValueError(f"dt_cache must be [{slots}, {H}, {R}], got {tuple(dt_cache.shape)}")
    for name, t, d in (("x_cache", x_cache, x.dtype), ("B_cache", B_cache, x.dtype),
                       ("dt_cache", dt_cache, torch.float32)):
        if t.dtype != d:
            raise ValueError(f"{name} must be {d}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    for name, t in (("ring_start", ring_start), ("prev_num_accepted", prev_num_accepted)):
        if t.dtype != torch.int32:
            raise NotImplementedError(f"{name} must be int32, got {t.dtype}")
        if t.dim() != 1 or (t.numel() > 1 and t.stride(0) != 1):
            raise ValueError(f"{name} must be a contiguous vector")
    sbi = state_batch_indices
    idx = _abi.SSU_I32
    sbi_stride = 1
    if sbi is not None:
        if sbi.dim() == 2:   # a [S, T] table: its column 0, as the pages' wrapper takes
            sbi = sbi[:, 0]
        if sbi.dim() != 1 or sbi.shape[0] != nseqs:
            raise ValueError(f"state_batch_indices must give one slot per sequence ({nseqs})")
        sbi_stride = sbi.stride(0)
        idx = _int_dtype(sbi, "state_batch_indices")
    if update_trackers and scratch is None:
        scratch = torch.zeros(max(1, nseqs), dtype=torch.int32, device=dev)
    rc = _abi.ReplayCache(x_cache.data_ptr(), B_cache.data_ptr(), dt_cache.data_ptr(), R,
                          ring_start.data_ptr(), prev_num_accepted.data_ptr(),
                          min(ring_start.numel(), prev_num_accepted.numel()),
                          int(logical_window))
    sb = 0 if scratch is None else scratch.numel() * scratch.element_size()
    _abi.check(_abi.lib().ssu_replay_update(
        ctypes.byref(p), ctypes.byref(rc), nseqs, rows, _ptr(cu_seqlens), meta, _ptr(sbi),
        sbi_stride, idx, int(bool(update_trackers)), _ptr(scratch), sb, _stream(dev, stream)))
    return out


def ssu_replay_update_static(state, x, dt, A, B, C, x_cache, B_cache, dt_cache, ring_start,
                             prev_num_accepted, logical_window, D=None, z=None, dt_bias=None,
                             dt_softplus=False, cu_seqlens=None, state_batch_indices=None,
                             pad_slot_id=-1, out=None, update_trackers=True, stream=None,
                             rand_seed=None, philox_rounds=10):
    """ssu_replay_update for callers that cannot pass scratch (C ABI
    ``ssu_replay_update_static``): the tracker counters live in a fixed array
    inside the library, so the call needs no buffer beyond its operands.  At
    most ``_abi.REPLAY_STATIC_MAX_SEQS`` sequences; the first call on a device
    must come before any stream capture there; calls that overlap on the device
    share the counters and must not be made.  ``out`` must be given (this
    entry point is for callers that allocate nothing)."""
    dev = _require_cuda(state, x, dt, A, B, C, D, z, dt_bias, x_cache, B_cache, dt_cache,
                        ring_start, prev_num_accepted, cu_seqlens, state_batch_indices, out)
    if out is None:
        raise ValueError("ssu_replay_update_static writes into a caller-provided out")
    rows = x.shape[0]
    if dt.dim() == 3 and dt.shape[2] == 1:
        dt = dt[:, :, 0]
    nseqs, meta = rows, _abi.SSU_I32
    if cu_seqlens is not None:
        nseqs = cu_seqlens.numel() - 1
        meta = _int_dtype(cu_seqlens, "cu_seqlens")
    p = _params(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out, False, rows,
                "auto", rand_seed, philox_rounds)
    slots, H, P, N = state.shape
    R = x_cache.shape[2]
    if (tuple(x_cache.shape) != (slots, H, R, P) or tuple(B_cache.shape) != (slots, B.shape[1], R, N)
            or tuple(dt_cache.shape) != (slots, H, R)):
        raise ValueError("ring caches must be [slots, H, R, P], [slots, G, R, N], [slots, H, R]")
    for t, d in ((x_cache, x.dtype), (B_cache, x.dtype), (dt_cache, torch.float32),
                 (ring_start, torch.int32), (prev_num_accepted, torch.int32)):
        if t.dtype != d or not t.is_contiguous():
            raise ValueError(f"ring caches and trackers must be contiguous {d}")
    sbi, stride, idx = state_batch_indices, 1, _abi.SSU_I32
    if sbi is not None:
        if sbi.dim() == 2:
            sbi = sbi[:, 0]
        stride, idx = sbi.stride(0), _int_dtype(sbi, "state_batch_indices")
    rc = _abi.ReplayCache(x_cache.data_ptr(), B_cache.data_ptr(), dt_cache.data_ptr(), R,
                          ring_start.data_ptr(), prev_num_accepted.data_ptr(),
                          min(ring_start.numel(), prev_num_accepted.numel()),
                          int(logical_window))
    _abi.check(_abi.lib().ssu_replay_update_static(
        ctypes.byref(p), ctypes.byref(rc), nseqs, rows, _ptr(cu_seqlens), meta, _ptr(sbi),
        stride, idx, int(bool(update_trackers)), _stream(dev, stream)))
    return out


def ssd_workspace_bytes(nchunks, nheads, ngroups, headdim, dstate, chunk_size):
    """Bytes of workspace ssd_combined_fwd_varlen needs (C ABI ``ssd_workspace_bytes``)."""
    return int(_abi.lib().ssd_workspace_bytes(nchunks, nheads, ngroups, headdim, dstate,
                                              chunk_size))


def ssd_combined_fwd_varlen(x, dt, A, B, C, chunk_size, cu_seqlens, cu_chunk_seqlens,
                            last_chunk_indices, seq_idx, out=None, D=None, z=None, dt_bias=None,
                            dt_softplus=False, dt_limit=(0.0, float("inf")),
                            initial_states=None, return_intermediate_states=False,
                            state_dtype=None, states=None, workspace=None, stream=None):
    """Packed variable-length SSD prefill (C ABI ``ssd_combined_fwd_varlen``),
    with the call contract of "mate.mamba" ``ssd_combined_fwd_varlen``.

    Returns the chunk states: [nchunks, H, P, N] with
    ``return_intermediate_states``, else [batch, H, P, N] (the last chunk of
    each sequence), in ``state_dtype`` (default: ``states``' dtype when given,
    else the initial states' dtype, else C's).  ``out`` and ``states`` are
    written in place when given.  ``workspace`` (a CUDA uint8 tensor of at
    least ssd_workspace_bytes(...) bytes) is allocated when not given; with
    ``out``, ``states`` and ``workspace`` given the call allocates nothing."""
    dev = _require_cuda(x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, last_chunk_indices,
                        seq_idx, out, D, z, dt_bias, initial_states, states, workspace)
    if x.dim() != 3 or dt.dim() != 2 or B.dim() != 3 or C.dim() != 3:
        raise ValueError("packed SSD expects x [tokens, heads, dim] and dt [tokens, heads]")
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    if tuple(dt.shape) != (T, H):
        raise ValueError("dt must be [tokens, heads]")
    if x.dtype not in (torch.bfloat16, torch.float16) or B.dtype != x.dtype or C.dtype != x.dtype:
        raise ValueError("x, B and C must share one of fp16 / bf16")
    if dt.dtype != torch.float32:
        raise NotImplementedError("dt must be fp32")
    if H % G:
        raise ValueError("heads must be divisible by groups")
    if tuple(A.shape) != (H,) or A.dtype != torch.float32:
        raise ValueError("A must be fp32 [heads]")
    if dt_bias is not None and (tuple(dt_bias.shape) != (H,) or dt_bias.dtype != torch.float32):
        raise ValueError("dt_bias must be fp32 [heads]")
    if chunk_size <= 0:
        raise ValueError("chunk_size must be positive")
    nchunks = cu_chunk_seqlens.numel() - 1
    if nchunks < 1:
        raise ValueError("cu_chunk_seqlens must have at least two entries")
    if seq_idx.numel() != nchunks:
        raise ValueError("seq_idx must hold one request id per logical chunk")
    if cu_seqlens.numel() != last_chunk_indices.numel() + 1:
        raise ValueError("cu_seqlens and last_chunk_indices must describe the same batch")
    batch = last_chunk_indices.numel()
    meta = _int_dtype(cu_chunk_seqlens, "cu_chunk_seqlens")
    for name, t in (("seq_idx", seq_idx), ("last_chunk_indices", last_chunk_indices)):
        if _int_dtype(t, name) != meta:
            raise ValueError("the chunk metadata must share one integer dtype")
    if initial_states is not None:
        if tuple(initial_states.shape) != (batch, H, P, N):
            raise ValueError("initial_states must be [batch, heads, dim, dstate]")
        if not initial_states.is_contiguous():
            raise ValueError("initial_states must be contiguous")
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must match x's shape and dtype")
    D_per_dim = 0
    if D is not None:
        if tuple(D.shape) == (H, P):
            D_per_dim = 1
        elif tuple(D.shape) != (H,):
            raise ValueError("D must be [heads, dim] or [heads]")
        if D.dtype != torch.float32 or not D.is_contiguous():
            raise NotImplementedError("D must be contiguous fp32")
    if z is not None and (z.shape != x.shape or z.dtype != x.dtype or not z.is_contiguous()):
        raise ValueError("z must match x's shape")
    if state_dtype is None:
        state_dtype = (states.dtype if states is not None else
                       initial_states.dtype if initial_states is not None else C.dtype)
    if state_dtype not in _FLOAT_DT:
        raise ValueError("state_dtype must be fp16, bf16 or fp32")
    for t in (x, dt, A, B, C, cu_seqlens, cu_chunk_seqlens, last_chunk_indices, seq_idx):
        if not t.is_contiguous():
            raise ValueError("x, dt, A, B, C and the chunk metadata must be contiguous")
    rows = nchunks if return_intermediate_states else batch
    if states is None:
        states = torch.empty((rows, H, P, N), dtype=state_dtype, device=dev)
    elif (tuple(states.shape) != (rows, H, P, N) or states.dtype != state_dtype
          or not states.is_contiguous()):
        raise ValueError(f"states must be a contiguous {state_dtype} tensor of shape "
                         f"{(rows, H, P, N)}")
    need = ssd_workspace_bytes(nchunks, H, G, P, N, chunk_size)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    p = _abi.SSDParams()
    p.x, p.dt, p.A, p.B, p.C = (x.data_ptr(), dt.data_ptr(), A.data_ptr(), B.data_ptr(),
                                C.data_ptr())
    p.D = D.data_ptr() if D is not None else None
    p.D_per_dim = D_per_dim
    p.z = z.data_ptr() if z is not None else None
    p.dt_bias = dt_bias.data_ptr() if dt_bias is not None else None
    p.dt_softplus = int(bool(dt_softplus))
    p.dt_min, p.dt_max = float(dt_limit[0]), float(dt_limit[1])
    p.out = out.data_ptr()
    p.io_dtype = _FLOAT_DT[x.dtype]
    p.tokens, p.nheads, p.headdim, p.dstate, p.ngroups = T, H, P, N, G
    p.chunk_size, p.nchunks, p.batch = int(chunk_size), nchunks, batch
    p.cu_chunk_seqlens = cu_chunk_seqlens.data_ptr()
    p.seq_idx = seq_idx.data_ptr()
    p.last_chunk_indices = last_chunk_indices.data_ptr()
    p.meta_dtype = meta
    p.initial_states = initial_states.data_ptr() if initial_states is not None else None
    p.initial_dtype = _FLOAT_DT[initial_states.dtype] if initial_states is not None else 0
    p.states = states.data_ptr()
    p.state_dtype = _FLOAT_DT[state_dtype]
    p.return_intermediate_states = int(bool(return_intermediate_states))
    _abi.check(_abi.lib().ssd_combined_fwd_varlen(
        ctypes.byref(p), ctypes.c_void_p(workspace.data_ptr()),
        workspace.numel() * workspace.element_size(), _stream(dev, stream)))
    return states


def _tracker_args(ring_start, prev_num_accepted, prev_query_len, state_batch_indices):
    for name, t in (("ring_start", ring_start), ("prev_num_accepted", prev_num_accepted),
                    ("prev_query_len", prev_query_len)):
        if t.dtype != torch.int32:
            raise NotImplementedError(f"{name} must be int32, got {t.dtype}")
        if t.dim() != 1 or (t.numel() > 1 and t.stride(0) != 1):
            raise ValueError(f"{name} must be a contiguous vector")
    sbi = state_batch_indices
    if sbi.dim() > 2:
        raise ValueError(f"state_batch_indices must be [S] or [S, T], got {tuple(sbi.shape)}")
    nseqs = sbi.shape[0]
    stride = sbi.stride(0)   # column 0 of a 2-D table
    return nseqs, stride, _int_dtype(sbi, "state_batch_indices")


def ssu_device_error(reset=False):
    """The current device's error word (C ABI ``ssu_device_error``; synchronises)."""
    v = ctypes.c_uint(0)
    _abi.check(_abi.lib().ssu_device_error(ctypes.byref(v), int(bool(reset))))
    return v.value


def ssu_selftest_bounded_wait(limit_ns):
    """Run the bounded-wait self-test (C ABI ``ssu_selftest_bounded_wait``); returns
    the nanoseconds the device waited before giving up.  Synchronises."""
    v = ctypes.c_uint64(0)
    _abi.check(_abi.lib().ssu_selftest_bounded_wait(int(limit_ns), ctypes.byref(v)))
    return v.value


def ssu_ring_update(ring_start, prev_num_accepted, prev_query_len, state_batch_indices,
                    logical_window=None, ring_buffer_len=None, pad_slot_id=-1, stream=None):
    """ReplaySSM tracker update (C ABI ``ssu_ring_update``); ``logical_window=None``
    resets the trackers of the given slots, as the pages' wrapper does."""
    dev = _require_cuda(ring_start, prev_num_accepted, prev_query_len, state_batch_indices)
    nseqs, stride, idt = _tracker_args(ring_start, prev_num_accepted, prev_query_len,
                                       state_batch_indices)
    reset = logical_window is None
    if not reset and ring_buffer_len is None:
        raise ValueError("ring_buffer_len is required when logical_window is given")
    _abi.check(_abi.lib().ssu_ring_update(
        _ptr(ring_start), ring_start.numel(), _ptr(prev_num_accepted), prev_num_accepted.numel(),
        _ptr(prev_query_len), prev_query_len.numel(), _ptr(state_batch_indices), stride, idt,
        nseqs, int(reset), 0 if reset else int(logical_window),
        1 if reset else int(ring_buffer_len), int(pad_slot_id), _stream(dev, stream)))


def ssu_ring_commit(ring_start, prev_num_accepted, prev_query_len, state_batch_indices,
                    num_accepted_tokens, query_start_loc, logical_window, ring_buffer_len,
                    pad_slot_id=-1, stream=None):
    """ReplaySSM tracker commit (C ABI ``ssu_ring_commit``)."""
    dev = _require_cuda(ring_start, prev_num_accepted, prev_query_len, state_batch_indices,
                        num_accepted_tokens, query_start_loc)
    nseqs, stride, idt = _tracker_args(ring_start, prev_num_accepted, prev_query_len,
                                       state_batch_indices)
    if num_accepted_tokens.numel() < nseqs or query_start_loc.numel() < nseqs + 1:
        raise ValueError("num_accepted_tokens needs one entry and query_start_loc one start "
                         "per sequence (plus the total)")
    mdt = _int_dtype(num_accepted_tokens, "num_accepted_tokens")
    if _int_dtype(query_start_loc, "query_start_loc") != mdt:
        raise ValueError("num_accepted_tokens and query_start_loc must share a dtype")
    for name, t in (("num_accepted_tokens", num_accepted_tokens),
                    ("query_start_loc", query_start_loc)):
        if t.dim() != 1 or (t.numel() > 1 and t.stride(0) != 1):
            raise ValueError(f"{name} must be a contiguous vector")
    _abi.check(_abi.lib().ssu_ring_commit(
        _ptr(ring_start), ring_start.numel(), _ptr(prev_num_accepted), prev_num_accepted.numel(),
        _ptr(prev_query_len), prev_query_len.numel(), _ptr(state_batch_indices), stride, idt,
        _ptr(num_accepted_tokens), _ptr(query_start_loc), mdt, nseqs, int(logical_window),
        int(ring_buffer_len), int(pad_slot_id), _stream(dev, stream)))
