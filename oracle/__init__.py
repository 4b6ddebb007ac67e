"""Plain fp64 CPU oracle for the Mamba2 selective state update and the ReplaySSM
ring trackers (and, in ``oracle/ssd.py``, for the packed SSD prefill).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the product path never
does.  The arithmetic lives in ``ssu_oracle.c`` (plain C, IEEE double, no
contraction of a*b+c); this module compiles it with gcc and marshals CPU torch
tensors into it.  It shares no code with the CUDA library.

Parity pins (tests/test_oracle_pins.py) tie every function here to closed
forms, invariants, library routines and hand-worked examples; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssu_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libssu_oracle.so")
_lock = threading.Lock()
_lib = None

# dtype codes of the C interface (ssu_oracle.c's own enum)
_DT = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2, torch.float64: 3}

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile ssu_oracle.c into an in-tree shared library; return its path."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB points the pins at another build of ssu_oracle.c (the
            # mutation test plants mistakes in a copy and expects the pins to fail)
            lib = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
            lib.oracle_ssu_update.restype = _int
            lib.oracle_ssu_update.argtypes = (
                [_p, _int, _i64, _i64, _i64, _i64, _i64, _i64,
                 _p, _p, _int, _p, _int, _p, _p, _p, _p, _p, _p, _p, _i64, _int, _int, _int,
                 _p, _p, _int])
            lib.oracle_ssu_update_varlen.restype = _int
            lib.oracle_ssu_update_varlen.argtypes = (
                [_p, _int, _i64, _i64, _i64, _i64, _i64, _i64, _i64,
                 _p, _p, _int, _p, _int, _p, _p, _p, _p, _p,
                 _p, _i64, _p,
                 _p, _i64, _i64, _i64, _i64,
                 _p, _i64, _i64, _i64, _i64,
                 _i64, _int, _int, _int, _p, _p, _int])
            lib.oracle_ring_update.restype = _int
            lib.oracle_ring_update.argtypes = (
                [_p, _i64, _p, _i64, _p, _i64, _p, _i64, _i64, _int, _i32, _i32, _i64])
            lib.oracle_ring_commit.restype = _int
            lib.oracle_ring_commit.argtypes = (
                [_p, _i64, _p, _i64, _p, _i64, _p, _i64, _p, _p, _i64, _i32, _i32, _i64])
            lib.oracle_replay_update.restype = _int
            lib.oracle_replay_update.argtypes = (
                [_p, _int, _i64, _i64, _i64, _i64, _i64, _i64, _i64,
                 _p, _p, _int, _p, _p, _p, _p, _p, _p,
                 _p, _p, _i64,
                 _p, _p, _p, _i64,
                 _p, _p, _i64, _i32, _int, _int, _int, _p, _p, _int])
            lib.oracle_replay_state.restype = _int
            lib.oracle_replay_state.argtypes = (
                [_p, _int, _i64, _i64, _i64, _i64, _i64, _int, _p, _p, _int, _int,
                 _i64, _p, _p, _p, _i64, _p, _p, _i64, _p])
            lib.oracle_philox4x64.restype = None
            lib.oracle_philox4x64.argtypes = [_p, _p, _int, _p]
            lib.oracle_sr_bits.restype = ctypes.c_uint32
            lib.oracle_sr_bits.argtypes = [ctypes.c_uint64, _int, _i64]
            for f in ("oracle_sr_bf16", "oracle_sr_f16"):
                getattr(lib, f).restype = ctypes.c_double
                getattr(lib, f).argtypes = [ctypes.c_double, ctypes.c_uint32]
            lib.oracle_encode.restype = None
            lib.oracle_encode.argtypes = [_p, _i64, _int, _p]
            lib.oracle_decode.restype = None
            lib.oracle_decode.argtypes = [_p, _i64, _int, _p]
            for f in ("oracle_round_bf16", "oracle_round_f16", "oracle_round_f32"):
                getattr(lib, f).restype = ctypes.c_double
                getattr(lib, f).argtypes = [ctypes.c_double]
            _lib = lib
    return _lib


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _seed(rand_seed):
    """(pointer, keep-alive box) of the call's 64-bit random seed (stochastic
    rounding of 16-bit state), or (None, None)."""
    if rand_seed is None:
        return None, None
    if isinstance(rand_seed, torch.Tensor):
        v = int(rand_seed.reshape(-1)[0].item())
    else:
        v = int(rand_seed)
    box = ctypes.c_uint64(v % (1 << 64))
    return ctypes.byref(box), box


def _cpu(t, dtype=None):
    """A contiguous CPU copy (or view) of t, optionally converted."""
    if t is None:
        return None
    t = t.detach().to("cpu")
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous()


def _params(A, D, dt_bias, H, P):
    """fp32 CPU copies of A, D, dt_bias and the per-(head, dim) bit mask: each is
    [H] (per head) or [H, P] (per channel; a [H, P, N] view with zero dstate
    stride or [H, 1] collapse to these)."""
    mask = 0
    out = []
    for bit, t in ((1, A), (2, D), (4, dt_bias)):
        if t is None:
            out.append(None)
            continue
        t = t.detach().to("cpu", torch.float32)
        if t.dim() == 3:
            t = t[:, :, 0]
        if t.dim() == 2 and t.shape[1] == 1:
            t = t[:, 0]
        if t.dim() == 2:
            assert tuple(t.shape) == (H, P)
            mask |= bit
        out.append(t.contiguous())
    return out[0], out[1], out[2], mask


def _check_io(x, z, B, C):
    io = x.dtype
    assert io in (torch.bfloat16, torch.float16), io
    for t in (z, B, C):
        assert t is None or t.dtype == io
    return _DT[io]


def ssu_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=False,
               state_batch_indices=None, dst_state_batch_indices=None, pad_slot_id=-1,
               disable_state_update=False, rand_seed=None, philox_rounds=10):
    """One-token decode on CPU tensors.

    state: [slots, H, P, N] CPU tensor, updated IN PLACE (must be contiguous).
    x, z: [batch, H, P]; dt: [batch, H] (per head) or [batch, H, P];
    B, C: [batch, G, N]; A, D, dt_bias: [H] or [H, P] fp32.  Returns y as float64
    [batch, H, P] (unrounded).
    """
    lib = _load()
    assert state.device.type == "cpu" and state.is_contiguous()
    slots, H, P, N = state.shape
    batch = x.shape[0]
    G = B.shape[1]
    io = _check_io(x, z, B, C)
    x, z, B, C = _cpu(x), _cpu(z), _cpu(B), _cpu(C)
    dt = _cpu(dt, torch.float32)
    dt_per_dim = int(dt.dim() == 3 and dt.shape[2] != 1)
    A, D, dt_bias, per_dim = _params(A, D, dt_bias, H, P)
    sbi = _cpu(state_batch_indices, torch.int64)
    dsbi = _cpu(dst_state_batch_indices, torch.int64)
    y = torch.empty((batch, H, P), dtype=torch.float64)
    seed, _box = _seed(rand_seed)
    rc = lib.oracle_ssu_update(
        _ptr(state), _DT[state.dtype], slots, H, P, N, G, batch,
        _ptr(x), _ptr(z), io, _ptr(dt), dt_per_dim, _ptr(A), _ptr(D), _ptr(dt_bias),
        _ptr(B), _ptr(C), _ptr(sbi), _ptr(dsbi), int(pad_slot_id), int(bool(dt_softplus)),
        int(bool(disable_state_update)), per_dim, _ptr(y), seed, int(philox_rounds))
    if rc != 0:
        raise ValueError(f"oracle_ssu_update rejected its arguments (code {rc})")
    return y


def _table(t):
    """(tensor, numel, seq_stride, step_stride, steps) for a [S] or [S, T] slot table,
    addressed the way the packed route addresses it: a flat [rows] table has
    strides (1, 1), a 2-D table (T, 1)."""
    if t is None:
        return None, 0, 0, 0, 0
    t64 = _cpu(t, torch.int64)
    if t64.dim() == 1:
        return t64, t64.numel(), 1, 1, t64.numel()
    assert t64.dim() == 2
    return t64.reshape(-1), t64.numel(), t64.shape[1], 1, t64.shape[1]


def ssu_update_varlen(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=False,
                      cu_seqlens=None, nseqs=None, dense_steps=1, num_accepted_tokens=None,
                      state_batch_indices=None, dst_state_batch_indices=None, pad_slot_id=-1,
                      disable_state_update=False, src_table=None, dst_table=None,
                      rand_seed=None, philox_rounds=10):
    """Packed varlen / MTP update on CPU tensors.

    x, z: [rows, H, P]; dt: [rows, H] or [rows, H, P]; B, C: [rows, G, N].
    cu_seqlens: [nseqs + 1] or None (then each sequence has `dense_steps` rows).
    Slot tables: [S] (flat, strides (1, 1)) or [S, T]; or give src_table /
    dst_table as explicit (tensor, numel, seq_stride, step_stride, steps).
    Returns y float64 [rows, H, P]; rows no sequence covers stay NaN.
    """
    lib = _load()
    assert state.device.type == "cpu" and state.is_contiguous()
    slots, H, P, N = state.shape
    rows = x.shape[0]
    G = B.shape[1]
    io = _check_io(x, z, B, C)
    x, z, B, C = _cpu(x), _cpu(z), _cpu(B), _cpu(C)
    dt = _cpu(dt, torch.float32)
    dt_per_dim = int(dt.dim() == 3 and dt.shape[2] != 1)
    A, D, dt_bias, per_dim = _params(A, D, dt_bias, H, P)
    cu = _cpu(cu_seqlens, torch.int64)
    if nseqs is None:
        if cu is not None:
            nseqs = cu.numel() - 1
        else:
            nseqs = rows // dense_steps
    na = _cpu(num_accepted_tokens, torch.int64)
    src = src_table if src_table is not None else _table(state_batch_indices)
    dst = dst_table if dst_table is not None else _table(dst_state_batch_indices)
    src = (_cpu(src[0], torch.int64),) + tuple(src[1:]) if src[0] is not None else src
    dst = (_cpu(dst[0], torch.int64),) + tuple(dst[1:]) if dst[0] is not None else dst
    y = torch.full((rows, H, P), float("nan"), dtype=torch.float64)
    seed, _box = _seed(rand_seed)
    rc = lib.oracle_ssu_update_varlen(
        _ptr(state), _DT[state.dtype], slots, H, P, N, G, nseqs, rows,
        _ptr(x), _ptr(z), io, _ptr(dt), dt_per_dim, _ptr(A), _ptr(D), _ptr(dt_bias),
        _ptr(B), _ptr(C), _ptr(cu), int(dense_steps), _ptr(na),
        _ptr(src[0]), src[1], src[2], src[3], src[4],
        _ptr(dst[0]), dst[1], dst[2], dst[3], dst[4],
        int(pad_slot_id), int(bool(dt_softplus)), int(bool(disable_state_update)), per_dim,
        _ptr(y), seed, int(philox_rounds))
    if rc != 0:
        raise ValueError(f"oracle_ssu_update_varlen rejected its arguments (code {rc})")
    return y


def _trackers(ring_start, prev_num_accepted, prev_query_len):
    for t in (ring_start, prev_num_accepted, prev_query_len):
        assert t.device.type == "cpu" and t.dtype == torch.int32 and t.is_contiguous()


def ring_update(ring_start, prev_num_accepted, prev_query_len, state_batch_indices,
                logical_window=None, ring_buffer_len=None, pad_slot_id=-1):
    """Tracker update on int32 CPU tensors (in place).  logical_window None = reset."""
    lib = _load()
    _trackers(ring_start, prev_num_accepted, prev_query_len)
    sbi = state_batch_indices
    # column 0 of a 2-D [S, T] table: entry i * T of the flattened table
    stride = 1 if sbi.dim() == 1 else sbi.shape[1]
    nseqs = sbi.shape[0]
    base = _cpu(sbi, torch.int64).reshape(-1)
    reset = logical_window is None
    rc = lib.oracle_ring_update(
        _ptr(ring_start), ring_start.numel(), _ptr(prev_num_accepted), prev_num_accepted.numel(),
        _ptr(prev_query_len), prev_query_len.numel(), _ptr(base), stride, nseqs, int(reset),
        0 if reset else int(logical_window), 1 if reset else int(ring_buffer_len), int(pad_slot_id))
    if rc != 0:
        raise ValueError(f"oracle_ring_update rejected its arguments (code {rc})")


def ring_commit(ring_start, prev_num_accepted, prev_query_len, state_batch_indices,
                num_accepted_tokens, query_start_loc, logical_window, ring_buffer_len,
                pad_slot_id=-1):
    """Tracker commit on int32 CPU tensors (in place)."""
    lib = _load()
    _trackers(ring_start, prev_num_accepted, prev_query_len)
    sbi = state_batch_indices
    stride = 1 if sbi.dim() == 1 else sbi.shape[1]
    nseqs = sbi.shape[0]
    base = _cpu(sbi, torch.int64).reshape(-1)
    na = _cpu(num_accepted_tokens, torch.int64)
    qsl = _cpu(query_start_loc, torch.int64)
    rc = lib.oracle_ring_commit(
        _ptr(ring_start), ring_start.numel(), _ptr(prev_num_accepted), prev_num_accepted.numel(),
        _ptr(prev_query_len), prev_query_len.numel(), _ptr(base), stride, _ptr(na), _ptr(qsl),
        nseqs, int(logical_window), int(ring_buffer_len), int(pad_slot_id))
    if rc != 0:
        raise ValueError(f"oracle_ring_commit rejected its arguments (code {rc})")


def _replay_caches(x_cache, B_cache, dt_cache, ring_start, prev_num_accepted, io):
    for name, t in (("x_cache", x_cache), ("B_cache", B_cache)):
        assert t.device.type == "cpu" and t.is_contiguous() and t.dim() == 4, name
        assert _DT[t.dtype] == io, f"{name} must have the x dtype"
    assert dt_cache.device.type == "cpu" and dt_cache.is_contiguous()
    assert dt_cache.dtype == torch.float32 and dt_cache.dim() == 3
    for t in (ring_start, prev_num_accepted):
        assert t.device.type == "cpu" and t.dtype == torch.int32 and t.is_contiguous()
    return x_cache.shape[2], min(ring_start.numel(), prev_num_accepted.numel())


def replay_update(state, x, dt, A, B, C, x_cache, B_cache, dt_cache, ring_start,
                  prev_num_accepted, logical_window, D=None, z=None, dt_bias=None,
                  dt_softplus=False, cu_seqlens=None, state_batch_indices=None, pad_slot_id=-1,
                  update_trackers=True, nseqs=None, rand_seed=None, philox_rounds=10):
    """ReplaySSM checkpointing update on CPU tensors (ssu_oracle.c,
    oracle_replay_update: the readings are stated there).

    state [slots, H, P, N] (checkpoints; fp32/bf16/fp16, or fp64 for pins), the
    caches x_cache [slots, H, R, P], B_cache [slots, G, R, N] (x dtype) and
    dt_cache [slots, H, R] fp32, the int32 trackers ring_start and
    prev_num_accepted: all updated IN PLACE.  x, z [rows, H, P]; dt [rows, H];
    B, C [rows, G, N]; cu_seqlens [S + 1] or None (one row per sequence);
    state_batch_indices [S] (slot per sequence) or None (slot s).  Returns y
    float64 [rows, H, P]."""
    lib = _load()
    assert state.device.type == "cpu" and state.is_contiguous()
    slots, H, P, N = state.shape
    rows = x.shape[0]
    G = B.shape[1]
    io = _check_io(x, z, B, C)
    R, num_states = _replay_caches(x_cache, B_cache, dt_cache, ring_start, prev_num_accepted,
                                   io)
    x, z, B, C = _cpu(x), _cpu(z), _cpu(B), _cpu(C)
    dt = _cpu(dt, torch.float32)
    if dt.dim() == 3:
        assert dt.shape[2] == 1, "ReplaySSM caches one dt per head"
        dt = dt[:, :, 0].contiguous()
    A, D, dt_bias, per_dim = _params(A, D, dt_bias, H, P)
    cu = _cpu(cu_seqlens, torch.int64)
    if nseqs is None:
        nseqs = cu.numel() - 1 if cu is not None else rows
    sbi = _cpu(state_batch_indices, torch.int64)
    if sbi is not None:
        sbi = sbi.reshape(sbi.shape[0], -1)[:, 0].contiguous()   # column 0 of a 2-D table
    y = torch.full((rows, H, P), float("nan"), dtype=torch.float64)
    seed, _box = _seed(rand_seed)
    rc = lib.oracle_replay_update(
        _ptr(state), _DT[state.dtype], slots, H, P, N, G, nseqs, rows,
        _ptr(x), _ptr(z), io, _ptr(dt), _ptr(A), _ptr(D), _ptr(dt_bias), _ptr(B), _ptr(C),
        _ptr(cu), _ptr(sbi), int(pad_slot_id),
        _ptr(x_cache), _ptr(B_cache), _ptr(dt_cache), R,
        _ptr(ring_start), _ptr(prev_num_accepted), num_states, int(logical_window),
        int(bool(update_trackers)), int(bool(dt_softplus)), per_dim, _ptr(y), seed,
        int(philox_rounds))
    if rc != 0:
        raise ValueError(f"oracle_replay_update rejected its arguments (code {rc})")
    return y


def replay_state(state, slot, A, x_cache, B_cache, dt_cache, ring_start, prev_num_accepted,
                 dt_bias=None, dt_softplus=False):
    """The logical state of one slot (checkpoint advanced through its cached
    tokens) as float64 [H, P, N]; nothing is written."""
    lib = _load()
    slots, H, P, N = state.shape
    G = B_cache.shape[1]
    io = _DT[x_cache.dtype]
    R, num_states = _replay_caches(x_cache, B_cache, dt_cache, ring_start, prev_num_accepted,
                                   io)
    A, _, dt_bias, per_dim = _params(A, None, dt_bias, H, P)
    out = torch.empty((H, P, N), dtype=torch.float64)
    rc = lib.oracle_replay_state(
        _ptr(state), _DT[state.dtype], slots, H, P, N, G, io, _ptr(A), _ptr(dt_bias),
        int(bool(dt_softplus)), per_dim, int(slot), _ptr(x_cache), _ptr(B_cache), _ptr(dt_cache),
        R, _ptr(ring_start), _ptr(prev_num_accepted), num_states, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_replay_state: slot {slot} has out-of-range trackers")
    return out


def philox4x64(counter, key, rounds=10):
    """Philox4x64 of a 4-word counter and a 2-word key (python ints) -> 4 ints."""
    lib = _load()
    c = (ctypes.c_uint64 * 4)(*[int(v) % (1 << 64) for v in counter])
    k = (ctypes.c_uint64 * 2)(*[int(v) % (1 << 64) for v in key])
    out = (ctypes.c_uint64 * 4)()
    lib.oracle_philox4x64(c, k, int(rounds), out)
    return list(out)


def sr_bits(seed, e, rounds=10):
    """The 16 random bits of stored element e (index in the state pool) under `seed`."""
    return int(_load().oracle_sr_bits(int(seed) % (1 << 64), int(rounds), int(e)))


def sr_round(v, dtype, r):
    """Stochastic rounding of the double v to bf16 / fp16 with random bits r."""
    lib = _load()
    f = {torch.bfloat16: lib.oracle_sr_bf16, torch.float16: lib.oracle_sr_f16}[dtype]
    return f(float(v), int(r))


def round_to(values: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Round float64 values to `dtype` (RNE, the oracle's rounding) -> tensor of dtype."""
    lib = _load()
    v = _cpu(values, torch.float64)
    out = torch.empty(v.shape, dtype=dtype)
    lib.oracle_encode(_ptr(v), v.numel(), _DT[dtype], _ptr(out))
    return out


def widen(values: torch.Tensor) -> torch.Tensor:
    """Exact float64 value of stored fp32/bf16/fp16 values (the oracle's decoding)."""
    lib = _load()
    v = _cpu(values)
    out = torch.empty(v.shape, dtype=torch.float64)
    lib.oracle_decode(_ptr(v), v.numel(), _DT[v.dtype], _ptr(out))
    return out


def round_scalar(v: float, dtype: torch.dtype) -> float:
    lib = _load()
    f = {torch.bfloat16: lib.oracle_round_bf16, torch.float16: lib.oracle_round_f16,
         torch.float32: lib.oracle_round_f32}[dtype]
    return f(float(v))
