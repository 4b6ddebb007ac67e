"""ctypes view of include/ssu.h and the loader of libssu_gb300.so.

The library is built in-tree by ``mamba2_ssm_decode_gb300.build`` (or
``__graft_entry__.build()``).  There is no fallback: if the library is missing
or cannot be loaded, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libssu_gb300.so")

# ssu_status
SSU_OK = 0
SSU_ERR_INVALID_ARGUMENT = 1
SSU_ERR_UNSUPPORTED = 2
SSU_ERR_CUDA = 3

# ssu_algorithm
SSU_ALGO_AUTO, SSU_ALGO_DIRECT, SSU_ALGO_BULK = 0, 1, 2
ALGORITHMS = {"auto": SSU_ALGO_AUTO, "direct": SSU_ALGO_DIRECT, "bulk": SSU_ALGO_BULK}

# ssu_dtype
SSU_F32, SSU_BF16, SSU_F16, SSU_I32, SSU_I64 = 0, 1, 2, 3, 4

ABI_VERSION = 4
REPLAY_STATIC_MAX_SEQS = 65536   # SSU_REPLAY_STATIC_MAX_SEQS

_c_i64 = ctypes.c_int64
_c_int = ctypes.c_int
_c_i32 = ctypes.c_int32
_c_p = ctypes.c_void_p


class SSUParams(ctypes.Structure):
    """struct ssu_params (field order and types exactly as in include/ssu.h)."""

    _fields_ = [
        ("state", _c_p), ("state_dtype", _c_int),
        ("slots", _c_i64), ("nheads", _c_i64), ("headdim", _c_i64), ("dstate", _c_i64),
        ("ngroups", _c_i64),
        ("io_dtype", _c_int),
        ("x", _c_p), ("x_row_stride", _c_i64), ("x_head_stride", _c_i64),
        ("z", _c_p), ("z_row_stride", _c_i64), ("z_head_stride", _c_i64),
        ("out", _c_p), ("out_dtype", _c_int), ("out_row_stride", _c_i64),
        ("out_head_stride", _c_i64),
        ("dt", _c_p), ("dt_row_stride", _c_i64), ("dt_head_stride", _c_i64),
        ("dt_dim_stride", _c_i64),
        ("B", _c_p), ("B_row_stride", _c_i64), ("B_group_stride", _c_i64),
        ("C", _c_p), ("C_row_stride", _c_i64), ("C_group_stride", _c_i64),
        ("A", _c_p), ("A_stride", _c_i64), ("A_dim_stride", _c_i64),
        ("D", _c_p), ("D_stride", _c_i64), ("D_dim_stride", _c_i64),
        ("dt_bias", _c_p), ("dt_bias_stride", _c_i64), ("dt_bias_dim_stride", _c_i64),
        ("dt_softplus", _c_int), ("disable_state_update", _c_int),
        ("pad_slot_id", _c_i64),
        ("algorithm", _c_int),
        ("rand_seed", _c_p), ("philox_rounds", _c_int),
    ]


class SlotTable(ctypes.Structure):
    """struct ssu_slot_table."""

    _fields_ = [("indices", _c_p), ("numel", _c_i64), ("seq_stride", _c_i64),
                ("step_stride", _c_i64), ("steps", _c_i64)]


class ReplayCache(ctypes.Structure):
    """struct ssu_replay_cache."""

    _fields_ = [("x_cache", _c_p), ("B_cache", _c_p), ("dt_cache", _c_p), ("ring_len", _c_i64),
                ("ring_start", _c_p), ("prev_num_accepted", _c_p), ("num_states", _c_i64),
                ("logical_window", _c_i32)]


class SSDParams(ctypes.Structure):
    """struct ssd_params."""

    _fields_ = [
        ("x", _c_p), ("dt", _c_p), ("A", _c_p), ("B", _c_p), ("C", _c_p), ("D", _c_p),
        ("D_per_dim", _c_int), ("z", _c_p), ("dt_bias", _c_p), ("dt_softplus", _c_int),
        ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float), ("out", _c_p),
        ("io_dtype", _c_int),
        ("tokens", _c_i64), ("nheads", _c_i64), ("headdim", _c_i64), ("dstate", _c_i64),
        ("ngroups", _c_i64), ("chunk_size", _c_i64), ("nchunks", _c_i64), ("batch", _c_i64),
        ("cu_chunk_seqlens", _c_p), ("seq_idx", _c_p), ("last_chunk_indices", _c_p),
        ("meta_dtype", _c_int), ("initial_states", _c_p), ("initial_dtype", _c_int),
        ("states", _c_p), ("state_dtype", _c_int), ("return_intermediate_states", _c_int),
    ]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libssu_gb300.so (once) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -m mamba2_ssm_decode_gb300.build` "
                "(the CUDA path has no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        L.ssu_update.restype = _c_int
        L.ssu_update.argtypes = [ctypes.POINTER(SSUParams), _c_i64, _c_p, _c_p, _c_int, _c_p]
        L.ssu_update_varlen.restype = _c_int
        L.ssu_update_varlen.argtypes = [ctypes.POINTER(SSUParams), _c_i64, _c_i64, _c_p, _c_i64,
                                        _c_p, _c_int, ctypes.POINTER(SlotTable),
                                        ctypes.POINTER(SlotTable), _c_int, _c_p]
        L.ssu_replay_update.restype = _c_int
        L.ssu_replay_update.argtypes = [ctypes.POINTER(SSUParams), ctypes.POINTER(ReplayCache),
                                        _c_i64, _c_i64, _c_p, _c_int, _c_p, _c_i64, _c_int, _c_int,
                                        _c_p, _c_i64, _c_p]
        L.ssu_replay_update_static.restype = _c_int
        L.ssu_replay_update_static.argtypes = [ctypes.POINTER(SSUParams),
                                               ctypes.POINTER(ReplayCache), _c_i64, _c_i64, _c_p,
                                               _c_int, _c_p, _c_i64, _c_int, _c_int, _c_p]
        L.ssd_workspace_bytes.restype = _c_i64
        L.ssd_workspace_bytes.argtypes = [_c_i64] * 6
        L.ssd_combined_fwd_varlen.restype = _c_int
        L.ssd_combined_fwd_varlen.argtypes = [ctypes.POINTER(SSDParams), _c_p, _c_i64, _c_p]
        L.ssu_ring_update.restype = _c_int
        L.ssu_ring_update.argtypes = [_c_p, _c_i64, _c_p, _c_i64, _c_p, _c_i64, _c_p, _c_i64,
                                      _c_int, _c_i64, _c_int, _c_i32, _c_i32, _c_i64, _c_p]
        L.ssu_ring_commit.restype = _c_int
        L.ssu_ring_commit.argtypes = [_c_p, _c_i64, _c_p, _c_i64, _c_p, _c_i64, _c_p, _c_i64,
                                      _c_int, _c_p, _c_p, _c_int, _c_i64, _c_i32, _c_i32, _c_i64,
                                      _c_p]
        L.ssu_status_string.restype = ctypes.c_char_p
        L.ssu_status_string.argtypes = [_c_int]
        L.ssu_last_error.restype = ctypes.c_char_p
        L.ssu_last_error.argtypes = []
        L.ssu_device_error.restype = _c_int
        L.ssu_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), _c_int]
        L.ssu_selftest_bounded_wait.restype = _c_int
        L.ssu_selftest_bounded_wait.argtypes = [ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64)]
        L.ssu_abi_version.restype = _c_int
        L.ssu_abi_version.argtypes = []
        if L.ssu_abi_version() != ABI_VERSION:
            raise RuntimeError(f"libssu_gb300.so ABI {L.ssu_abi_version()} != {ABI_VERSION}")
        _lib = L
        return _lib


def check(status: int) -> None:
    """Raise the exception class the pages use for this status."""
    if status == SSU_OK:
        return
    L = lib()
    msg = L.ssu_last_error().decode() or L.ssu_status_string(status).decode()
    if status == SSU_ERR_INVALID_ARGUMENT:
        raise ValueError(msg)
    if status == SSU_ERR_UNSUPPORTED:
        raise NotImplementedError(msg)
    raise RuntimeError(f"libssu_gb300: {msg}")
