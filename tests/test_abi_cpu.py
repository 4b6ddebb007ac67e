"""The C ABI without a GPU: the library loads, exports every function that
include/ssu.h declares, its struct layout matches the header, and rejected
arguments come back as the documented status codes before any launch.

Nothing here launches a kernel: every call below is rejected on the host or
has zero sequences (which returns before any CUDA call)."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

from mamba2_ssm_decode_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssu.h")


@pytest.fixture(scope="module")
def lib():
    from mamba2_ssm_decode_gb300 import build
    build.build()
    return _abi.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(ss[ud]_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"ssu_update", "ssu_update_varlen", "ssu_ring_update", "ssu_ring_commit"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libssu_gb300.so does not export {n}"
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(names), f"unexpected exports: {exported ^ set(names)}"
    assert lib.ssu_abi_version() == _abi.ABI_VERSION


def test_struct_layout_matches_header(tmp_path):
    """offsetof / sizeof from a C compile of include/ssu.h equal the ctypes mirror."""
    fields = [f for f, _ in _abi.SSUParams._fields_]
    tfields = [f for f, _ in _abi.SlotTable._fields_]
    rfields = [f for f, _ in _abi.ReplayCache._fields_]
    src = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', 'int main(void){']
    src.append('printf("%zu\\n", sizeof(ssu_params));')
    src += [f'printf("%zu\\n", offsetof(ssu_params, {f}));' for f in fields]
    src.append('printf("%zu\\n", sizeof(ssu_slot_table));')
    src += [f'printf("%zu\\n", offsetof(ssu_slot_table, {f}));' for f in tfields]
    src.append('printf("%zu\\n", sizeof(ssu_replay_cache));')
    src += [f'printf("%zu\\n", offsetof(ssu_replay_cache, {f}));' for f in rfields]
    sfields = [f for f, _ in _abi.SSDParams._fields_]
    src.append('printf("%zu\\n", sizeof(ssd_params));')
    src += [f'printf("%zu\\n", offsetof(ssd_params, {f}));' for f in sfields]
    src.append('printf("%zu\\n", sizeof(ssu_dtype)); return 0; }')
    c = tmp_path / "layout.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-o", str(exe), str(c)], check=True)
    vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    want = [ctypes.sizeof(_abi.SSUParams)] + [getattr(_abi.SSUParams, f).offset for f in fields]
    want += [ctypes.sizeof(_abi.SlotTable)] + [getattr(_abi.SlotTable, f).offset for f in tfields]
    want += [ctypes.sizeof(_abi.ReplayCache)]
    want += [getattr(_abi.ReplayCache, f).offset for f in rfields]
    want += [ctypes.sizeof(_abi.SSDParams)] + [getattr(_abi.SSDParams, f).offset for f in sfields]
    want += [ctypes.sizeof(ctypes.c_int)]
    assert vals == want


def test_header_compiles_as_c_and_cpp(tmp_path):
    for lang, comp in (("c", "gcc"), ("cpp", "g++")):
        f = tmp_path / f"inc.{lang}"
        f.write_text(f'#include "{HEADER}"\nint main(void) {{ return SSU_ABI_VERSION - 1; }}\n')
        subprocess.run([comp, "-Wall", "-Werror", "-o", str(tmp_path / f"inc_{lang}"), str(f)],
                       check=True)


FAKE = 0x10000  # a 16-byte aligned address the host code never dereferences


def valid_params(**over):
    p = _abi.SSUParams()
    p.state, p.state_dtype = FAKE, _abi.SSU_F32
    p.slots, p.nheads, p.headdim, p.dstate, p.ngroups = 8, 4, 16, 128, 2
    p.io_dtype = _abi.SSU_BF16
    p.x, p.x_row_stride, p.x_head_stride = FAKE, 64, 16
    p.out, p.out_dtype, p.out_row_stride, p.out_head_stride = FAKE, _abi.SSU_BF16, 64, 16
    p.dt, p.dt_row_stride, p.dt_head_stride, p.dt_dim_stride = FAKE, 4, 1, 0
    p.B, p.B_row_stride, p.B_group_stride = FAKE, 256, 128
    p.C, p.C_row_stride, p.C_group_stride = FAKE, 256, 128
    p.A, p.A_stride = FAKE, 1
    p.dt_softplus, p.pad_slot_id = 1, -1
    for k, v in over.items():
        setattr(p, k, v)
    return p


def call_update(lib, p, batch=2, sbi=None, dsbi=None, idx=_abi.SSU_I32):
    return lib.ssu_update(ctypes.byref(p), batch, sbi, dsbi, idx, None)


@pytest.mark.parametrize("over,code,needle", [
    (dict(state_dtype=_abi.SSU_I32), _abi.SSU_ERR_UNSUPPORTED, "state dtype"),
    (dict(io_dtype=_abi.SSU_F32), _abi.SSU_ERR_UNSUPPORTED, "x/z/B/C dtype"),
    (dict(out_dtype=_abi.SSU_F16), _abi.SSU_ERR_INVALID_ARGUMENT, "out must have"),
    (dict(dstate=100), _abi.SSU_ERR_UNSUPPORTED, "dstate"),
    (dict(ngroups=3), _abi.SSU_ERR_INVALID_ARGUMENT, "multiple of ngroups"),
    (dict(nheads=0), _abi.SSU_ERR_INVALID_ARGUMENT, "positive sizes"),
    (dict(state=FAKE + 8), _abi.SSU_ERR_INVALID_ARGUMENT, "16-byte aligned"),
    (dict(x=None), _abi.SSU_ERR_INVALID_ARGUMENT, "must not be NULL"),
    (dict(A=None), _abi.SSU_ERR_INVALID_ARGUMENT, "must not be NULL"),
])
def test_update_rejections(lib, over, code, needle):
    st = call_update(lib, valid_params(**over))
    assert st == code
    assert needle in lib.ssu_last_error().decode()


def test_update_slot_rules(lib):
    p = valid_params()
    assert call_update(lib, p, batch=9) == _abi.SSU_ERR_INVALID_ARGUMENT   # > slots, no table
    assert "uses slot b" in lib.ssu_last_error().decode()
    assert call_update(lib, p, batch=2, sbi=FAKE, idx=_abi.SSU_F32) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call_update(lib, p, batch=-1) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call_update(lib, p, batch=0) == _abi.SSU_OK                      # nothing to launch
    assert lib.ssu_last_error().decode() == ""


def call_varlen(lib, p, nseqs=2, rows=4, cu=None, dense=2, na=None, meta=_abi.SSU_I32,
                src=None, dst=None, idx=_abi.SSU_I32):
    src = src or _abi.SlotTable(None, 0, 0, 0, 0)
    dst = dst or _abi.SlotTable(None, 0, 0, 0, 0)
    return lib.ssu_update_varlen(ctypes.byref(p), nseqs, rows, cu, dense, na, meta,
                                 ctypes.byref(src), ctypes.byref(dst), idx, None)


def test_varlen_rejections(lib):
    p = valid_params()
    table = _abi.SlotTable(FAKE, 8, 4, 1, 4)
    # acceptance counts need a read table ("mate.mamba", _packed_selective_state_update)
    assert call_varlen(lib, p, na=FAKE) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert "needs state_batch_indices" in lib.ssu_last_error().decode()
    # rows must split evenly without cu_seqlens
    assert call_varlen(lib, p, rows=5) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call_varlen(lib, p, dense=0) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call_varlen(lib, p, cu=FAKE, meta=_abi.SSU_BF16) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call_varlen(lib, p, src=table, idx=_abi.SSU_F16) == _abi.SSU_ERR_INVALID_ARGUMENT
    bad = _abi.SlotTable(FAKE, -1, 4, 1, 4)
    assert call_varlen(lib, p, src=bad) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call_varlen(lib, p, nseqs=9, rows=18) == _abi.SSU_ERR_INVALID_ARGUMENT  # > slots
    assert call_varlen(lib, p, nseqs=0, rows=0) == _abi.SSU_OK


def test_tracker_rejections(lib):
    f = ctypes.c_void_p(FAKE)
    upd = lambda **k: lib.ssu_ring_update(  # noqa: E731
        f, 8, f, 8, f, 8, f, 1, k.get("idx", _abi.SSU_I32), k.get("n", 4), k.get("reset", 0),
        4, k.get("rb", 8), -1, None)
    assert upd(rb=0) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert "ring_buffer_len" in lib.ssu_last_error().decode()
    assert upd(idx=_abi.SSU_F32) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert upd(n=-1) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert upd(n=0) == _abi.SSU_OK
    assert upd(n=0, reset=1, rb=0) == _abi.SSU_OK   # a reset ignores the ring length
    com = lambda **k: lib.ssu_ring_commit(  # noqa: E731
        f, 8, f, 8, f, 8, f, 1, _abi.SSU_I32, k.get("na", f), k.get("qsl", f),
        k.get("meta", _abi.SSU_I32), k.get("n", 4), 4, k.get("rb", 8), -1, None)
    assert com(na=None) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert com(meta=_abi.SSU_F16) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert com(rb=0) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert com(n=0) == _abi.SSU_OK


def call_replay(lib, p, nseqs=2, rows=2, cu=None, meta=_abi.SSU_I32, sbi=None, idx=_abi.SSU_I32,
                update=0, scratch=None, sbytes=0, rc=None):
    f = FAKE
    rc = rc or _abi.ReplayCache(f, f, f, 8, f, f, 8, 4)
    return lib.ssu_replay_update(ctypes.byref(p), ctypes.byref(rc), nseqs, rows, cu, meta, sbi,
                                 1, idx, update, scratch, sbytes, None)


def test_replay_rejections(lib):
    p = valid_params()
    assert call_replay(lib, valid_params(disable_state_update=1)) == _abi.SSU_ERR_UNSUPPORTED
    assert call_replay(lib, valid_params(dt_dim_stride=1)) == _abi.SSU_ERR_UNSUPPORTED
    assert "one dt per head" in lib.ssu_last_error().decode()
    assert call_replay(lib, p, rows=3) == _abi.SSU_ERR_INVALID_ARGUMENT     # rows != nseqs
    assert call_replay(lib, p, nseqs=9, rows=9) == _abi.SSU_ERR_INVALID_ARGUMENT   # > slots
    assert call_replay(lib, p, cu=FAKE, meta=_abi.SSU_F32, rows=5) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call_replay(lib, p, sbi=FAKE, idx=_abi.SSU_BF16) == _abi.SSU_ERR_INVALID_ARGUMENT
    bad = _abi.ReplayCache(FAKE, FAKE, FAKE, 0, FAKE, FAKE, 8, 4)
    assert call_replay(lib, p, rc=bad) == _abi.SSU_ERR_INVALID_ARGUMENT       # ring_len 0
    nul = _abi.ReplayCache(FAKE, None, FAKE, 8, FAKE, FAKE, 8, 4)
    assert call_replay(lib, p, rc=nul) == _abi.SSU_ERR_INVALID_ARGUMENT
    # the fused tracker update needs 4 * nseqs bytes of counters
    assert call_replay(lib, p, update=1) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert "scratch" in lib.ssu_last_error().decode()
    assert call_replay(lib, p, update=1, scratch=FAKE, sbytes=7) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call_replay(lib, p, nseqs=0, rows=0) == _abi.SSU_OK


def test_ssd_rejections(lib):
    def params(**over):
        p = _abi.SSDParams()
        p.x = p.dt = p.A = p.B = p.C = p.out = p.states = FAKE
        p.cu_chunk_seqlens = p.seq_idx = p.last_chunk_indices = FAKE
        p.io_dtype, p.meta_dtype, p.state_dtype = _abi.SSU_BF16, _abi.SSU_I64, _abi.SSU_F32
        p.tokens, p.nheads, p.headdim, p.dstate, p.ngroups = 512, 8, 64, 128, 2
        p.chunk_size, p.nchunks, p.batch = 256, 2, 1
        p.dt_min, p.dt_max = 0.0, float("inf")
        for k, v in over.items():
            setattr(p, k, v)
        return p

    need = lib.ssd_workspace_bytes(2, 8, 2, 64, 128, 256)
    assert need > 0 and lib.ssd_workspace_bytes(-1, 8, 2, 64, 128, 256) == -1
    call = lambda p, ws=FAKE, n=need: lib.ssd_combined_fwd_varlen(  # noqa: E731
        ctypes.byref(p), ws, n, None)
    assert call(params(headdim=32)) == _abi.SSU_ERR_UNSUPPORTED
    assert call(params(chunk_size=512)) == _abi.SSU_ERR_UNSUPPORTED
    assert call(params(chunk_size=0)) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call(params(ngroups=3)) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call(params(io_dtype=_abi.SSU_F32)) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call(params(nchunks=0)) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call(params(dt_min=1.0, dt_max=0.5)) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call(params(x=FAKE + 8)) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert call(params(states=FAKE + 8)) == _abi.SSU_ERR_INVALID_ARGUMENT   # vector stores
    assert call(params(initial_states=FAKE + 4, initial_dtype=_abi.SSU_F32)) == \
        _abi.SSU_ERR_INVALID_ARGUMENT
    assert call(params(nheads=65536 * 2, ngroups=2)) == _abi.SSU_ERR_UNSUPPORTED  # grid y
    assert call(params(nchunks=1 << 30)) == _abi.SSU_ERR_UNSUPPORTED
    assert call(params(), n=need - 1) == _abi.SSU_ERR_INVALID_ARGUMENT
    assert "workspace" in lib.ssu_last_error().decode()


def test_status_strings(lib):
    assert lib.ssu_status_string(0) == b"ok"
    assert lib.ssu_status_string(2) == b"unsupported"
    assert lib.ssu_status_string(99) == b"unknown status"


def test_python_binding_refuses_cpu_tensors():
    import torch

    import mamba2_ssm_decode_gb300 as m
    s = torch.zeros(2, 1, 4, 16)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        m.ssu_update(s, torch.zeros(2, 1, 4, dtype=torch.bfloat16), torch.zeros(2, 1),
                     torch.zeros(1), torch.zeros(2, 1, 16, dtype=torch.bfloat16),
                     torch.zeros(2, 1, 16, dtype=torch.bfloat16))
