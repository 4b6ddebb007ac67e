"""Pins of the packed SSD prefill oracle (oracle/ssd.py).

Source: "mate.mamba", ssd_combined_fwd_varlen (the call contract and its five
stages; the stages' arithmetic is not printed).  The oracle is the one-token
recurrence run over each sequence's tokens; these tests tie it to things other
than itself:
  * the chunked matrix ("dual") form of SSD written out independently: within a
    chunk y_t = sum_{s<=t} e^{S_t - S_s} (C_t . B_s) dt'_s x_s + e^{S_t} C_t . h_in
    and h_out = e^{S_L} h_in + sum_s e^{S_L - S_s} dt'_s x_s (outer) B_s, with
    S_t the running sum of A dt' -- the five stages' mathematics;
  * invariance of every output to the chunking;
  * the entering-state rule (seq_idx is the authority) and the closed form of a
    sequence with x = 0;
  * closed forms of the dt clamp (applied after softplus);
  * agreement with the C oracle of the one-token update (a different
    implementation), states taken at chunk ends through its write-slot table.
"""
from __future__ import annotations

import importlib.util
import os

import numpy as np
import pytest
import torch

if os.environ.get("SSD_ORACLE_PATH"):   # a planted-mistake copy (test_oracle_ssd_mutations.py)
    _spec = importlib.util.spec_from_file_location("ssd_under_test", os.environ["SSD_ORACLE_PATH"])
    ssd = importlib.util.module_from_spec(_spec)
    _spec.loader.exec_module(ssd)
else:
    from oracle import ssd


def chunks(lengths, chunk_size):
    """cu_seqlens, cu_chunk_seqlens, seq_idx, last_chunk_indices of a packed batch."""
    cu, cuc, seq, last = [0], [0], [], []
    for b, L in enumerate(lengths):
        start, pos = cu[-1], 0
        while pos < L:
            n = min(chunk_size, L - pos)
            pos += n
            cuc.append(start + pos)
            seq.append(b)
        last.append(len(seq) - 1)
        cu.append(start + L)
    return [np.array(v, dtype=np.int64) for v in (cu, cuc, seq, last)]


def inputs(lengths, H=4, G=2, P=8, N=16, seed=0, with_init=True):
    rng = np.random.default_rng(seed)
    T = int(sum(lengths))
    return dict(
        x=rng.normal(size=(T, H, P)), dt=rng.normal(size=(T, H)),
        A=-np.exp(rng.uniform(0.0, np.log(16.0), size=H)),
        B=rng.normal(size=(T, G, N)), C=rng.normal(size=(T, G, N)),
        D=rng.uniform(0.0, 1.0, size=H), z=rng.normal(size=(T, H, P)),
        dt_bias=rng.uniform(-4.0, -1.0, size=H),
        initial_states=(0.1 * rng.normal(size=(len(lengths), H, P, N)) if with_init else None))


def run(inp, lengths, chunk_size, **kw):
    cu, cuc, seq, last = chunks(lengths, chunk_size)
    return ssd.ssd_combined_fwd_varlen(
        inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], chunk_size, cu, cuc, last, seq,
        D=inp["D"], z=inp["z"], dt_bias=inp["dt_bias"], dt_softplus=kw.get("softplus", True),
        dt_limit=kw.get("dt_limit", (0.0, np.inf)), initial_states=inp["initial_states"],
        return_intermediate_states=kw.get("intermediate", False))


def dual_form(inp, lengths, chunk_size, softplus=True, dt_limit=(0.0, np.inf)):
    """The chunked matrix form, written out independently of the oracle's loop."""
    x, dt, A, B, C = inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"]
    T, H, P = x.shape
    G = B.shape[1]
    grp = np.arange(H) // (H // G)
    _, cuc, seq, _ = chunks(lengths, chunk_size)
    out = np.zeros_like(x)
    states = []
    h_in = None
    for c in range(len(cuc) - 1):
        if c == 0 or seq[c] != seq[c - 1]:
            h_in = inp["initial_states"][seq[c]] if inp["initial_states"] is not None \
                else np.zeros((H, P, B.shape[2]))
        ts = np.arange(cuc[c], cuc[c + 1])
        d = dt[ts] + inp["dt_bias"][None, :]
        if softplus:
            d = np.log1p(np.exp(-np.abs(d))) + np.maximum(d, 0.0)
        d = np.clip(d, dt_limit[0], dt_limit[1])                          # [L, H]
        S = np.cumsum(A[None, :] * d, axis=0)                             # [L, H]
        Bt, Ct = B[ts][:, grp], C[ts][:, grp]                              # [L, H, N]
        u = d[:, :, None] * x[ts]                                         # [L, H, P]
        L = len(ts)
        mask = np.tril(np.ones((L, L)))
        decay = np.exp(S.T[:, :, None] - S.T[:, None, :]) * mask          # [H, t, s]
        CB = np.einsum("thn,shn->hts", Ct, Bt)
        y = np.einsum("hts,shp->thp", CB * decay, u)
        y += np.exp(S)[:, :, None] * np.einsum("thn,hpn->thp", Ct, h_in)
        y += inp["D"][None, :, None] * x[ts]
        zt = inp["z"][ts]
        out[ts] = y * (zt / (1.0 + np.exp(-zt)))
        h_out = np.exp(S[-1])[:, None, None] * h_in + np.einsum(
            "sh,shp,shn->hpn", np.exp(S[-1][None, :] - S), u, Bt)
        states.append(h_out)
        h_in = h_out
    return out, np.stack(states)


@pytest.mark.parametrize("lengths,chunk_size", [([9], 4), ([7, 12, 1], 4), ([16, 5], 8),
                                                ([3, 3, 3], 2)])
def test_matches_the_chunked_dual_form(lengths, chunk_size):
    inp = inputs(lengths, seed=len(lengths) + chunk_size)
    out, st = run(inp, lengths, chunk_size, intermediate=True)
    ref_out, ref_st = dual_form(inp, lengths, chunk_size)
    np.testing.assert_allclose(out, ref_out, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(st, ref_st, rtol=1e-10, atol=1e-12)


def test_outputs_do_not_depend_on_the_chunking():
    lengths = [11, 6]
    inp = inputs(lengths, seed=3)
    ref_out, ref_last = run(inp, lengths, 1)
    for cs in (2, 3, 5, 16):
        out, last = run(inp, lengths, cs)
        np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(last, ref_last, rtol=1e-12, atol=1e-13)


def test_intermediate_states_and_last_chunk_selection():
    lengths = [5, 9]
    inp = inputs(lengths, seed=4)
    _, every = run(inp, lengths, 4, intermediate=True)
    _, last = run(inp, lengths, 4)
    _, _, _, last_idx = chunks(lengths, 4)
    assert every.shape[0] == 5          # chunks of 4 + 1 and of 4 + 4 + 1 tokens
    np.testing.assert_array_equal(last, every[last_idx])


def test_entering_state_follows_seq_idx():
    lengths = [6, 7]
    inp = inputs(lengths, seed=5)
    out, last = run(inp, lengths, 4)
    # the second sequence does not see the first one's tokens
    other = {k: (v.copy() if v is not None else None) for k, v in inp.items()}
    other["x"][:6] += 1.0
    other["B"][:6] *= -2.0
    out2, last2 = run(other, lengths, 4)
    np.testing.assert_array_equal(out[6:], out2[6:])
    np.testing.assert_array_equal(last[1], last2[1])
    # ... and starts from its own initial state: with x = 0 the state only decays
    zero = {k: (v.copy() if v is not None else None) for k, v in inp.items()}
    zero["x"][:] = 0.0
    _, lz = run(zero, lengths, 4)
    d = zero["dt"][6:] + zero["dt_bias"][None, :]
    d = np.logaddexp(0.0, d)
    decay = np.exp((zero["A"][None, :] * d).sum(axis=0))
    np.testing.assert_allclose(lz[1], decay[:, None, None] * zero["initial_states"][1],
                               rtol=1e-12)


def test_dt_limit_clamps_after_softplus():
    lengths = [1]
    inp = inputs(lengths, seed=6, with_init=False)
    inp["z"] = np.full_like(inp["z"], 50.0)    # silu(50) = 50 (1 + e^-50)^-1
    inp["D"] = np.zeros_like(inp["D"])
    out, last = run(inp, lengths, 4, dt_limit=(0.25, 0.25))
    grp = np.arange(4) // 2
    h = 0.25 * inp["x"][0][:, :, None] * inp["B"][0][grp][:, None, :]
    np.testing.assert_allclose(last[0], h, rtol=1e-13)
    y = np.einsum("hpn,hn->hp", h, inp["C"][0][grp]) * (50.0 / (1.0 + np.exp(-50.0)))
    np.testing.assert_allclose(out[0], y, rtol=1e-12)
    # an upper limit below softplus(dt + dt_bias) caps it; a lower one lifts it
    sp = np.logaddexp(0.0, inp["dt"][0] + inp["dt_bias"])
    for lo, hi in ((0.0, float(sp.min()) / 2), (float(sp.max()) * 2, np.inf)):
        _, last = run(inp, lengths, 4, dt_limit=(lo, hi))
        d = np.clip(sp, lo, hi)
        h = d[:, None, None] * inp["x"][0][:, :, None] * inp["B"][0][grp][:, None, :]
        np.testing.assert_allclose(last[0], h, rtol=1e-13)


def test_agrees_with_the_one_token_oracle():
    """The same tokens through the C oracle of the packed one-token update: read
    slot b holds sequence b's initial state, and each chunk's last token writes
    its own slot, so the slots hold the chunk-end states (rounded to fp32)."""
    import oracle
    lengths = [6, 9, 3]
    chunk_size = 4
    H, G, P, N = 4, 2, 8, 16
    g = torch.Generator().manual_seed(7)
    T = sum(lengths)
    x = torch.randn(T, H, P, generator=g).to(torch.bfloat16)
    z = torch.randn(T, H, P, generator=g).to(torch.bfloat16)
    B = torch.randn(T, G, N, generator=g).to(torch.bfloat16)
    C = torch.randn(T, G, N, generator=g).to(torch.bfloat16)
    dt = torch.randn(T, H, generator=g)
    A = -torch.exp(torch.rand(H, generator=g) * float(np.log(16.0)))
    D = torch.rand(H, generator=g)
    dt_bias = -1.0 - 3.0 * torch.rand(H, generator=g)
    init = 0.1 * torch.randn(len(lengths), H, P, N, generator=g)
    cu, cuc, seq, last = chunks(lengths, chunk_size)
    nchunks = len(seq)
    pool = torch.zeros(len(lengths) + nchunks, H, P, N)
    pool[: len(lengths)] = init
    Lmax = max(lengths)
    dst = torch.full((len(lengths), Lmax), -1, dtype=torch.int64)
    for c in range(nchunks):
        b = int(seq[c])
        dst[b, int(cuc[c + 1]) - 1 - int(cu[b])] = len(lengths) + c
    src = torch.arange(len(lengths), dtype=torch.int64)[:, None]
    y_c = oracle.ssu_update_varlen(pool, x, dt, A, B, C, D=D, z=z, dt_bias=dt_bias,
                                   dt_softplus=True, cu_seqlens=torch.tensor(cu),
                                   state_batch_indices=src, dst_state_batch_indices=dst)
    out, every = ssd.ssd_combined_fwd_varlen(
        x, dt, A, B, C, chunk_size, cu, cuc, last, seq, D=D, z=z, dt_bias=dt_bias,
        dt_softplus=True, initial_states=init, return_intermediate_states=True)
    np.testing.assert_allclose(out, y_c.numpy().reshape(out.shape), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(pool[len(lengths):].double().numpy(), every, rtol=2e-7,
                               atol=1e-9)
