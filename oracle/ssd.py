"""Plain fp64 oracle of the packed SSD prefill ("mate.mamba",
``ssd_combined_fwd_varlen``).

TEST INFRASTRUCTURE ONLY: like the rest of this package it is imported by the
tests alone; no product code uses it.  It shares no code with the CUDA library.

The pages give this call's contract (argument shapes, the chunk metadata and
which of them is the authority) and the names of its five stages, but not the
stages' arithmetic.  The plainest reading, taken here: the call computes what
the one-token update computes, token by token over each sequence in order --

    dt' = dt[t, h] + dt_bias[h];  dt' = softplus(dt') if dt_softplus
    dt' = min(max(dt', dt_limit[0]), dt_limit[1])
    dA  = exp(A[h] dt')
    h   <- h dA + dt' x[t, h, :] (outer) B[t, g, :]
    y[t, h, :] = h C[t, g, :] + D x[t, h, :];   y *= silu(z[t, h, :]) with z

-- and the state after chunk ``c`` is ``states[c]``.  Chunk ``c`` covers tokens
``[cu_chunk_seqlens[c], cu_chunk_seqlens[c + 1])``; it opens a sequence when
``seq_idx[c]`` differs from ``seq_idx[c - 1]`` (the pages make ``seq_idx`` the
authority), and then starts from ``initial_states[seq_idx[c]]`` (zeros without
initial states); otherwise it continues from the previous chunk's state.  The
result is ``(out, states)``: every chunk's state when
``return_intermediate_states``, else ``states[last_chunk_indices]``.

Pins: tests/test_oracle_ssd.py (the chunked matrix form of SSD written out
independently, invariance to the chunking, the entering-state rule, closed
forms of the dt clamp, agreement with the C oracle of the one-token update).
"""
from __future__ import annotations

import math

import numpy as np


def _f64(t):
    if t is None:
        return None
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        import torch
        return t.to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def _ints(t):
    if hasattr(t, "detach"):
        t = t.detach().cpu().numpy()
    return np.asarray(t, dtype=np.int64)


def softplus(v):
    """log(1 + e^v) with no cutoff (logaddexp is that function, without overflow)."""
    return np.logaddexp(0.0, v)


def ssd_combined_fwd_varlen(x, dt, A, B, C, chunk_size, cu_seqlens, cu_chunk_seqlens,
                            last_chunk_indices, seq_idx, D=None, z=None, dt_bias=None,
                            dt_softplus=False, dt_limit=(0.0, math.inf), initial_states=None,
                            return_intermediate_states=False):
    """x [tokens, H, P], dt [tokens, H], A [H], B / C [tokens, G, N], D [H] or
    [H, P], z [tokens, H, P], dt_bias [H], initial_states [batch, H, P, N];
    returns (out [tokens, H, P], states), both float64 numpy arrays."""
    x, dt, A, B, C = _f64(x), _f64(dt), _f64(A), _f64(B), _f64(C)
    D, z, dt_bias, h0 = _f64(D), _f64(z), _f64(dt_bias), _f64(initial_states)
    cu_chunk = _ints(cu_chunk_seqlens)
    seq = _ints(seq_idx)
    last = _ints(last_chunk_indices)
    tokens, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    if H % G or chunk_size <= 0:
        raise ValueError("heads must be divisible by groups; chunk_size must be positive")
    group = np.arange(H) // (H // G)
    Dv = None if D is None else (D[:, None] if D.ndim == 1 else D)  # [H, 1] or [H, P]
    lo, hi = dt_limit
    nchunks = len(cu_chunk) - 1
    out = np.zeros((tokens, H, P))
    states = np.zeros((nchunks, H, P, N))
    h = np.zeros((H, P, N))
    for c in range(nchunks):
        if c == 0 or seq[c] != seq[c - 1]:   # the chunk opens sequence seq[c]
            h = h0[seq[c]].copy() if h0 is not None else np.zeros((H, P, N))
        for t in range(cu_chunk[c], cu_chunk[c + 1]):
            d = dt[t] + (dt_bias if dt_bias is not None else 0.0)
            if dt_softplus:
                d = softplus(d)
            d = np.minimum(np.maximum(d, lo), hi)
            dA = np.exp(A * d)
            Bt, Ct = B[t][group], C[t][group]                        # [H, N]
            h = h * dA[:, None, None] + (d[:, None] * x[t])[:, :, None] * Bt[:, None, :]
            y = np.einsum("hpn,hn->hp", h, Ct)
            if Dv is not None:
                y = y + Dv * x[t]
            if z is not None:
                y = y * (z[t] / (1.0 + np.exp(-z[t])))
            out[t] = y
        states[c] = h
    return out, (states if return_intermediate_states else states[last])
