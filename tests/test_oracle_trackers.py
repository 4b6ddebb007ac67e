"""Pins of the oracle's ReplaySSM ring-tracker update / commit.

Source: "vllm.model_executor.layers.mamba.ops.ssu_dispatch", the kernels
_update_replayssm_ring_trackers_kernel and _commit_replayssm_ring_trackers_kernel
and their wrappers (update / reset / commit_replayssm_ring_trackers).

Pins: hand-worked cases of the printed kernels (tests/golden/ring_trackers.json),
the closed form of repeated single-token updates from a reset, the invariant
that a commit advances the ring's logical position (start + count) by exactly
the accepted count, and the validity mask.
"""
from __future__ import annotations

import itertools
import json
import os

import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ring_trackers.json")


def trackers(n, start=0, prev=0, pql=0):
    return (torch.full((n,), start, dtype=torch.int32), torch.full((n,), prev, dtype=torch.int32),
            torch.full((n,), pql, dtype=torch.int32))


def test_golden_cases(oracle_mod):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        rs, pna, pql = (torch.tensor([v], dtype=torch.int32) for v in c["before"])
        sbi = torch.tensor([0], dtype=torch.int32)
        if c["kernel"] == "update":
            oracle_mod.ring_update(rs, pna, pql, sbi, c["W"], c["Rb"])
        elif c["kernel"] == "reset":
            oracle_mod.ring_update(rs, pna, pql, sbi)
        else:
            oracle_mod.ring_commit(rs, pna, pql, sbi, torch.tensor([c["a"]]),
                                   torch.tensor([0, c["qlen"]]), c["W"], c["Rb"])
        got = [int(rs[0]), int(pna[0]), int(pql[0])]
        assert got == c["after"], (c, got)


@pytest.mark.parametrize("W", [0, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("Rb", [1, 2, 3, 7, 8, 9])
def test_repeated_updates_closed_form(oracle_mod, W, Rb):
    """From a reset, k single-token updates leave c = floor((k-1)/W) checkpoints:
    start = (c*W) mod Rb and count = k - c*W (W = 0: start = (k-1) mod Rb, count 1)."""
    rs, pna, pql = trackers(1, 5, 5, 3)
    sbi = torch.tensor([0])
    oracle_mod.ring_update(rs, pna, pql, sbi)
    assert (int(rs[0]), int(pna[0]), int(pql[0])) == (0, 0, 0)
    pql[0] = 7  # the update leaves prev_query_len alone
    for k in range(1, 40):
        oracle_mod.ring_update(rs, pna, pql, sbi, W, Rb)
        if W == 0:
            want = ((k - 1) % Rb, 1)
        else:
            c = (k - 1) // W
            want = ((c * W) % Rb, k - c * W)
        assert (int(rs[0]), int(pna[0])) == want, (k, W, Rb)
        assert int(pql[0]) == 7


def test_commit_invariants_exhaustive(oracle_mod):
    """Over a small domain: with a previous query (pql > 0) the logical position
    start + count advances by exactly the accepted count a (mod Rb); the ring
    moves only when acc + pql > W, and then the count restarts at a; with no
    previous query nothing moves and the count is 0; the new query length is
    always recorded."""
    for W, Rb in [(4, 8), (3, 5), (1, 2), (6, 4)]:
        dom = list(itertools.product(range(Rb), range(0, W + 2), range(0, 5), range(1, 5),
                                     range(0, 6)))
        n = len(dom)
        rs = torch.tensor([d[0] for d in dom], dtype=torch.int32)
        pna = torch.tensor([d[1] for d in dom], dtype=torch.int32)
        pql = torch.tensor([d[2] for d in dom], dtype=torch.int32)
        a = torch.tensor([d[3] for d in dom])
        qlen = torch.tensor([d[4] for d in dom])
        qsl = torch.zeros(n + 1, dtype=torch.int64)
        qsl[1:] = torch.cumsum(qlen, 0)
        r0, p0, q0 = rs.clone(), pna.clone(), pql.clone()
        oracle_mod.ring_commit(rs, pna, pql, torch.arange(n), a, qsl, W, Rb)
        for i in range(n):
            s, acc, pq, ai = int(r0[i]), int(p0[i]), int(q0[i]), int(a[i])
            assert int(pql[i]) == int(qlen[i])
            if pq == 0:
                assert (int(rs[i]), int(pna[i])) == (s, 0)
                continue
            assert (int(rs[i]) + int(pna[i])) % Rb == (s + acc + ai) % Rb
            moved = acc + pq > W
            if moved:
                assert int(pna[i]) == ai and 0 <= int(rs[i]) < Rb
            else:
                assert int(rs[i]) == s and int(pna[i]) == acc + ai


def test_update_invariant_exhaustive(oracle_mod):
    """Each non-reset update advances start + count by exactly one (mod Rb) and
    keeps the count within [1, max(W, 1)] once it starts inside [0, W]."""
    for W, Rb in [(4, 8), (2, 3), (5, 5)]:
        dom = list(itertools.product(range(Rb), range(0, W + 1)))
        n = len(dom)
        rs = torch.tensor([d[0] for d in dom], dtype=torch.int32)
        pna = torch.tensor([d[1] for d in dom], dtype=torch.int32)
        pql = torch.zeros(n, dtype=torch.int32)
        r0, p0 = rs.clone(), pna.clone()
        oracle_mod.ring_update(rs, pna, pql, torch.arange(n), W, Rb)
        for i in range(n):
            assert (int(rs[i]) + int(pna[i])) % Rb == (int(r0[i]) + int(p0[i]) + 1) % Rb
            assert 1 <= int(pna[i]) <= max(W, 1)


@pytest.mark.parametrize("pad", [-1, 3])
def test_validity_mask(oracle_mod, pad):
    """Pad, negative and >= num_states slots are skipped; num_states is the
    shortest tracker array; a 2-D table contributes its column 0."""
    rs = torch.arange(10, dtype=torch.int32) % 8
    pna = torch.full((12,), 4, dtype=torch.int32)
    pql = torch.full((11,), 2, dtype=torch.int32)
    table = torch.tensor([[1, 9], [pad, 1], [-2, 1], [10, 1], [9, 1], [5, 6]])
    before = (rs.clone(), pna.clone(), pql.clone())
    oracle_mod.ring_update(rs, pna, pql, table, 4, 8, pad_slot_id=pad)
    touched = {i for i in range(10) if int(rs[i]) != int(before[0][i]) or
               int(pna[i]) != int(before[1][i])}
    want = {1, 9, 5} - ({pad} if pad >= 0 else set())
    assert touched == want
    assert torch.equal(pna[10:], before[1][10:])

    rs2, pna2, pql2 = trackers(10, 1, 2, 3)
    b2 = (rs2.clone(), pna2.clone(), pql2.clone())
    oracle_mod.ring_commit(rs2, pna2, pql2, table, torch.full((6,), 1),
                           torch.arange(7) * 2, 4, 8, pad_slot_id=pad)
    touched = {i for i in range(10) if int(pql2[i]) != int(b2[2][i])}
    assert touched == want


def test_int32_wraparound(oracle_mod):
    """The tracker arithmetic is int32: sums wrap modulo 2^32, remainders
    truncate toward zero."""
    big = 2**31 - 1
    rs, pna, pql = (torch.tensor([v], dtype=torch.int32) for v in (big, 1, 1))
    oracle_mod.ring_commit(rs, pna, pql, torch.tensor([0]), torch.tensor([big]),
                           torch.tensor([0, 1]), 0, 7)
    # must: 1 + 1 > 0; start = (big + 1) wraps to -2^31, and -2^31 % 7 = -2
    assert int(rs[0]) == (-(2**31)) - 7 * int(-(2**31) / 7)
    assert int(pna[0]) == big
    rs, pna, pql = (torch.tensor([v], dtype=torch.int32) for v in (0, big, 0))
    oracle_mod.ring_update(rs, pna, pql, torch.tensor([0]), 4, 8)
    # prev + 1 wraps to -2^31, which is not > 4: the count becomes -2^31
    assert int(pna[0]) == -(2**31) and int(rs[0]) == 0
