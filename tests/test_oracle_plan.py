"""Pins for the oracle's chunk plan, strided membership and buffer bound (CPU only).

Values come from the pages (tests/golden/*.json, each with its citation) or
from invariants that eq. (1) and the strided-membership rule fix.
"""
import json
import os

import numpy as np
import pytest

from oracle import moe_ref as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _gold("chunk_plan.json")["cases"], ids=lambda c: f"N{c['N']}c{c['c']}K{c['K_max']}")
def test_chunk_plan_golden(case):
    assert O.chunk_plan(case["N"], case["c"], case["K_max"]) == (case["K"], case["c_eff"])


@pytest.mark.parametrize("N,c,K_max", [(1, 1, 1), (7, 2, 3), (100, 7, 16), (4096, 4096, 1), (65537, 4096, 16),
                                       (999, 1000, 5), (12345, 100, 1000)])
def test_chunk_plan_invariants(N, c, K_max):
    K, c_eff = O.chunk_plan(N, c, K_max)
    assert 1 <= K <= K_max
    assert K * (c_eff - 1) < N <= K * c_eff                   # c_eff is the smallest chunk size that covers N
    assert K == K_max or K * c >= N                           # K chunks of budget c cover N unless the cap binds
    assert K == 1 or (K - 1) * c < N                          # and no fewer chunks would do
    if -(-N // c) <= K_max:
        assert c_eff <= c                                     # the budget holds unless the cap binds


@pytest.mark.parametrize("N,K", [(512, 4), (1000, 3), (17, 16), (5, 1), (65536, 10)])
def test_strided_membership(N, K):
    seen = np.zeros(N, dtype=np.int64)
    sizes = []
    for i in range(K):
        toks = O.chunk_tokens(N, K, i)
        assert np.all(toks % K == i)                           # chunk i holds i, i+K, i+2K, ...
        assert np.all(np.diff(toks) == K)
        seen[toks] += 1
        sizes.append(len(toks))
    assert np.all(seen == 1)                                   # every token in exactly one chunk
    assert set(sizes) <= {N // K, -(-N // K)}
    assert max(sizes) == -(-N // K)


def test_buffer_bound_closed_form():
    g = _gold("buffer_bound.json")
    assert O.routed_bound_bytes(g["k"], g["c_eff"], g["H"], g["b"], g["E_p"]) == g["bytes"]


def test_dispatch_expansion_is_k_fold():
    """A chunk of n tokens expands to exactly k*n permuted rows (RelayMoE 2.2: 336 MiB -> ~2.6 GiB at top-8)."""
    g = _gold("dispatch_expansion.json")
    rng = np.random.default_rng(0)
    N, E, k, K = 96, 12, g["k"], 3
    idx = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    for i in range(K):
        rr, off, row_of = O.permute_chunk(idx, K, i, E)
        n = len(O.chunk_tokens(N, K, i))
        assert len(rr) == k * n and off[-1] == k * n
    gib = g["input_mib"] * g["k"] / 1024.0
    assert abs(gib - g["dispatch_gib_printed"]) <= g["rounding"]
