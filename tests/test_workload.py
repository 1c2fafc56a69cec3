"""Closed-form work counters of the library against the oracle's brute-force counts."""

import pytest

import oracle
from oracle import RETRIEVAL, STREAMING
from streaming_kv_cache_duo_gb300 import workload as wl


@pytest.mark.parametrize("S,R", [(64, 256), (4, 32), (0, 1), (3, 5), (0, 7)])
@pytest.mark.parametrize("n,T", [(0, 1), (0, 300), (10, 50), (400, 123), (0, 1000)])
def test_pair_counts_match_brute_force(S, R, n, T):
    assert wl.causal_pairs(T, n) == oracle.visible_pair_count(T, RETRIEVAL, S, R, pos0=n)
    assert wl.streaming_pairs(T, S, R, n) == oracle.visible_pair_count(T, STREAMING, S, R, pos0=n)


def test_headline_counts():
    # one-shot prefill of 32768 tokens: causal pairs, and sink 64 / recent 256
    assert wl.causal_pairs(32768) == 536_887_296
    assert wl.streaming_pairs(32768, 64, 256) == 10_434_720
    fr, fs = wl.prefill_flops(1, 32, 8, 128, 64, 256, [1, 1, 1, 1, 0, 0, 0, 0], 32768)
    assert fr == 16 * 536_887_296 * 512
    assert fs == 16 * 10_434_720 * 512
    # chunked prefill of 8 x 4096 equals the one-shot count
    tot = sum(wl.causal_pairs(4096, 4096 * c) for c in range(8))
    assert tot == wl.causal_pairs(32768)
    tot = sum(wl.streaming_pairs(4096, 64, 256, 4096 * c) for c in range(8))
    assert tot == wl.streaming_pairs(32768, 64, 256)


@pytest.mark.parametrize("S,R", [(4, 32), (64, 256), (0, 3)])
def test_append_survivors(S, R):
    for n in [0, 1, S, S + R, 1000]:
        for T in [1, 3, R, R + 7, 5000]:
            assert wl.append_survivors(n, T, S, R) == len(oracle.append_survivors(n, T, S, R))
