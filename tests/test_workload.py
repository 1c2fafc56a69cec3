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


@pytest.mark.parametrize("B,Hq,Hkv,D,S,R,kinds,n", [
    (1, 32, 8, 128, 64, 256, [1, 0, 0, 0, 0, 0, 1, 0], 1 << 20),
    (8, 32, 8, 128, 64, 256, [0, 1, 0, 0, 1, 0, 0, 0], 131073),
    (1, 4, 4, 64, 4, 32, [1, 0, 1, 0], 17),       # ring not yet full
    (2, 16, 2, 128, 0, 1, [0, 1], 5),             # window of one
    (1, 8, 4, 64, 8, 40, [0, 0, 0, 0], 1000),     # no retrieval head
])
def test_decode_bytes_count_what_the_cache_holds(B, Hq, Hkv, D, S, R, kinds, n):
    """Decode reads each held K and V row once per KV head: a retrieval head holds n
    rows, a streaming head the slots the ring model has filled after n appends (each
    with its int32 position), plus q and o; 4-bit rows are D / 2 bytes of codes and a
    4-byte (scale, zero) pair."""
    sim = oracle.RingCacheSim(S, R)
    sim.append(n)
    held = sum(1 for x in sim.positions() if x >= 0)
    n_ret = sum(kinds)
    n_str = Hkv - n_ret
    qo = 2 * B * Hq * D * 2
    assert wl.decode_bytes(B, Hq, Hkv, D, S, R, kinds, n) == (
        B * n_ret * n * 2 * D * 2, B * n_str * held * (2 * D * 2 + 4), qo)
    assert wl.decode_bytes_kv4(B, Hq, Hkv, D, S, R, kinds, n) == (
        B * n_ret * n * 2 * (D // 2 + 4), B * n_str * held * (2 * (D // 2 + 4) + 4), qo)


def test_decode_bytes_of_the_million_token_step():
    # 2 retrieval KV heads of 1,048,577 rows x 512 bytes (K + V, bf16, D 128) ~ 1.074 GB
    br, bs, bq = wl.decode_bytes(1, 32, 8, 128, 64, 256, [1, 1, 0, 0, 0, 0, 0, 0], 1048577)
    assert br == 2 * 1048577 * 512
    assert bs == 6 * 320 * 516 and bq == 2 * 32 * 128 * 2
    assert abs(br + bs + bq - 1.0748e9) < 1e6
