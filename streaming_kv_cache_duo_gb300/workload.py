"""Algorithmic work of the hot path, in closed form (for throughput and roofline numbers).

FLOPs count 4 * D per visible (query, key) pair per query head: 2 * D for q.k
and 2 * D for p * v; masked pairs and partially masked tiles are not counted.
Bytes count what the method must move at least once: for decode, the K and V
bytes of every stored key once per KV head (all its query heads share them),
the ring positions, plus q and o; for append, the rows read and written.
"""

from __future__ import annotations


def causal_pairs(T: int, n: int = 0) -> int:
    """Visible pairs of a retrieval head: queries n ... n+T-1, each sees keys 0 ... i."""
    return T * n + T * (T + 1) // 2


def streaming_pairs(T: int, S: int, R: int, n: int = 0) -> int:
    """Visible pairs of a streaming head (j <= i and (j < S or i - j < R)), queries n ... n+T-1.

    Row i sees min(i + 1, S + R) keys: all earlier keys until the sinks and the
    window stop overlapping, then S sinks plus R recent keys."""
    K = S + R
    lo, hi = n, n + T
    a_hi = min(hi, K)  # rows with i + 1 <= K
    growing = (a_hi * (a_hi + 1) - lo * (lo + 1)) // 2 if a_hi > lo else 0
    flat = (hi - max(lo, K)) * K if hi > max(lo, K) else 0
    return growing + flat


def prefill_flops(B, Hq, Hkv, D, S, R, is_retrieval, T, n=0):
    """(retrieval FLOPs, streaming FLOPs) of one prefill of T tokens after n cached ones."""
    g = Hq // Hkv
    n_ret = sum(1 for x in is_retrieval if x)
    n_str = Hkv - n_ret
    return (4 * D * B * g * n_ret * causal_pairs(T, n), 4 * D * B * g * n_str * streaming_pairs(T, S, R, n))


def append_survivors(n, T, S, R):
    """Tokens of an append of T after n that a streaming head still holds afterwards."""
    e = n + T
    sinks = max(0, min(e, S) - n)
    ring = max(0, e - max(n, S, e - R))
    return sinks + ring


def decode_bytes(B, Hq, Hkv, D, S, R, is_retrieval, n):
    """(retrieval bytes, streaming bytes, q + o bytes) of one decode step with n keys stored."""
    n_ret = sum(1 for x in is_retrieval if x)
    n_str = Hkv - n_ret
    row = 2 * D * 2  # K and V rows, bf16
    return B * n_ret * n * row, B * n_str * min(n, S + R) * (row + 4), 2 * B * Hq * D * 2


def decode_bytes_kv4(B, Hq, Hkv, D, S, R, is_retrieval, n):
    """decode_bytes for 4-bit caches: a K or V row is D / 2 bytes of codes plus a
    4-byte (scale, zero) pair."""
    n_ret = sum(1 for x in is_retrieval if x)
    n_str = Hkv - n_ret
    row = 2 * (D // 2 + 4)
    return B * n_ret * n * row, B * n_str * min(n, S + R) * (row + 4), 2 * B * Hq * D * 2


def append_bytes(B, Hkv, D, S, R, is_retrieval, n, T):
    """Bytes read plus written by one append of T tokens after n stored ones."""
    n_ret = sum(1 for x in is_retrieval if x)
    n_str = Hkv - n_ret
    surv = append_survivors(n, T, S, R)
    row = 2 * D * 2
    return 2 * B * (n_ret * T + n_str * surv) * row + B * surv * 4
