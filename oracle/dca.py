"""Dual Chunk Attention (DCA), float64 restatement. TEST INFRASTRUCTURE ONLY.

Source: vLLM pull request "[Model] Implement DualChunkAttention for Qwen2 Models".

* The sequence is cut into chunks; every position carries three query vectors
  (query, query_succ, query_inter) made by the rotary layer (outside this path).
* Query i attends causally to every key j <= i. Which query vector it uses depends
  on where j lies relative to i (the PR's reply on writing the kernel): the same
  chunk -> query; the chunk just before i's (the query sits in the succeeding
  chunk) -> query_succ; any earlier chunk -> query_inter.
* Chunk boundaries fall at multiples of chunk_len; the last chunk may be shorter
  (the PR's reply about the intra chunk), i.e. chunk(t) = t // chunk_len.
* The weight is (query . key) * softmax_scale * mscale[i] with mscale an fp32
  per-position factor applied to the product (the PR's reply on precision), then
  the usual softmax over j.
* The PR's brute-force version runs one attention per (query chunk, kind) -- intra,
  succ, inter -- and merges the partial softmaxes by their log-sum-exp.

``attention`` is the definition written out row by row; ``attention_bruteforce``
follows the PR's brute-force schedule. They share no arithmetic beyond the
library routines (a dot product, exp) and pin each other.
"""

from __future__ import annotations

import numpy as np

from .attention import lse_merge

INTRA, SUCC, INTER = 0, 1, 2


def relation(i: int, j: int, chunk_len: int) -> int:
    """Which query vector query position i uses for key position j <= i."""
    if chunk_len < 1 or j > i or j < 0:
        raise ValueError("need chunk_len >= 1 and 0 <= j <= i")
    ci, cj = i // chunk_len, j // chunk_len
    if ci == cj:
        return INTRA
    if ci == cj + 1:
        return SUCC
    return INTER


def attention(Q, QS, QI, K, V, mscale, chunk_len: int, rows=None, heads=None) -> np.ndarray:
    """One-shot causal DCA prefill. Q, QS, QI [T, Hq, D]; K, V [T, Hkv, D] at positions
    0 ... T-1; mscale [T] (float32 values, used exactly). Query head h uses KV head
    h // g. Returns O [len(rows), len(heads), D]."""
    Q, QS, QI = (np.asarray(x, np.float64) for x in (Q, QS, QI))
    K, V = np.asarray(K, np.float64), np.asarray(V, np.float64)
    ms = np.asarray(mscale, np.float64)
    T, Hq, D = Q.shape
    g = Hq // K.shape[1]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    heads = list(range(Hq) if heads is None else heads)
    scale = 1.0 / np.sqrt(D)
    out = np.empty((len(rows), len(heads), D))
    for c, h in enumerate(heads):
        hk = h // g
        for r, i in enumerate(rows):
            i = int(i)
            s = np.empty(i + 1)
            for j in range(i + 1):
                qv = (Q, QS, QI)[relation(i, j, chunk_len)][i, h]
                s[j] = (qv @ K[j, hk]) * scale * ms[i]
            e = np.exp(s - s.max())
            out[r, c] = e @ V[: i + 1, hk] / e.sum()
    return out


def _partial(q, keys, vals, factor):
    """(o, m, l) of one query over a key subset, scores (q . k) * factor."""
    s = (np.asarray(keys, np.float64) @ q) * factor
    m = s.max()
    e = np.exp(s - m)
    return e @ np.asarray(vals, np.float64), m, e.sum()


def attention_bruteforce(Q, QS, QI, K, V, mscale, chunk_len: int, rows=None, heads=None) -> np.ndarray:
    """The PR's brute-force schedule: for the chunk c of each query, one attention with
    query over chunk c (causal), one with query_succ over chunk c - 1 and one with
    query_inter over chunks 0 ... c - 2, merged by log-sum-exp."""
    Q, QS, QI = (np.asarray(x, np.float64) for x in (Q, QS, QI))
    K, V = np.asarray(K, np.float64), np.asarray(V, np.float64)
    ms = np.asarray(mscale, np.float64)
    T, Hq, D = Q.shape
    g = Hq // K.shape[1]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    heads = list(range(Hq) if heads is None else heads)
    out = np.empty((len(rows), len(heads), D))
    for c, h in enumerate(heads):
        hk = h // g
        for r, i in enumerate(rows):
            i = int(i)
            f = ms[i] / np.sqrt(D)
            start = (i // chunk_len) * chunk_len
            parts = [_partial(Q[i, h], K[start:i + 1, hk], V[start:i + 1, hk], f)]
            if start >= chunk_len:
                parts.append(_partial(QS[i, h], K[start - chunk_len:start, hk], V[start - chunk_len:start, hk], f))
            if start >= 2 * chunk_len:
                parts.append(_partial(QI[i, h], K[:start - chunk_len, hk], V[:start - chunk_len, hk], f))
            out[r, c] = lse_merge(parts)
    return out


def decode(q, qs, qi, keys, vals, mscale_p: float, p: int, chunk_len: int) -> np.ndarray:
    """One decode step of one query head at position p over keys/vals [p + 1, D] (the
    positions 0 ... p its KV head holds), by the definition."""
    q, qs, qi = (np.asarray(x, np.float64) for x in (q, qs, qi))
    keys, vals = np.asarray(keys, np.float64), np.asarray(vals, np.float64)
    D = q.shape[-1]
    s = np.array([((q, qs, qi)[relation(p, j, chunk_len)] @ keys[j]) for j in range(p + 1)])
    s = s * (1.0 / np.sqrt(D)) * float(mscale_p)
    e = np.exp(s - s.max())
    return e @ vals / e.sum()
