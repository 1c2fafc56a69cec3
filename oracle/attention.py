"""Masked softmax attention of retrieval and streaming heads, in float64 on the CPU.

Source: DuoAttention README (mit-han-lab/duo-attention), Abstract. Retrieval
heads keep a full KV cache and attend to every earlier token; streaming heads
keep a small fixed-length cache and attend to the attention sinks and the
recent tokens only. Read as a rule on absolute positions (query i, key j):

    retrieval:  j <= i
    streaming:  j <= i  and  (j < S  or  i - j < R)

S = sink_size, R = recent_size (the quick start uses S = 64, R = 256); the
recent window counts the current token, so it is (i - R, i].

Attention of query i of head h (KV head h // g, g = Hq / Hkv) is the plain
softmax over the visible keys with scale D**-0.5:

    s_j = (q_i . k_j) / sqrt(D),   O_i = sum_j exp(s_j - max) v_j / sum_j exp(s_j - max)

Decode (the transformers pull request "[WIP] Dynamic length in static cache")
attends only to positions up to the current one, never to cache slots beyond
the current length. Partial softmaxes over disjoint key sets are merged by
their log-sum-exp, as the vLLM Dual Chunk Attention pull request merges its
``*_softmax_lse`` outputs.
"""

from __future__ import annotations

import numpy as np

from .ring_cache import RingCacheSim

RETRIEVAL = 1
STREAMING = 0


def is_visible(i: int, j: int, kind: int, S: int, R: int) -> bool:
    """Key position j is visible to query position i for a head of this kind."""
    if j < 0 or j > i:
        return False
    if kind == RETRIEVAL:
        return True
    return j < S or i - j < R


def visible_keys(i: int, kind: int, S: int, R: int) -> np.ndarray:
    """All visible key positions of query i, by testing every j in [0, i]."""
    return np.array([j for j in range(i + 1) if is_visible(i, j, kind, S, R)], dtype=np.int64)


def visible_pair_count(L: int, kind: int, S: int, R: int, pos0: int = 0) -> int:
    """Number of (query, key) pairs a prefill of queries pos0 ... pos0+L-1 attends to."""
    total = 0
    for i in range(pos0, pos0 + L):
        j = np.arange(i + 1)
        if kind == RETRIEVAL:
            total += i + 1
        else:
            total += int(np.count_nonzero((j < S) | (i - j < R)))
    return total


def _softmax_attend(q: np.ndarray, keys: np.ndarray, vals: np.ndarray) -> np.ndarray:
    D = q.shape[-1]
    s = keys @ q / np.sqrt(D)
    e = np.exp(s - s.max())
    return (e @ vals) / e.sum()


def attention_dense_mask(Q, K, V, kind: int, S: int, R: int, pos0: int = 0) -> np.ndarray:
    """Brute force: build the full boolean mask element by element, then softmax.

    Q [Lq, D] are queries at positions pos0 ... pos0+Lq-1; K, V [Lk, D] are keys
    at positions 0 ... Lk-1. Tiny inputs only."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    Lq, D = Q.shape
    Lk = K.shape[0]
    mask = np.zeros((Lq, Lk), dtype=bool)
    for r in range(Lq):
        for j in range(Lk):
            mask[r, j] = is_visible(pos0 + r, j, kind, S, R)
    scores = (Q @ K.T) / np.sqrt(D)
    scores = np.where(mask, scores, -np.inf)
    scores = scores - scores.max(axis=1, keepdims=True)
    w = np.exp(scores)
    w /= w.sum(axis=1, keepdims=True)
    return w @ V


def attend_rows(q_rows, q_pos, keys, vals, key_pos, kind: int, S: int, R: int) -> np.ndarray:
    """Per-row gather: for each query, take the keys whose position is visible, softmax.

    ``key_pos`` gives each key row's absolute position (-1 = empty slot, never
    visible). Keys may come in any order (a ring cache is rotated)."""
    q_rows = np.asarray(q_rows, np.float64)
    keys = np.asarray(keys, np.float64)
    vals = np.asarray(vals, np.float64)
    key_pos = np.asarray(key_pos, np.int64)
    out = np.empty_like(q_rows)
    for r, i in enumerate(q_pos):
        i = int(i)
        vis = (key_pos >= 0) & (key_pos <= i)
        if kind != RETRIEVAL:
            vis &= (key_pos < S) | (i - key_pos < R)
        if not vis.any():
            raise ValueError(f"query {i} sees no key")
        out[r] = _softmax_attend(q_rows[r], keys[vis], vals[vis])
    return out


def prefill(Q, K, V, kinds, S: int, R: int, rows=None, heads=None) -> np.ndarray:
    """One-shot prefill. Q [T, Hq, D], K/V [T, Hkv, D] at positions 0 ... T-1.

    ``kinds[h_kv]`` is RETRIEVAL or STREAMING; query head h uses KV head h // g.
    Returns O [len(rows), len(heads), D] (all rows / heads by default)."""
    Q = np.asarray(Q, np.float64)
    T, Hq, D = Q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    rows = np.arange(T) if rows is None else np.asarray(rows)
    heads = range(Hq) if heads is None else heads
    heads = list(heads)
    out = np.empty((len(rows), len(heads), D))
    pos = np.arange(T)
    for c, h in enumerate(heads):
        hk = h // g
        out[:, c] = attend_rows(Q[rows, h], rows, K[:, hk], V[:, hk], pos, kinds[hk], S, R)
    return out


def prefill_chunked(Q, K, V, kinds, S: int, R: int, chunk: int) -> np.ndarray:
    """Chunked prefill against a growing cache (same shapes as ``prefill``).

    For a chunk at positions [s, s+C): a retrieval head attends to its full
    cache (positions [0, s)) plus the chunk; a streaming head attends to what its
    sink + ring cache holds before the chunk plus the chunk. Then the chunk is
    appended to the caches."""
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    T, Hq, D = Q.shape
    Hkv = K.shape[1]
    g = Hq // Hkv
    out = np.empty_like(Q)
    rings = [RingCacheSim(S, R) for _ in range(Hkv)]
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        cpos = np.arange(s, e)
        for hk in range(Hkv):
            if kinds[hk] == RETRIEVAL:
                keys, vals, kpos = K[:e, hk], V[:e, hk], np.arange(e)
            else:
                ring = rings[hk]
                slots = ring.valid_slots()
                ck = np.array([ring.payload[x][0] for x in slots]).reshape(-1, D)
                cv = np.array([ring.payload[x][1] for x in slots]).reshape(-1, D)
                keys = np.concatenate([ck, K[s:e, hk]])
                vals = np.concatenate([cv, V[s:e, hk]])
                kpos = np.concatenate([np.array([ring.pos[x] for x in slots], np.int64), cpos])
            for h in range(hk * g, (hk + 1) * g):
                out[s:e, h] = attend_rows(Q[s:e, h], cpos, keys, vals, kpos, kinds[hk], S, R)
        for hk in range(Hkv):
            if kinds[hk] != RETRIEVAL:
                rings[hk].append(e - s, [(K[t, hk], V[t, hk]) for t in range(s, e)])
    return out


class OracleCache:
    """What the caches of one sequence hold: every row for retrieval heads, a sink +
    ring ``RingCacheSim`` (payload = (k, v)) for streaming heads."""

    def __init__(self, kinds, S: int, R: int, D: int):
        self.kinds, self.S, self.R, self.D = list(kinds), S, R, D
        self.full_k = {h: [] for h, k in enumerate(kinds) if k == RETRIEVAL}
        self.full_v = {h: [] for h, k in enumerate(kinds) if k == RETRIEVAL}
        self.rings = {h: RingCacheSim(S, R) for h, k in enumerate(kinds) if k != RETRIEVAL}
        self.n = 0

    def append(self, K, V) -> None:
        """K, V [T, Hkv, D] for positions n ... n+T-1."""
        K = np.asarray(K, np.float64)
        V = np.asarray(V, np.float64)
        T = K.shape[0]
        for h in self.full_k:
            self.full_k[h].extend(K[:, h])
            self.full_v[h].extend(V[:, h])
        for h, ring in self.rings.items():
            ring.append(T, [(K[t, h], V[t, h]) for t in range(T)])
        self.n += T

    def view(self, h: int):
        """(keys, values, positions) of KV head h as stored."""
        if h in self.full_k:
            return (np.array(self.full_k[h]).reshape(-1, self.D), np.array(self.full_v[h]).reshape(-1, self.D),
                    np.arange(len(self.full_k[h])))
        ring = self.rings[h]
        slots = ring.valid_slots()
        return (np.array([ring.payload[s][0] for s in slots]).reshape(-1, self.D),
                np.array([ring.payload[s][1] for s in slots]).reshape(-1, self.D),
                np.array([ring.pos[s] for s in slots], np.int64))


def decode_from_cache(q, p: int, cache: OracleCache) -> np.ndarray:
    """Decode step at position p, after token p has been appended: q [Hq, D] -> O [Hq, D],
    reading keys only from what ``cache`` holds (not from the full history)."""
    q = np.asarray(q, np.float64)
    Hq, D = q.shape
    Hkv = len(cache.kinds)
    g = Hq // Hkv
    out = np.empty_like(q)
    for hk in range(Hkv):
        keys, vals, kpos = cache.view(hk)
        out[hk * g:(hk + 1) * g] = attend_rows(q[hk * g:(hk + 1) * g], [p] * g, keys, vals, kpos,
                                               cache.kinds[hk], cache.S, cache.R)
    return out


def partial_softmax(q, keys, vals):
    """Unnormalised partial softmax of one query over a key subset: (o, m, l) with
    m = max score, l = sum exp(s - m), o = sum exp(s - m) v."""
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    s = keys @ q / np.sqrt(q.shape[-1])
    m = s.max()
    e = np.exp(s - m)
    return e @ np.asarray(vals, np.float64), m, e.sum()


def lse_merge(parts) -> np.ndarray:
    """Merge partial softmaxes over disjoint key sets into the full softmax output."""
    M = max(m for _, m, _ in parts)
    num = sum(np.exp(m - M) * o for o, m, _ in parts)
    den = sum(np.exp(m - M) * l for _, m, l in parts)
    return num / den
