"""Pins of the oracle's attention (CPU only): brute force, closed forms, a library
routine (torch's scaled_dot_product_attention in float64) and invariants."""

import numpy as np
import pytest
import torch

import oracle
import oracle.attention as oa
from oracle import (RETRIEVAL, STREAMING, attention_dense_mask, attend_rows, prefill,
                    prefill_chunked, lse_merge, partial_softmax, visible_pair_count)
from oracle.attention import OracleCache, decode_from_cache


def _rng(seed=0):
    return np.random.default_rng(seed)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


def _visible_intervals(i, kind, S, R):
    """Closed form of the visible set as two intervals (independent of is_visible)."""
    if kind == RETRIEVAL:
        return list(range(0, i + 1))
    sink = set(range(0, min(S, i + 1)))
    recent = set(range(max(0, i - R + 1), i + 1))
    return sorted(sink | recent)


def _sdpa_f64(Q, K, V, mask):
    q = torch.from_numpy(Q)[None, None]
    k = torch.from_numpy(K)[None, None]
    v = torch.from_numpy(V)[None, None]
    m = torch.from_numpy(mask)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m)[0, 0].numpy()


CASES = [(STREAMING, 4, 32), (STREAMING, 0, 1), (STREAMING, 0, 7), (STREAMING, 3, 5), (STREAMING, 64, 256),
         (RETRIEVAL, 4, 32)]


@pytest.mark.parametrize("kind,S,R", CASES)
@pytest.mark.parametrize("pos0", [0, 9])
def test_dense_mask_equals_row_gather(kind, S, R, pos0):
    rng = _rng(1)
    L, D = 48, 16
    Q = _bf16(rng.standard_normal((L, D)))
    K = _bf16(rng.standard_normal((pos0 + L, D)))
    V = _bf16(rng.standard_normal((pos0 + L, D)))
    a = attention_dense_mask(Q, K, V, kind, S, R, pos0=pos0)
    b = attend_rows(Q, pos0 + np.arange(L), K, V, np.arange(pos0 + L), kind, S, R)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


@pytest.mark.parametrize("kind,S,R", CASES)
def test_equal_keys_give_mean_of_visible_values(kind, S, R):
    # With every key equal, all scores tie and O_i is the plain mean of the
    # visible values: this pins the membership and size of every visible set.
    rng = _rng(2)
    L, D = 70, 8
    Q = rng.standard_normal((L, D))
    K = np.tile(rng.standard_normal((1, D)), (L, 1))
    V = rng.standard_normal((L, D))
    out = attend_rows(Q, np.arange(L), K, V, np.arange(L), kind, S, R)
    for i in range(L):
        want = V[_visible_intervals(i, kind, S, R)].mean(axis=0)
        np.testing.assert_allclose(out[i], want, rtol=0, atol=1e-12)


def test_window_of_one_returns_own_value():
    rng = _rng(3)
    L, D = 33, 8
    Q, K, V = (rng.standard_normal((L, D)) for _ in range(3))
    out = attend_rows(Q, np.arange(L), K, V, np.arange(L), STREAMING, 0, 1)
    np.testing.assert_array_equal(out, V)


@pytest.mark.parametrize("S,R", [(4, 28), (0, 32), (16, 40), (31, 1)])
def test_streaming_with_large_budget_is_causal(S, R):
    rng = _rng(4)
    L, D = 32, 16
    Q, K, V = (rng.standard_normal((L, D)) for _ in range(3))
    a = attend_rows(Q, np.arange(L), K, V, np.arange(L), STREAMING, S, R)
    b = attend_rows(Q, np.arange(L), K, V, np.arange(L), RETRIEVAL, S, R)
    assert S + R >= L
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("kind,S,R", CASES)
def test_against_torch_sdpa_float64(kind, S, R):
    rng = _rng(5)
    L, D = 96, 32
    Q, K, V = (rng.standard_normal((L, D)) for _ in range(3))
    i = torch.arange(L)[:, None]
    j = torch.arange(L)[None, :]
    mask = j <= i
    if kind == STREAMING:
        mask &= (j < S) | (i - j < R)
    want = _sdpa_f64(Q, K, V, mask.numpy())
    got = attend_rows(Q, np.arange(L), K, V, np.arange(L), kind, S, R)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    if kind == RETRIEVAL:
        q, k, v = (torch.from_numpy(x)[None, None] for x in (Q, K, V))
        causal = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)[0, 0].numpy()
        np.testing.assert_allclose(got, causal, rtol=0, atol=1e-12)


def test_planted_window_mistake_fails_pins(monkeypatch):
    # Off-by-one in the recent window (i - j <= R) must break the closed forms.
    orig = oa.attend_rows

    def bad(q_rows, q_pos, keys, vals, key_pos, kind, S, R):
        return orig(q_rows, q_pos, keys, vals, key_pos, kind, S, R + 1)

    monkeypatch.setattr(oa, "attend_rows", bad)
    rng = _rng(3)
    L, D = 20, 8
    Q, K, V = (rng.standard_normal((L, D)) for _ in range(3))
    out = oa.attend_rows(Q, np.arange(L), K, V, np.arange(L), STREAMING, 0, 1)
    assert not np.array_equal(out, V)


def test_planted_scale_mistake_fails_sdpa(monkeypatch):
    monkeypatch.setattr(oa, "_softmax_attend",
                        lambda q, k, v: (lambda e: (e @ v) / e.sum())(np.exp(k @ q - (k @ q).max())))
    rng = _rng(5)
    L, D = 24, 32
    Q, K, V = (rng.standard_normal((L, D)) for _ in range(3))
    mask = np.tril(np.ones((L, L), dtype=bool))
    got = oa.attend_rows(Q, np.arange(L), K, V, np.arange(L), RETRIEVAL, 0, 1)
    assert np.abs(got - _sdpa_f64(Q, K, V, mask)).max() > 1e-3


@pytest.mark.parametrize("kinds", [[RETRIEVAL, STREAMING], [STREAMING, STREAMING], [RETRIEVAL, RETRIEVAL]])
def test_gqa_equals_mha_with_repeated_kv(kinds):
    rng = _rng(6)
    T, Hq, Hkv, D, S, R = 40, 8, 2, 16, 3, 9
    Q = rng.standard_normal((T, Hq, D))
    K = rng.standard_normal((T, Hkv, D))
    V = rng.standard_normal((T, Hkv, D))
    g = Hq // Hkv
    a = prefill(Q, K, V, kinds, S, R)
    Kr = np.repeat(K, g, axis=1)
    Vr = np.repeat(V, g, axis=1)
    b = prefill(Q, Kr, Vr, np.repeat(kinds, g), S, R)
    np.testing.assert_array_equal(a, b)
    # and each head separately is plain single-head attention on KV head h // g
    for h in range(Hq):
        c = attend_rows(Q[:, h], np.arange(T), K[:, h // g], V[:, h // g], np.arange(T), kinds[h // g], S, R)
        np.testing.assert_array_equal(a[:, h], c)


def test_lse_merge_of_any_partition_equals_unsplit():
    rng = _rng(7)
    N, D = 500, 64
    q = rng.standard_normal(D) * 3
    K = rng.standard_normal((N, D))
    V = rng.standard_normal((N, D))
    whole = attend_rows(q[None], [N - 1], K, V, np.arange(N), RETRIEVAL, 0, 1)[0]
    for trial in range(5):
        cuts = np.sort(rng.choice(np.arange(1, N), size=trial * 3 + 1, replace=False))
        parts = [partial_softmax(q, K[a:b], V[a:b]) for a, b in zip([0, *cuts], [*cuts, N])]
        np.testing.assert_allclose(lse_merge(parts), whole, rtol=0, atol=1e-12)
    # a permuted, non-contiguous partition too
    perm = rng.permutation(N)
    parts = [partial_softmax(q, K[perm[k::3]], V[perm[k::3]]) for k in range(3)]
    np.testing.assert_allclose(lse_merge(parts), whole, rtol=0, atol=1e-12)


@pytest.mark.parametrize("S,R", [(4, 32), (2, 5), (0, 3)])
def test_decode_equals_prefill_row_and_reads_only_the_cache(S, R):
    rng = _rng(8)
    T, Hq, Hkv, D = 90, 4, 2, 16
    kinds = [RETRIEVAL, STREAMING]
    Q = rng.standard_normal((T, Hq, D))
    K = rng.standard_normal((T, Hkv, D))
    V = rng.standard_normal((T, Hkv, D))
    full = prefill(Q, K, V, kinds, S, R)
    cache = OracleCache(kinds, S, R, D)
    for p in range(T):
        cache.append(K[p:p + 1], V[p:p + 1])
        got = decode_from_cache(Q[p], p, cache)
        np.testing.assert_allclose(got, full[p], rtol=0, atol=1e-13)
    # the streaming head holds S + R rows, the retrieval head all T
    assert cache.view(1)[0].shape[0] == min(T, S + R)
    assert cache.view(0)[0].shape[0] == T


@pytest.mark.parametrize("chunk", [1, 7, 32, 64, 200])
def test_chunked_prefill_equals_one_shot(chunk):
    rng = _rng(9)
    T, Hq, Hkv, D, S, R = 130, 4, 4, 16, 4, 32
    kinds = [RETRIEVAL, STREAMING, RETRIEVAL, STREAMING]
    Q = rng.standard_normal((T, Hq, D))
    K = rng.standard_normal((T, Hkv, D))
    V = rng.standard_normal((T, Hkv, D))
    a = prefill(Q, K, V, kinds, S, R)
    b = prefill_chunked(Q, K, V, kinds, S, R, chunk)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_visible_pair_counts():
    # causal: L(L+1)/2; streaming: rows i < S+R see i+1 keys, later rows S+R
    for L in [1, 5, 64, 300, 1000]:
        assert visible_pair_count(L, RETRIEVAL, 64, 256) == L * (L + 1) // 2
        for S, R in [(64, 256), (4, 32), (0, 1)]:
            k = min(L, S + R)
            want = k * (k + 1) // 2 + (L - k) * (S + R)
            assert visible_pair_count(L, STREAMING, S, R) == want
    # brute force over the dense mask on a tiny case
    L, S, R = 40, 3, 6
    dense = sum(oracle.is_visible(i, j, STREAMING, S, R) for i in range(L) for j in range(L))
    assert visible_pair_count(L, STREAMING, S, R) == dense


def test_empty_visible_set_is_an_error():
    with pytest.raises(ValueError):
        attend_rows(np.zeros((1, 4)), [0], np.zeros((1, 4)), np.zeros((1, 4)), np.array([-1]), RETRIEVAL, 0, 1)
