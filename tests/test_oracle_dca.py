"""Pins of the oracle's Dual Chunk Attention (CPU only): the chunk-relation table written
from the page's wording, the definition against the page's brute-force schedule, and the
special cases that reduce to plain causal attention."""

import os

import numpy as np
import pytest

import oracle
import oracle.dca as dca
from oracle.attention import RETRIEVAL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(rng, T, Hq, Hkv, D):
    Q, QS, QI = (rng.standard_normal((T, Hq, D)) for _ in range(3))
    K, V = rng.standard_normal((T, Hkv, D)), rng.standard_normal((T, Hkv, D))
    ms = (0.5 + rng.random(T)).astype(np.float32)
    return Q, QS, QI, K, V, ms


def test_relation_table_from_the_page():
    code = {"I": dca.INTRA, "S": dca.SUCC, "X": dca.INTER}
    n = 0
    with open(os.path.join(GOLDEN, "dca_relation_chunk3.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            tok = line.split()
            i = int(tok[0][1:])
            assert len(tok) - 1 == i + 1
            for j, t in enumerate(tok[1:]):
                assert dca.relation(i, j, 3) == code[t], (i, j)
            n += 1
    assert n == 8


@pytest.mark.parametrize("T,chunk_len", [(9, 1), (10, 2), (11, 3), (17, 5), (16, 8), (7, 7), (6, 50)])
def test_definition_equals_the_bruteforce_schedule(T, chunk_len):
    rng = np.random.default_rng(T * 100 + chunk_len)
    args = _inputs(rng, T, 4, 2, 16)
    a = dca.attention(*args, chunk_len)
    b = dca.attention_bruteforce(*args, chunk_len)
    assert np.abs(a - b).max() < 1e-12


def test_one_query_and_unit_mscale_is_causal_attention():
    rng = np.random.default_rng(1)
    Q, _, _, K, V, _ = _inputs(rng, 13, 4, 2, 8)
    got = dca.attention(Q, Q, Q, K, V, np.ones(13, np.float32), 4)
    ref = oracle.prefill(Q, K, V, [RETRIEVAL, RETRIEVAL], 0, 1)
    assert np.abs(got - ref).max() < 1e-12


def test_single_chunk_ignores_succ_and_inter():
    rng = np.random.default_rng(2)
    Q, QS, QI, K, V, ms = _inputs(rng, 12, 2, 2, 8)
    a = dca.attention(Q, QS, QI, K, V, ms, 12)
    b = dca.attention(Q, QS * 3.0, -QI, K, V, ms, 12)
    assert np.array_equal(a, b)


def test_mscale_scales_the_product():
    # a constant mscale c equals queries scaled by c (exact arithmetic; fp64 to 1e-12)
    rng = np.random.default_rng(3)
    Q, QS, QI, K, V, _ = _inputs(rng, 10, 2, 1, 8)
    c = np.float32(1.375)
    a = dca.attention(Q, QS, QI, K, V, np.full(10, c), 3)
    b = dca.attention(Q * c, QS * c, QI * c, K, V, np.ones(10, np.float32), 3)
    assert np.abs(a - b).max() < 1e-12


def test_decode_equals_the_prefill_row():
    rng = np.random.default_rng(4)
    Q, QS, QI, K, V, ms = _inputs(rng, 14, 4, 2, 8)
    pre = dca.attention(Q, QS, QI, K, V, ms, 4)
    for p in (0, 3, 4, 8, 13):
        for h in range(4):
            d = dca.decode(Q[p, h], QS[p, h], QI[p, h], K[:p + 1, h // 2], V[:p + 1, h // 2], ms[p], p, 4)
            assert np.abs(d - pre[p, h]).max() < 1e-12


def test_planted_swap_of_succ_and_inter_fails(monkeypatch):
    real = dca.relation

    def swapped(i, j, chunk_len):
        r = real(i, j, chunk_len)
        return {dca.SUCC: dca.INTER, dca.INTER: dca.SUCC}.get(r, r)

    monkeypatch.setattr(dca, "relation", swapped)
    with pytest.raises(AssertionError):
        test_relation_table_from_the_page()
    with pytest.raises(AssertionError):
        test_definition_equals_the_bruteforce_schedule(11, 3)
