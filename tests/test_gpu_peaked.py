"""Parity on peaked attention rows, against the float64 oracle.

The DuoAttention README (Abstract) and the attention-sink issue describe real
attention rows as dominated by a few keys: the sinks, a few recent tokens, a few
retrieved ones. The kernels keep a running row maximum and rescale the running
output only when a later key tile's best score beats that maximum by more than 2^8
(log2 units); the bounded seeded generator alone never gets there after the first
tile. Every case here does, by one of four input recipes (the same bf16 values go to
both sides):

* ``qscale16``: queries times 16 (exact in bf16): score rows with a spread of ~23
  log2 units, so rows rescale many times, with every kind of factor;
* ``spikes``: every query row shifted along one dimension and a few keys pointing
  along it, planted at later positions with jumps of 9 ... 33 log2 units over the
  row's earlier maximum (some absorbed by the lazy rule, some rescaling);
* ``sink``: the first keys made dominant for every row (the attention-sink pattern);
* ``gauss``: queries, keys and values from torch's seeded normal generator (unbounded
  Gaussian tails; queries times 4).

Each retrieval-head case also checks, on the oracle's own scores, that its rows do take
the rescale after their first tile, with the keys before it still carrying weight.
"""

import numpy as np
import pytest
import torch

import duo_synth as ds
import oracle
import oracle.dca as dca
import oracle.kv4 as kv4
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import (LOG2E, assert_close, bf16_pair, decode_rescale_hits, host_stream, lazy_rescale_hits, plant,
                      to_np)

pytestmark = pytest.mark.gpu

TILE = 128  # keys per prefill and decode tile


def _gauss(seed, shape, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64).numpy() * scale


def _inputs(recipe, seed, B, P, Hq, Hkv, D, spike_pos=None, q0=0):
    """float64 Q [B, P - q0, Hq, D] (positions q0 ... P - 1), K and V [B, P, Hkv, D]
    holding bf16 values, and their device copies. spike_pos: list of (position, KV
    head, jump in log2 units)."""
    if recipe == "gauss":
        Q = _gauss(seed, (B, P - q0, Hq, D), 4.0)
        K = _gauss(seed + 1, (B, P, Hkv, D))
        V = _gauss(seed + 2, (B, P, Hkv, D))
    else:
        Q = host_stream(seed, ds.STREAM_Q, B, q0, P - q0, Hq, D)
        K = host_stream(seed, ds.STREAM_K, B, 0, P, Hkv, D)
        V = host_stream(seed, ds.STREAM_V, B, 0, P, Hkv, D)
        if recipe == "qscale16":
            Q *= 16.0
        elif recipe in ("spikes", "sink"):
            plant(Q, K, spike_pos, D)
    out = []
    for x in (Q, K, V):
        t, h = bf16_pair(x)
        out.append((t.cuda(), h))
    return out


def _prefill_spikes(recipe, seed, T, Hkv, S, R):
    rng = np.random.default_rng(seed)
    if recipe == "sink":
        # the first sink (and, with several sinks, the second) dominates every row
        return [(0, h, 12.0) for h in range(Hkv)] + ([(1, h, 10.0) for h in range(Hkv)] if S > 1 else [])
    spikes = []
    jumps = [9.0, 11.0, 13.5, 22.0, 24.0, 33.0]
    for h in range(Hkv):
        pos = np.sort(rng.choice(np.arange(TILE + 32, T), size=len(jumps), replace=False))
        spikes += [(int(p), h, j) for p, j in zip(pos, jumps)]
        # a spike inside the recent window of a few later rows of every streaming CTA
        spikes += [(int(p), h, 10.0) for p in range(TILE + 200, T, 3 * R + 17)]
    return spikes


def _scores_log2(q, k, D):
    return (q @ k.T) / np.sqrt(D) * LOG2E


PREFILL_CASES = [
    # recipe, B, Hq, Hkv, D, S, R, kinds, chunks
    ("qscale16", 1, 8, 2, 128, 4, 64, [1, 0], [1500]),
    ("qscale16", 1, 4, 4, 64, 16, 200, [0, 1, 0, 1], [600, 513, 387]),
    ("spikes", 2, 8, 2, 128, 4, 256, [1, 0], [1400]),
    ("spikes", 1, 8, 4, 64, 8, 300, [1, 0, 0, 1], [500, 700, 300]),
    ("sink", 1, 8, 2, 128, 64, 256, [1, 0], [1300]),
    ("sink", 1, 4, 2, 64, 4, 100, [0, 1], [400, 400, 333]),
    ("gauss", 1, 8, 2, 128, 64, 256, [1, 0], [1024, 700]),
    ("gauss", 1, 16, 2, 64, 4, 64, [0, 1], [900]),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[f"{c[0]}-{i}" for i, c in enumerate(PREFILL_CASES)])
def test_prefill_peaked_rows_match_oracle(case):
    """Prefill (one shot, or chunk by chunk against the growing cache) of retrieval and
    streaming heads on peaked rows: every row of every head against the oracle."""
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    recipe, B, Hq, Hkv, D, S, R, kinds, chunks = case
    T = sum(chunks)
    seed = 1200 + T + D
    (q, Qh), (k, Kh), (v, Vh) = _inputs(recipe, seed, B, T, Hq, Hkv, D, _prefill_spikes(recipe, seed, T, Hkv, S, R))
    layer = DuoLayer(B, Hq, Hkv, D, S, R, T, kinds)
    outs, t = [], 0
    for c in chunks:
        qs, ks, vs = (x[:, t:t + c].contiguous() for x in (q, k, v))
        outs.append(layer.prefill(qs, ks, vs))
        layer.append(ks, vs)
        t += c
    torch.cuda.synchronize()
    assert duo_device_error() == 0
    got = to_np(torch.cat(outs, dim=1))
    for b in range(B):
        assert_close(got[b], oracle.prefill(Qh[b], Kh[b], Vh[b], kinds, S, R), f"{recipe} b{b}")

    g = Hq // Hkv
    rows = np.arange(T)
    causal = rows[None, :] <= rows[:, None]
    if recipe == "sink":
        # the attention-sink pattern: most of every row's weight on the first keys
        for hq in range(Hq):
            s = np.where(causal, _scores_log2(Qh[0, :, hq], Kh[0, :, hq // g], D), -np.inf)
            w = np.exp2(s - s.max(axis=1, keepdims=True))
            assert np.median(w[:, :2].sum(axis=1) / w.sum(axis=1)) > 0.9
        return
    # the rows of retrieval heads take the rescale after their first tile; tiles as the
    # kernel visits them: the cache rows before each chunk, then the chunk's tiles
    n0 = np.repeat(np.cumsum([0] + chunks[:-1]), chunks)  # cache length before each row's chunk
    hit_rows = 0
    for hq in [h for h in range(Hq) if kinds[h // g]]:
        s = np.where(causal, _scores_log2(Qh[0, :, hq], Kh[0, :, hq // g], D), -np.inf)
        for c0, c in zip(np.cumsum([0] + chunks[:-1]), chunks):
            keys = np.arange(c0 + c)
            tile = np.where(keys < c0, keys // TILE, -(-c0 // TILE) + (keys - c0) // TILE)
            sel = n0 == c0
            hits, share = lazy_rescale_hits(s[sel][:, :c0 + c], tile)
            hit_rows += int(((hits > 0) & (share > 1e-2)).sum())
    assert hit_rows >= 20, f"only {hit_rows} rows rescale with weight left before the new maximum"


def _decode_spikes(seed, ctx, Hkv, kinds, R):
    rng = np.random.default_rng(seed)
    spikes = []
    for h in range(Hkv):
        if kinds[h]:
            pos = rng.choice(np.arange(2000, ctx), size=40, replace=False)
            spikes += [(int(p), h, float(j)) for p, j in zip(pos, rng.uniform(9.0, 12.0, 40))]
        else:  # inside the window the decode steps see, and one sink
            spikes += [(ctx - R // 2, h, 9.0), (ctx - 3, h, 20.0), (0, h, 5.0)]
    return spikes


def _decode_layer_run(layer, k, v, q, ctx, steps, decode):
    """Append ctx tokens, then per step append one token and decode q[:, step]."""
    for c0 in range(0, ctx, 65536):
        T = min(65536, ctx - c0)
        layer.append(k[:, c0:c0 + T].contiguous(), v[:, c0:c0 + T].contiguous())
    outs = []
    for s in range(steps):
        p = ctx + s
        layer.append(k[:, p:p + 1].contiguous(), v[:, p:p + 1].contiguous())
        outs.append(decode(q[:, s].contiguous()))
    torch.cuda.synchronize()
    return [to_np(o) for o in outs]


def _check_decode_coverage(q, Kh, kinds, D, n_ctas, p, recipe):
    """Retrieval units' per-warp streams of the decode at position p (queries q [B, Hq,
    D]) rescale after their first slice (the work split as the decode kernel documents it)."""
    B, Hq, _ = q.shape
    Hkv = len(kinds)
    g = Hq // Hkv
    units = [_scores_log2(q[b, h * g:(h + 1) * g], Kh[b, :p + 1, h], D)
             for b in range(B) for h in range(Hkv) if kinds[h]]
    n_str = B * (Hkv - sum(kinds))
    if units:
        hits = decode_rescale_hits(units, p + 1, n_ctas, n_str)
        assert hits >= 4, f"{recipe}: only {hits} per-warp streams rescale"


DECODE_CASES = [
    # recipe, B, Hq, Hkv, D, S, R, kinds, ctx, steps
    ("qscale16", 1, 2, 2, 128, 4, 64, [1, 0], 60000, 2),    # g = 1: CUDA-core consumer
    ("spikes", 1, 2, 2, 128, 4, 64, [1, 0], 60000, 2),
    ("qscale16", 2, 4, 2, 64, 8, 100, [1, 0], 40000, 2),    # g = 2
    ("spikes", 2, 4, 2, 64, 8, 100, [0, 1], 40000, 2),
    ("qscale16", 1, 8, 2, 128, 64, 256, [1, 0], 60000, 2),  # g = 4: tensor-core slices
    ("spikes", 1, 8, 2, 128, 64, 256, [1, 0], 60000, 2),
    ("qscale16", 1, 16, 2, 64, 4, 64, [0, 1], 60000, 2),    # g = 8
    ("gauss", 1, 16, 2, 128, 4, 64, [1, 0], 60000, 2),
    ("gauss", 1, 4, 4, 128, 64, 256, [1, 0, 0, 1], 40000, 2),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=[f"{c[0]}-g{c[2] // c[3]}-{i}" for i, c in enumerate(DECODE_CASES)])
def test_decode_peaked_rows_match_oracle(case):
    """Decode steps over long caches (several tiles per CTA, so a warp's later slices
    can beat its earlier ones) on peaked rows, both consumers, against the oracle."""
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    recipe, B, Hq, Hkv, D, S, R, kinds, ctx, steps = case
    seed = 1300 + ctx % 997 + Hq
    total = ctx + steps
    (q, Qh), (k, Kh), (v, Vh) = _inputs(recipe, seed, B, total, Hq, Hkv, D, _decode_spikes(seed, ctx, Hkv, kinds, R),
                                        q0=ctx)
    layer = DuoLayer(B, Hq, Hkv, D, S, R, total, kinds)
    outs = _decode_layer_run(layer, k, v, q, ctx, steps, layer.decode)
    assert duo_device_error() == 0
    for b in range(B):
        cache = OracleCache(kinds, S, R, D)
        cache.append(Kh[b, :ctx], Vh[b, :ctx])
        for s in range(steps):
            p = ctx + s
            cache.append(Kh[b, p:p + 1], Vh[b, p:p + 1])
            assert_close(outs[s][b], decode_from_cache(Qh[b, s], p, cache), f"{recipe} b{b} step {s}")
    n_ctas = torch.cuda.get_device_properties(0).multi_processor_count
    _check_decode_coverage(Qh[:, 0], Kh, kinds, D, n_ctas, ctx, recipe)


KV4_CASES = [
    # recipe, B, Hq, Hkv, D, S, R, kinds, ctx, steps
    ("qscale16", 1, 8, 2, 128, 4, 64, [1, 0], 120000, 2),   # g = 4
    ("spikes", 1, 16, 2, 64, 8, 100, [1, 0], 120000, 2),    # g = 8, D 64
    ("spikes", 2, 4, 2, 128, 4, 64, [1, 1], 60000, 2),      # g = 2
    ("gauss", 1, 2, 2, 128, 64, 256, [1, 0], 120000, 2),    # g = 1
]


@pytest.mark.parametrize("case", KV4_CASES, ids=[f"{c[0]}-g{c[2] // c[3]}-{i}" for i, c in enumerate(KV4_CASES)])
def test_kv4_decode_peaked_rows_match_oracle(case):
    """4-bit caches: decode on peaked rows against the oracle attending over the
    dequantized rows (the lazy rescale also scales the per-head zero-point sums)."""
    from streaming_kv_cache_duo_gb300 import DuoKv4Layer, duo_device_error
    recipe, B, Hq, Hkv, D, S, R, kinds, ctx, steps = case
    seed = 1400 + ctx % 991 + Hq
    total = ctx + steps
    (q, Qh), (k, Kh), (v, Vh) = _inputs(recipe, seed, B, total, Hq, Hkv, D, _decode_spikes(seed, ctx, Hkv, kinds, R),
                                        q0=ctx)
    layer = DuoKv4Layer(B, Hq, Hkv, D, S, R, total, kinds)
    outs = _decode_layer_run(layer, k, v, q, ctx, steps, layer.decode)
    assert duo_device_error() == 0
    Kq, Vq = kv4.roundtrip(Kh.astype(np.float32)), kv4.roundtrip(Vh.astype(np.float32))
    for b in range(B):
        cache = OracleCache(kinds, S, R, D)
        cache.append(Kq[b, :ctx], Vq[b, :ctx])
        for s in range(steps):
            p = ctx + s
            cache.append(Kq[b, p:p + 1], Vq[b, p:p + 1])
            assert_close(outs[s][b], decode_from_cache(Qh[b, s], p, cache), f"{recipe} b{b} step {s}")
    n_ctas = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    _check_decode_coverage(Qh[:, 0], Kq, kinds, D, n_ctas, ctx, recipe)


def _dca_inputs(seed, B, P, Hq, Hkv, D, scale):
    out = []
    for s, H, f in ((ds.STREAM_Q, Hq, scale), (ds.STREAM_Q_SUCC, Hq, scale), (ds.STREAM_Q_INTER, Hq, scale),
                    (ds.STREAM_K, Hkv, 1.0), (ds.STREAM_V, Hkv, 1.0)):
        t, h = bf16_pair(host_stream(seed, s, B, 0, P, H, D) * f)
        out.append((t.cuda(), h))
    return out


def test_dca_prefill_peaked_rows_match_oracle():
    """Dual Chunk Attention prefill with all three query vectors times 16 (exact),
    five chunks with a ragged last one: every row against oracle.dca."""
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    B, Hq, Hkv, D, T, CL = 1, 4, 2, 128, 1100, 256
    seed = 1501
    (q, Qh), (qs, QSh), (qi, QIh), (k, Kh), (v, Vh) = _dca_inputs(seed, B, T, Hq, Hkv, D, 16.0)
    ms = ds.dca_mscale(B, T, CL)
    layer = DuoLayer(B, Hq, Hkv, D, 0, 1, T, [1] * Hkv)
    o = layer.dca_prefill(q, qs, qi, k, v, CL, mscale=torch.from_numpy(ms).cuda())
    torch.cuda.synchronize()
    assert duo_device_error() == 0
    assert_close(to_np(o)[0], dca.attention(Qh[0], QSh[0], QIh[0], Kh[0], Vh[0], ms[0], CL), "dca prefill")


def test_dca_decode_peaked_rows_match_oracle():
    """Dual Chunk Attention decode over 40000 cached tokens (chunks of 8192) with the
    query vectors times 16: several key tiles per CTA, against oracle.dca."""
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    B, Hq, Hkv, D, ctx, CL, steps = 1, 8, 2, 128, 40000, 8192, 2
    seed = 1502
    total = ctx + steps
    (q, Qh), (qs, QSh), (qi, QIh), (k, Kh), (v, Vh) = _dca_inputs(seed, B, total, Hq, Hkv, D, 16.0)
    ms = ds.dca_mscale(B, total, CL)
    msd = torch.from_numpy(ms).cuda()
    layer = DuoLayer(B, Hq, Hkv, D, 0, 1, total, [1] * Hkv)
    layer.append(k[:, :ctx].contiguous(), v[:, :ctx].contiguous())
    g = Hq // Hkv
    for s in range(steps):
        p = ctx + s
        layer.append(k[:, p:p + 1].contiguous(), v[:, p:p + 1].contiguous())
        o = layer.dca_decode(q[:, p].contiguous(), qs[:, p].contiguous(), qi[:, p].contiguous(), CL,
                             mscale=msd[:, p].contiguous())
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        ref = np.stack([dca.decode(Qh[0, p, h], QSh[0, p, h], QIh[0, p, h], Kh[0, :p + 1, h // g],
                                   Vh[0, :p + 1, h // g], ms[0, p], p, CL) for h in range(Hq)])
        assert_close(to_np(o[0]), ref, f"dca decode step {s}")
