"""Seeded random shapes through the whole path (chunked prefill against the growing
cache, appends, decode steps) against the float64 oracle: batch, head counts and
grouping, head_dim, sink and window sizes, which KV heads are retrieval heads, chunk
lengths and the number of decode steps are all drawn from a fixed generator, so the
cases are the same on every run but cover combinations no hand-written case lists."""

import numpy as np
import pytest
import torch

import duo_synth as ds
import oracle
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import assert_close, device_stream, host_stream, to_np

pytestmark = pytest.mark.gpu


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 4))
    Hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8]))
    D = int(rng.choice([64, 128]))
    S = int(rng.integers(0, 70))
    R = int(rng.integers(1, 400))
    kinds = [int(x) for x in rng.integers(0, 2, Hkv)]
    chunks = [int(x) for x in rng.integers(1, 700, int(rng.integers(1, 4)))]
    steps = int(rng.integers(1, 4))
    return B, Hkv * g, Hkv, D, S, R, kinds, chunks, steps


@pytest.mark.parametrize("seed", range(12))
def test_random_shape_matches_oracle(seed):
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    B, Hq, Hkv, D, S, R, kinds, chunks, steps = _case(seed)
    total = sum(chunks) + steps
    layer = DuoLayer(B, Hq, Hkv, D, S, R, total, kinds)
    ks = 77 + seed
    Q = device_stream(ks, ds.STREAM_Q, B, 0, total, Hq, D, "cuda")
    K = device_stream(ks, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    V = device_stream(ks, ds.STREAM_V, B, 0, total, Hkv, D, "cuda")
    Qh = host_stream(ks, ds.STREAM_Q, B, 0, total, Hq, D)
    Kh = host_stream(ks, ds.STREAM_K, B, 0, total, Hkv, D)
    Vh = host_stream(ks, ds.STREAM_V, B, 0, total, Hkv, D)
    rng = np.random.default_rng(seed)
    t = 0
    for T in chunks:
        q, k, v = (x[:, t:t + T].contiguous() for x in (Q, K, V))
        o = layer.prefill(q, k, v)
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        # every row of short chunks; boundary and random rows of longer ones
        rows = np.arange(T) if T <= 64 else np.unique(np.concatenate(
            [[0, 1, T - 2, T - 1], rng.integers(0, T, 24)]))
        got = to_np(o)[:, rows]
        for b in range(B):
            ref = oracle.prefill(Qh[b, :t + T], Kh[b, :t + T], Vh[b, :t + T], kinds, S, R, rows=rows + t)
            assert_close(got[b], ref, f"case {_case(seed)} chunk at {t} b{b}")
        layer.append(k, v)
        t += T
    for s in range(steps):
        layer.append(K[:, t:t + 1].contiguous(), V[:, t:t + 1].contiguous())
        o = layer.decode(Q[:, t].contiguous())
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        for b in range(B):
            cache = OracleCache(kinds, S, R, D)
            cache.append(Kh[b, :t + 1], Vh[b, :t + 1])
            assert_close(to_np(o[b]), decode_from_cache(Qh[b, t], t, cache), f"case {_case(seed)} decode {s} b{b}")
        t += 1


@pytest.mark.parametrize("seed", range(6))
def test_random_shape_pool_layout_matches_oracle(seed):
    """The same random cases with both head kinds in the paged pool (256-token blocks),
    the caller freeing every block the library names dead."""
    from test_gpu_paged_stream import Allocator, _layer
    from streaming_kv_cache_duo_gb300 import duo_device_error
    B, Hq, Hkv, D, S, R, kinds, chunks, steps = _case(seed)
    total = sum(chunks) + steps
    bs = 256
    max_blocks = -(-total // bs)
    num_blocks = B * Hkv * max_blocks + 4
    layer = _layer(B, Hq, Hkv, D, S, R, kinds, bs, max_blocks, num_blocks)
    alloc = Allocator(layer, num_blocks, seed=seed)
    ks = 77 + seed
    Q = device_stream(ks, ds.STREAM_Q, B, 0, total, Hq, D, "cuda")
    K = device_stream(ks, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    V = device_stream(ks, ds.STREAM_V, B, 0, total, Hkv, D, "cuda")
    Qh = host_stream(ks, ds.STREAM_Q, B, 0, total, Hq, D)
    Kh = host_stream(ks, ds.STREAM_K, B, 0, total, Hkv, D)
    Vh = host_stream(ks, ds.STREAM_V, B, 0, total, Hkv, D)
    t = 0
    for T in chunks:
        q, k, v = (x[:, t:t + T].contiguous() for x in (Q, K, V))
        o = layer.prefill(q, k, v)
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        rows = np.unique(np.array([0, T // 2, T - 1]))
        for b in range(B):
            ref = oracle.prefill(Qh[b, :t + T], Kh[b, :t + T], Vh[b, :t + T], kinds, S, R, rows=rows + t)
            assert_close(to_np(o)[b, rows], ref, f"pool case {_case(seed)} chunk at {t} b{b}")
        alloc.before_append(t, T)
        layer.append(k, v)
        t += T
        alloc.after_append(t)
    for s in range(steps):
        alloc.before_append(t, 1)
        layer.append(K[:, t:t + 1].contiguous(), V[:, t:t + 1].contiguous())
        alloc.after_append(t + 1)
        o = layer.decode(Q[:, t].contiguous())
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        for b in range(B):
            cache = OracleCache(kinds, S, R, D)
            cache.append(Kh[b, :t + 1], Vh[b, :t + 1])
            assert_close(to_np(o[b]), decode_from_cache(Qh[b, t], t, cache), f"pool case {_case(seed)} decode {s}")
        t += 1


@pytest.mark.parametrize("seed", range(6))
def test_random_shape_kv4_decode_matches_oracle(seed):
    """The same random cases appended into 4-bit caches and decoded, against the oracle
    attending over the dequantized rows."""
    import oracle.kv4 as kv4
    from streaming_kv_cache_duo_gb300 import DuoKv4Layer, duo_device_error
    B, Hq, Hkv, D, S, R, kinds, chunks, steps = _case(seed)
    total = sum(chunks) + steps
    layer = DuoKv4Layer(B, Hq, Hkv, D, S, R, total, kinds)
    ks = 77 + seed
    Q = device_stream(ks, ds.STREAM_Q, B, 0, total, Hq, D, "cuda")
    K = device_stream(ks, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    V = device_stream(ks, ds.STREAM_V, B, 0, total, Hkv, D, "cuda")
    Qh = host_stream(ks, ds.STREAM_Q, B, 0, total, Hq, D)
    Kq = kv4.roundtrip(host_stream(ks, ds.STREAM_K, B, 0, total, Hkv, D).astype(np.float32))
    Vq = kv4.roundtrip(host_stream(ks, ds.STREAM_V, B, 0, total, Hkv, D).astype(np.float32))
    t = 0
    for T in chunks:
        layer.append(K[:, t:t + T].contiguous(), V[:, t:t + T].contiguous())
        t += T
    for s in range(steps):
        layer.append(K[:, t:t + 1].contiguous(), V[:, t:t + 1].contiguous())
        o = layer.decode(Q[:, t].contiguous())
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        for b in range(B):
            cache = OracleCache(kinds, S, R, D)
            cache.append(Kq[b, :t + 1], Vq[b, :t + 1])
            assert_close(to_np(o[b]), decode_from_cache(Qh[b, t], t, cache), f"kv4 case {_case(seed)} decode {s}")
        t += 1
