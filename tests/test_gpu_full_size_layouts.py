"""Full-size parity in the cache layouts the benchmark also times, each layer built
exactly as the benchmark builds it (bench.make_layer: paged pools with a seeded
scattered block order, streaming heads in the pool, 4-bit caches, 4-bit caches in a pool):
- the million-token decode (1 sequence, 1,048,576 context tokens, 32 q / 8 kv heads,
  D 128, 2 retrieval kv heads, sink 64 + ring 256), filled by the same 65536-token
  appends: sampled heads of the last decode step against the oracle;
- the 8 x 4096 chunked prefill: sampled rows of every chunk against the oracle."""

import numpy as np
import pytest
import torch

import duo_synth as ds
import oracle
import oracle.kv4 as kv4
from gpu_util import assert_close, head_keys, to_np

pytestmark = pytest.mark.gpu

STEPS = 2


def _run(paged_block=0, pool=False, use_kv4=False):
    import bench
    from streaming_kv_cache_duo_gb300 import duo_device_error
    w = ds.WORKLOADS["decode_ctx1m"]
    dev = torch.device("cuda", torch.cuda.current_device())
    layer = bench.make_layer(w, w.context + STEPS, dev, paged_block, pool, use_kv4)
    for c0 in range(0, w.context, 65536):
        layer.append(ds.stream_torch(w.seed, ds.STREAM_K, w.B, c0, 65536, w.Hkv, w.D, device=dev),
                     ds.stream_torch(w.seed, ds.STREAM_V, w.B, c0, 65536, w.Hkv, w.D, device=dev))
    q = ds.stream_torch(w.seed, ds.STREAM_Q, w.B, w.context, STEPS, w.Hq, w.D, device=dev)
    kn = ds.stream_torch(w.seed, ds.STREAM_K, w.B, w.context, STEPS, w.Hkv, w.D, device=dev)
    vn = ds.stream_torch(w.seed, ds.STREAM_V, w.B, w.context, STEPS, w.Hkv, w.D, device=dev)
    for s in range(STEPS):
        layer.append(kn[:, s:s + 1].contiguous(), vn[:, s:s + 1].contiguous())
        o = layer.decode(q[:, s].contiguous())
    torch.cuda.synchronize()
    assert duo_device_error() == 0
    return w, to_np(o)


def _check(w, got, use_kv4):
    """Head 0 of each kind and one more streaming head, at the last step's position."""
    g = w.Hq // w.Hkv
    p = w.context + STEPS - 1
    Qp = ds.stream_f64(w.seed, ds.STREAM_Q, w.B, p, 1, w.Hq, w.D)[0, 0]
    ret = [h for h in range(w.Hkv) if w.is_retrieval[h]]
    strm = [h for h in range(w.Hkv) if not w.is_retrieval[h]]
    for h in ret[:1] + strm[:2]:
        if w.is_retrieval[h]:
            K, V = head_keys(w.seed, 0, h, 0, p + 1, w.D)
            kpos = np.arange(p + 1)
        else:
            sim = oracle.RingCacheSim(w.S, w.R)
            sim.append(p + 1)
            kpos = np.array([x for x in sim.positions() if x >= 0])
            K = np.stack([ds.stream_f64(w.seed, ds.STREAM_K, w.B, int(t), 1, w.Hkv, w.D)[0, 0, h] for t in kpos])
            V = np.stack([ds.stream_f64(w.seed, ds.STREAM_V, w.B, int(t), 1, w.Hkv, w.D)[0, 0, h] for t in kpos])
        if use_kv4:  # the cache holds the 4-bit rows: attend over what it holds
            K, V = kv4.roundtrip(K.astype(np.float32)), kv4.roundtrip(V.astype(np.float32))
        ref = oracle.attend_rows(Qp[h * g:(h + 1) * g], [p] * g, K, V, kpos, w.is_retrieval[h], w.S, w.R)
        assert_close(got[0, h * g:(h + 1) * g], ref, f"kv head {h}")


def test_full_size_decode_1m_paged_sampled():
    """Retrieval caches in a pool of 256-token blocks in a scattered order."""
    w, got = _run(paged_block=256)
    _check(w, got, False)


def test_full_size_decode_1m_pool_sampled():
    """Both head kinds in the pool (streaming heads' blocks past the window untouched)."""
    w, got = _run(paged_block=256, pool=True)
    _check(w, got, False)


def test_full_size_decode_1m_kv4_paged_sampled():
    """4-bit retrieval rows in a pool of 256-token blocks in a scattered order."""
    w, got = _run(paged_block=256, use_kv4=True)
    _check(w, got, True)


def test_full_size_decode_1m_kv4_sampled():
    """4-bit caches: two CTAs per SM, tensor-core slices on fp16 operands."""
    w, got = _run(use_kv4=True)
    _check(w, got, True)


def _chunked(paged_block, pool):
    """llama2-7B-shaped chunked prefill (32768 tokens in 8 chunks of 4096, 32 / 32 heads,
    8 retrieval heads, sink 64 / recent 256) into a layer built by bench.make_layer;
    returns the workload, the sampled rows and their outputs [rows, Hq, D]."""
    import bench
    from streaming_kv_cache_duo_gb300 import duo_device_error
    w = ds.WORKLOADS["llama2_7b_chunked_prefill32k"]
    dev = torch.device("cuda", torch.cuda.current_device())
    L, C = w.prefill_len, w.chunk
    layer = bench.make_layer(w, L, dev, paged_block, pool)
    rng = np.random.default_rng(5)
    rows, got = [], []
    for c0 in range(0, L, C):
        q = ds.stream_torch(w.seed, ds.STREAM_Q, w.B, c0, C, w.Hq, w.D, device=dev)
        k = ds.stream_torch(w.seed, ds.STREAM_K, w.B, c0, C, w.Hkv, w.D, device=dev)
        v = ds.stream_torch(w.seed, ds.STREAM_V, w.B, c0, C, w.Hkv, w.D, device=dev)
        o = layer.prefill(q, k, v)
        r = np.unique([0, 1, 255, 256, C - 1] + list(rng.integers(0, C, 2)))
        got.append(to_np(o[0, r]))
        rows += list(c0 + r)
        layer.append(k, v)
    torch.cuda.synchronize()
    assert duo_device_error() == 0
    return w, np.array(rows), np.concatenate(got)


def _check_chunked(w, rows, got):
    L = w.prefill_len
    ret = [h for h in range(w.Hkv) if w.is_retrieval[h]]
    strm = [h for h in range(w.Hkv) if not w.is_retrieval[h]]
    for h in ret[:2] + strm[:3]:  # MHA: query head h uses KV head h
        K, V = head_keys(w.seed, 0, h, 0, L, w.D)
        Q = ds.stream_f64(w.seed, ds.STREAM_Q, 1, 0, L, h + 1, w.D, heads=[h], batches=[0])[0, :, 0]
        ref = oracle.attend_rows(Q[rows], rows, K, V, np.arange(L), w.is_retrieval[h], w.S, w.R)
        assert_close(got[:, h], ref, f"head {h}")


def test_full_size_chunked_prefill_paged_sampled():
    """Chunked prefill reading the retrieval cache from scattered 256-token blocks."""
    _check_chunked(*_chunked(256, False))


def test_full_size_chunked_prefill_pool_sampled():
    """Chunked prefill with both head kinds in the pool."""
    _check_chunked(*_chunked(256, True))
