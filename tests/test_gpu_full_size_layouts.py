"""The million-token decode (1 sequence, 1,048,576 context tokens, 32 q / 8 kv heads,
D 128, 2 retrieval kv heads, sink 64 + ring 256) in the other cache layouts, built
exactly as the benchmark builds them (bench.make_layer: paged pools with a seeded
scattered block order, streaming heads in the pool, 4-bit caches) and filled by the
same 65536-token appends: sampled heads of the last decode step against the oracle."""

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


def test_full_size_decode_1m_kv4_sampled():
    """4-bit caches: two CTAs per SM, tensor-core slices on fp16 operands."""
    w, got = _run(use_kv4=True)
    _check(w, got, True)
