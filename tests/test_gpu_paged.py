"""Paged retrieval caches: the same appends, chunked prefills and decodes through a
block table over a shared pool give bit-identical results to the contiguous layout
(and so the same parity with the oracle), whatever the block order."""

import numpy as np
import pytest
import torch

import duo_synth as ds
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import assert_close, device_stream, host_stream, to_np

pytestmark = pytest.mark.gpu


def _layers(B, Hq, Hkv, D, S, R, kinds, block_size, max_blocks, seed=0):
    from streaming_kv_cache_duo_gb300 import DuoLayer, DuoPagedLayer
    n_ret = sum(kinds)
    num_blocks = B * n_ret * max_blocks + 3  # a few blocks nobody uses
    rng = np.random.default_rng(seed)
    ids = rng.permutation(num_blocks)[:B * n_ret * max_blocks].reshape(B, n_ret, max_blocks)
    table = torch.tensor(ids, dtype=torch.int32, device="cuda")
    paged = DuoPagedLayer(B, Hq, Hkv, D, S, R, block_size, max_blocks, num_blocks, table, kinds)
    paged.k_full.fill_(float("nan"))  # unwritten rows must never be read
    paged.v_full.fill_(float("nan"))
    contig = DuoLayer(B, Hq, Hkv, D, S, R, block_size * max_blocks, kinds)
    return paged, contig, ids


@pytest.mark.parametrize("block_size", [128, 256])
def test_paged_equals_contiguous(block_size):
    B, Hq, Hkv, D, S, R = 2, 8, 4, 128, 4, 64
    kinds = [1, 0, 1, 0]
    chunks = [300, 100, 37, 400]
    steps = 3
    total = sum(chunks) + steps
    max_blocks = -(-total // block_size)
    paged, contig, ids = _layers(B, Hq, Hkv, D, S, R, kinds, block_size, max_blocks)
    seed = 21
    Q = device_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D, "cuda")
    K = device_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    V = device_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D, "cuda")
    t = 0
    for T in chunks:
        q, k, v = (x[:, t:t + T].contiguous() for x in (Q, K, V))
        a = paged.prefill(q, k, v)
        b = contig.prefill(q, k, v)
        torch.cuda.synchronize()
        assert torch.equal(a, b), f"prefill chunk at {t}"
        paged.append(k, v)
        contig.append(k, v)
        t += T
    for s in range(steps):
        k, v = K[:, t:t + 1].contiguous(), V[:, t:t + 1].contiguous()
        paged.append(k, v)
        contig.append(k, v)
        q = Q[:, t].contiguous()
        a = paged.decode(q)
        b = contig.decode(q)
        torch.cuda.synchronize()
        assert torch.equal(a, b), f"decode step {s}"
        t += 1
    # the pool rows at the table's blocks are the contiguous cache rows
    n = t
    for bb in range(B):
        for ri in range(sum(kinds)):
            rows = torch.cat([paged.k_full[ids[bb, ri, blk]] for blk in range(max_blocks)])[:n]
            assert torch.equal(rows, contig.k_full[bb, ri, :n])
    from streaming_kv_cache_duo_gb300 import duo_device_error
    assert duo_device_error() == 0


def test_paged_decode_against_oracle():
    B, Hq, Hkv, D, S, R = 1, 4, 2, 128, 2, 16
    kinds = [1, 0]
    block_size, ctx = 128, 1000
    paged, _, _ = _layers(B, Hq, Hkv, D, S, R, kinds, block_size, -(-(ctx + 1) // block_size), seed=3)
    seed = 5
    K = device_stream(seed, ds.STREAM_K, B, 0, ctx + 1, Hkv, D, "cuda")
    V = device_stream(seed, ds.STREAM_V, B, 0, ctx + 1, Hkv, D, "cuda")
    paged.append(K.contiguous(), V.contiguous())
    q = device_stream(seed, ds.STREAM_Q, B, ctx, 1, Hq, D, "cuda")[:, 0].contiguous()
    o = paged.decode(q)
    torch.cuda.synchronize()
    Kh = host_stream(seed, ds.STREAM_K, B, 0, ctx + 1, Hkv, D)[0]
    Vh = host_stream(seed, ds.STREAM_V, B, 0, ctx + 1, Hkv, D)[0]
    Qh = host_stream(seed, ds.STREAM_Q, B, ctx, 1, Hq, D)[0, 0]
    cache = OracleCache(kinds, S, R, D)
    cache.append(Kh, Vh)
    assert_close(to_np(o[0]), decode_from_cache(Qh, ctx, cache), "paged decode")


def test_bad_block_id_is_reported_not_dereferenced():
    from streaming_kv_cache_duo_gb300 import _lib
    B, Hq, Hkv, D, S, R = 1, 2, 2, 64, 2, 8
    paged, _, _ = _layers(B, Hq, Hkv, D, S, R, [1, 0], 128, 2)
    paged.block_table[0, 0, 1] = 10_000  # outside the pool
    K = device_stream(1, ds.STREAM_K, B, 0, 200, Hkv, D, "cuda")
    paged.append(K, K)  # rows 128 ... 199 fall in the bad block
    code = _lib.duo_device_error()
    assert code & (1 << 21)
    q = device_stream(1, ds.STREAM_Q, B, 199, 1, Hq, D, "cuda")[:, 0].contiguous()
    paged.decode(q)
    paged.prefill(device_stream(1, ds.STREAM_Q, B, 200, 4, Hq, D, "cuda"),
                  device_stream(1, ds.STREAM_K, B, 200, 4, Hkv, D, "cuda"),
                  device_stream(1, ds.STREAM_V, B, 200, 4, Hkv, D, "cuda"))
    assert _lib.duo_device_error() & (1 << 21)
    assert _lib.duo_device_error() == 0


def test_paged_capacity_and_block_size_checks():
    from streaming_kv_cache_duo_gb300 import DuoError, DuoPagedLayer, _lib
    B, Hq, Hkv, D = 1, 2, 2, 64
    table = torch.zeros((B, 1, 1), dtype=torch.int32, device="cuda")
    paged = DuoPagedLayer(B, Hq, Hkv, D, 2, 8, 128, 1, 1, table, [1, 0])
    K = torch.zeros((B, 129, Hkv, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(DuoError, match="DUO_ERR_CAPACITY"):
        paged.append(K, K)
    bad = _lib.duo_paged(table.data_ptr(), 96, 1, 1)
    with pytest.raises(DuoError, match="DUO_ERR_UNSUPPORTED"):
        _lib.duo_kv_append_paged(paged.handle, paged.cache, bad, K[:, :1].contiguous(), K[:, :1].contiguous(), 1)
