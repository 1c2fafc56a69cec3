"""4-bit caches with the retrieval rows in a paged pool (duo_kv_append_kv4_paged,
duo_attn_decode_kv4_paged): the block allocator of the attention-sink issue holding the
4-bit rows the DuoAttention README pairs the method with. Through a scattered block
table the stored codes and (scale, zero) pairs equal the oracle's encoding bit for bit,
the decode gives exactly the contiguous 4-bit layout's bits, and so matches the float64
oracle over the dequantized rows; a bad block id is reported, never followed."""

import numpy as np
import pytest
import torch

import duo_synth as ds
import oracle.kv4 as kv4
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import assert_close, device_stream, host_stream, kv4_v_rows, to_np

pytestmark = pytest.mark.gpu


def _bits(sz):
    u = sz.cpu().numpy().astype(np.uint32)
    return (u & 0xFFFF).astype(np.uint16), (u >> 16).astype(np.uint16)


def _layers(B, Hq, Hkv, D, S, R, kinds, block_size, max_blocks, seed):
    from streaming_kv_cache_duo_gb300 import DuoKv4Layer, DuoKv4PagedLayer
    n_ret = sum(kinds)
    num_blocks = B * n_ret * max_blocks + 3  # a few blocks nobody uses
    ids = np.random.default_rng(seed).permutation(num_blocks)[:B * n_ret * max_blocks].reshape(B, n_ret, max_blocks)
    table = torch.tensor(ids, dtype=torch.int32, device="cuda")
    paged = DuoKv4PagedLayer(B, Hq, Hkv, D, S, R, block_size, max_blocks, num_blocks, table, kinds)
    # unwritten rows hold codes 0xFF and (NaN, NaN) pairs: they must never be read
    paged.k_codes.fill_(0xFF)
    paged.v_codes.fill_(0xFF)
    paged.k_sz.fill_(0x7E007E00)
    paged.v_sz.fill_(0x7E007E00)
    contig = DuoKv4Layer(B, Hq, Hkv, D, S, R, block_size * max_blocks, kinds)
    return paged, contig, ids


CASES = [
    # B, Hq, Hkv, D, S, R, kinds, chunks, steps, block_size
    (2, 16, 4, 128, 4, 64, [1, 0, 1, 0], [700, 300, 1], 3, 128),   # g = 4
    (1, 16, 2, 64, 8, 40, [1, 0], [1000], 4, 256),                  # g = 8, D 64
    (2, 4, 2, 128, 3, 29, [1, 1], [129, 250], 3, 128),              # g = 2, all retrieval
    (1, 32, 8, 128, 64, 256, [1, 0, 0, 0, 0, 0, 1, 0], [5000], 2, 256),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_kv4_paged_matches_contiguous_and_oracle(case):
    from streaming_kv_cache_duo_gb300 import duo_device_error
    B, Hq, Hkv, D, S, R, kinds, chunks, steps, bs = case
    ctx = sum(chunks)
    total = ctx + steps
    max_blocks = -(-total // bs)
    seed = 1600 + ctx % 97
    paged, contig, ids = _layers(B, Hq, Hkv, D, S, R, kinds, bs, max_blocks, seed)
    K = device_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    V = device_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D, "cuda")
    Q = device_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D, "cuda")
    t = 0
    for c in chunks:
        for layer in (paged, contig):
            layer.append(K[:, t:t + c].contiguous(), V[:, t:t + c].contiguous())
        t += c
    outs = []
    for s in range(steps):
        p = ctx + s
        for layer in (paged, contig):
            layer.append(K[:, p:p + 1].contiguous(), V[:, p:p + 1].contiguous())
        q = Q[:, p].contiguous()
        a = paged.decode(q)
        b = contig.decode(q)
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        assert torch.equal(a, b), f"step {s}: paged and contiguous 4-bit decodes differ"
        outs.append(to_np(a))
    # stored rows through the table, bit for bit against the oracle's encoding
    Kh = host_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D).astype(np.float32)
    Vh = host_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D).astype(np.float32)
    ret = [h for h in range(Hkv) if kinds[h]]
    k_pool = paged.k_codes.cpu().numpy().reshape(-1, bs, D // 2)
    v_pool = kv4_v_rows(paged.v_codes.cpu().numpy().reshape(-1, bs, D // 2), D)
    for X, pool, sz in ((Kh, k_pool, paged.k_sz), (Vh, v_pool, paged.v_sz)):
        c_all, s_all, z_all = kv4.quantize_rows(X)
        got_s, got_z = _bits(sz.reshape(-1, bs))
        for b in range(B):
            for ri, h in enumerate(ret):
                for t0 in range(0, total, bs):
                    blk, n = ids[b, ri, t0 // bs], min(bs, total - t0)
                    assert np.array_equal(pool[blk, :n], kv4.pack_codes(c_all[b, t0:t0 + n, h])), (b, h, t0)
                    assert np.array_equal(got_s[blk, :n], s_all[b, t0:t0 + n, h].view(np.uint16))
                    assert np.array_equal(got_z[blk, :n], z_all[b, t0:t0 + n, h].view(np.uint16))
    # decode against the oracle over the dequantized rows
    Qh = host_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D)
    Kq, Vq = kv4.roundtrip(Kh), kv4.roundtrip(Vh)
    for b in range(B):
        cache = OracleCache(kinds, S, R, D)
        cache.append(Kq[b, :ctx], Vq[b, :ctx])
        for s in range(steps):
            p = ctx + s
            cache.append(Kq[b, p:p + 1], Vq[b, p:p + 1])
            assert_close(outs[s][b], decode_from_cache(Qh[b, p], p, cache), f"b{b} step {s}")


def test_kv4_paged_bad_block_is_reported_not_followed():
    from streaming_kv_cache_duo_gb300 import DuoKv4PagedLayer, duo_device_error
    B, Hq, Hkv, D, S, R, kinds, bs = 1, 8, 2, 128, 4, 32, [1, 0], 128
    max_blocks, num_blocks = 4, 6
    table = torch.tensor([[[3, 1, num_blocks + 5, 0]]], dtype=torch.int32, device="cuda")
    layer = DuoKv4PagedLayer(B, Hq, Hkv, D, S, R, bs, max_blocks, num_blocks, table, kinds)
    K = device_stream(5, ds.STREAM_K, B, 0, 300, Hkv, D, "cuda")
    layer.append(K, K)  # rows 256 ... 299 fall in the bad block
    assert duo_device_error() & (1 << 21)  # the bad-block code
    q = device_stream(5, ds.STREAM_Q, B, 299, 1, Hq, D, "cuda")[:, 0].contiguous()
    o = layer.decode(q)
    assert duo_device_error() & (1 << 21)
    assert duo_device_error() == 0  # read and cleared
    assert torch.isfinite(o.float()).all()
    table[0, 0, 2] = 2  # a good table again: the same layer decodes normally
    layer.append(K[:, :1].contiguous(), K[:, :1].contiguous())
    layer.decode(q)
    assert duo_device_error() == 0


def test_kv4_paged_rejects_streaming_heads_in_the_pool():
    from streaming_kv_cache_duo_gb300 import DuoError, DuoKv4PagedLayer, _lib
    B, Hq, Hkv, D, S, R, kinds, bs = 1, 4, 2, 64, 4, 32, [1, 0], 128
    table = torch.zeros((1, 1, 2), dtype=torch.int32, device="cuda")
    layer = DuoKv4PagedLayer(B, Hq, Hkv, D, S, R, bs, 2, 2, table, kinds)
    stream_table = torch.zeros((1, 1, 2), dtype=torch.int32, device="cuda")
    bad = _lib.duo_paged(table.data_ptr(), bs, 2, 2, stream_table.data_ptr())
    k = torch.zeros((1, 1, Hkv, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(DuoError, match="DUO_ERR_UNSUPPORTED"):
        _lib.duo_kv_append_kv4_paged(layer.handle, layer.cache, bad, layer.kv4, k, k, 1)
