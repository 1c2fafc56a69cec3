"""4-bit KV caches on the GPU: the codes and (scale, zero) pairs duo_kv_append_kv4
stores equal the oracle's encoding bit for bit (retrieval rows and the sink + ring
slots), and duo_attn_decode_kv4 matches the float64 oracle attending over the
dequantized rows."""

import numpy as np
import pytest
import torch

import duo_synth as ds
import oracle.kv4 as kv4
from oracle import RingCacheSim
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import assert_close, device_stream, host_stream, kv4_v_rows, to_np

pytestmark = pytest.mark.gpu


def _bits(sz):
    """int32 (scale | zero << 16) -> (scale fp16, zero fp16) arrays."""
    u = sz.cpu().numpy().astype(np.uint32)
    return (u & 0xFFFF).astype(np.uint16).view(np.float16), (u >> 16).astype(np.uint16).view(np.float16)


def _run(seed, B, Hq, Hkv, D, S, R, kinds, ctx, steps, chunk=None, poison=False):
    from streaming_kv_cache_duo_gb300 import DuoKv4Layer, duo_device_error
    total = ctx + steps
    layer = DuoKv4Layer(B, Hq, Hkv, D, S, R, total, kinds)
    if poison:  # codes 0xFF and (NaN, NaN) pairs wherever nothing has been appended
        for t in (layer.k_codes, layer.v_codes, layer.ks_codes, layer.vs_codes):
            t.fill_(0xFF)
        for t in (layer.k_sz, layer.v_sz, layer.ks_sz, layer.vs_sz):
            t.fill_(0x7E007E00)
    K = device_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    V = device_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D, "cuda")
    Q = device_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D, "cuda")
    chunk = chunk or max(ctx, 1)
    for c0 in range(0, ctx, chunk):
        T = min(chunk, ctx - c0)
        layer.append(K[:, c0:c0 + T].contiguous(), V[:, c0:c0 + T].contiguous())
    outs = []
    for s in range(steps):
        p = ctx + s
        layer.append(K[:, p:p + 1].contiguous(), V[:, p:p + 1].contiguous())
        outs.append(layer.decode(Q[:, p].contiguous()))
    torch.cuda.synchronize()
    assert duo_device_error() == 0
    return layer, outs


CASES = [
    # B, Hq, Hkv, D, S, R, kinds, ctx, steps, append chunk
    (2, 8, 4, 128, 4, 64, [1, 0, 1, 0], 700, 3, 300),
    (1, 4, 4, 64, 4, 32, [1, 0, 1, 0], 256, 4, None),           # the tiny workload's shape
    (1, 32, 8, 128, 64, 256, [1, 0, 0, 0, 0, 0, 1, 0], 3000, 2, 1024),
    (1, 16, 2, 128, 8, 40, [0, 1], 1000, 2, None),              # GQA 8
    (2, 2, 2, 128, 3, 5, [1, 1], 5, 4, None),                   # all retrieval, tiny context
    (1, 16, 2, 128, 35, 115, [0, 0], 600, 2, 250),              # no retrieval head at all
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_kv4_append_is_bit_exact_and_decode_matches_oracle(case):
    B, Hq, Hkv, D, S, R, kinds, ctx, steps, chunk = case
    seed = 700 + ctx % 89
    layer, outs = _run(seed, B, Hq, Hkv, D, S, R, kinds, ctx, steps, chunk)
    total = ctx + steps
    Kh = host_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D).astype(np.float32)
    Vh = host_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D).astype(np.float32)
    Qh = host_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D)
    ret = [h for h in range(Hkv) if kinds[h]]
    strm = [h for h in range(Hkv) if not kinds[h]]
    # stored rows, bit for bit
    rows = lambda t: t.cpu().numpy()
    v_rows = lambda t: kv4_v_rows(t.cpu().numpy(), D)  # V codes are kept in 16-row groups
    for X, codes, sz, scodes, ssz, as_rows in ((Kh, layer.k_codes, layer.k_sz, layer.ks_codes, layer.ks_sz, rows),
                                               (Vh, layer.v_codes, layer.v_sz, layer.vs_codes, layer.vs_sz, v_rows)):
        codes, scodes = as_rows(codes), as_rows(scodes)
        c_all, s_all, z_all = kv4.quantize_rows(X)  # [B, total, Hkv, ...]
        if ret:
            got_s, got_z = _bits(sz[:, :, :total])
            for ri, h in enumerate(ret):
                assert np.array_equal(codes[:, ri, :total], kv4.pack_codes(c_all[:, :, h]))
                assert np.array_equal(got_s[:, ri].view(np.uint16), s_all[:, :, h].view(np.uint16))
                assert np.array_equal(got_z[:, ri].view(np.uint16), z_all[:, :, h].view(np.uint16))
        if strm:
            sim = RingCacheSim(S, R)
            sim.append(total)
            pos = sim.positions()
            assert layer.pos.cpu().numpy().tolist() == [pos] * B
            got_s, got_z = _bits(ssz)
            for si, h in enumerate(strm):
                for slot, t in enumerate(pos):
                    if t < 0:
                        continue
                    assert np.array_equal(scodes[:, si, slot], kv4.pack_codes(c_all[:, t, h]))
                    assert np.array_equal(got_s[:, si, slot].view(np.uint16), s_all[:, t, h].view(np.uint16))
                    assert np.array_equal(got_z[:, si, slot].view(np.uint16), z_all[:, t, h].view(np.uint16))
    # decode over what the cache holds: the dequantized rows
    Kq, Vq = kv4.roundtrip(Kh), kv4.roundtrip(Vh)
    for b in range(B):
        cache = OracleCache(kinds, S, R, D)
        if ctx:
            cache.append(Kq[b, :ctx], Vq[b, :ctx])
        for s in range(steps):
            p = ctx + s
            cache.append(Kq[b, p:p + 1], Vq[b, p:p + 1])
            assert_close(to_np(outs[s][b]), decode_from_cache(Qh[b, p], p, cache), f"b{b} step {s}")


def test_constant_rows_have_zero_scale():
    from streaming_kv_cache_duo_gb300 import DuoKv4Layer
    B, Hq, Hkv, D = 1, 2, 2, 64
    layer = DuoKv4Layer(B, Hq, Hkv, D, 2, 8, 32, [1, 0])
    k = torch.full((B, 3, Hkv, D), 1.5, dtype=torch.bfloat16, device="cuda")
    layer.append(k, k)
    q = torch.ones((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    o = layer.decode(q)
    torch.cuda.synchronize()
    s, z = _bits(layer.k_sz[:, :, :3])
    assert (s == 0).all() and (z == np.float16(1.5)).all()
    assert (layer.k_codes[:, :, :3] == 0).all()
    assert torch.equal(o, torch.full_like(o, 1.5))


def test_kv4_argument_checks():
    from streaming_kv_cache_duo_gb300 import DuoError, DuoKv4Layer, _lib
    layer = DuoKv4Layer(1, 2, 2, 64, 2, 8, 32, [1, 0])
    k = torch.zeros((1, 1, 2, 64), dtype=torch.bfloat16, device="cuda")
    bad = _lib.duo_kv4_cache(None, layer.v_codes.data_ptr(), layer.k_sz.data_ptr(), layer.v_sz.data_ptr(),
                             layer.ks_codes.data_ptr(), layer.vs_codes.data_ptr(), layer.ks_sz.data_ptr(),
                             layer.vs_sz.data_ptr())
    with pytest.raises(DuoError, match="DUO_ERR_INVALID_ARG"):
        _lib.duo_kv_append_kv4(layer.handle, layer.cache, bad, k, k, 1)
    with pytest.raises(DuoError, match="DUO_ERR_CAPACITY"):
        layer.append(torch.zeros((1, 33, 2, 64), dtype=torch.bfloat16, device="cuda"),
                     torch.zeros((1, 33, 2, 64), dtype=torch.bfloat16, device="cuda"))


def test_kv4_poisoned_tail_is_never_used():
    """Decode copies whole 16-row chunks, so rows past the tokens held (and empty ring
    slots) reach shared memory: their codes and NaN (scale, zero) pairs must not reach
    the output. Every GQA grouping and both head dims, against an unpoisoned run."""
    for case in [(2, 8, 4, 128, 4, 64, [1, 0, 1, 0], 150, 3, None),     # g = 2
                 (1, 16, 4, 64, 3, 29, [0, 1, 1, 0], 301, 3, 100),      # g = 4, D 64
                 (2, 16, 2, 128, 8, 40, [1, 0], 77, 4, None)]:          # g = 8
        _, clean = _run(31, *case)
        _, dirty = _run(31, *case, poison=True)
        for a, b in zip(clean, dirty):
            assert torch.isfinite(b.float()).all()
            assert torch.equal(a, b)


def test_kv4_wide_value_rows_do_not_overflow_fp16():
    """V rows 1024 times wider than the generator's (exact in bf16; |v| up to ~5000, row
    scales ~650): p (up to 2^8 under the lazy rescale) times the row scale would pass
    the fp16 maximum if stored unscaled; the decode must still match the oracle."""
    from streaming_kv_cache_duo_gb300 import DuoKv4Layer, duo_device_error
    B, Hq, Hkv, D, S, R, kinds, ctx, steps = 1, 16, 4, 128, 4, 64, [1, 0, 1, 1], 900, 3
    seed = 77
    total = ctx + steps
    layer = DuoKv4Layer(B, Hq, Hkv, D, S, R, total, kinds)
    K = device_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    V = device_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D, "cuda") * 1024
    Q = device_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D, "cuda")
    layer.append(K[:, :ctx].contiguous(), V[:, :ctx].contiguous())
    Kq = kv4.roundtrip(host_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D).astype(np.float32))
    Vq = kv4.roundtrip((host_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D) * 1024).astype(np.float32))
    Qh = host_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D)
    for s in range(steps):
        p = ctx + s
        layer.append(K[:, p:p + 1].contiguous(), V[:, p:p + 1].contiguous())
        o = layer.decode(Q[:, p].contiguous())
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        cache = OracleCache(kinds, S, R, D)
        cache.append(Kq[0, :p + 1], Vq[0, :p + 1])
        ref = decode_from_cache(Qh[0, p], p, cache)
        assert_close(to_np(o[0]) / 1024, ref / 1024, f"step {s}")


def test_kv4_decode_one_unit_split_over_every_cta():
    """One retrieval unit of 160000 keys spread over the whole 4-bit grid (two CTAs per SM,
    one partial each), so the merge kernel takes its partials in more than one round of
    loads per warp; two decode steps against the oracle over the dequantized rows."""
    B, Hq, Hkv, D, S, R, kinds, ctx, steps = 1, 8, 2, 128, 4, 64, [1, 0], 160000, 2
    seed = 741
    layer, outs = _run(seed, B, Hq, Hkv, D, S, R, kinds, ctx, steps, 65536)
    total = ctx + steps
    Kq = kv4.roundtrip(host_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D).astype(np.float32))
    Vq = kv4.roundtrip(host_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D).astype(np.float32))
    Qh = host_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D)
    cache = OracleCache(kinds, S, R, D)
    cache.append(Kq[0, :ctx], Vq[0, :ctx])
    for s in range(steps):
        p = ctx + s
        cache.append(Kq[0, p:p + 1], Vq[0, p:p + 1])
        assert_close(to_np(outs[s][0]), decode_from_cache(Qh[0, p], p, cache), f"step {s}")
