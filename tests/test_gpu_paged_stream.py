"""Streaming heads kept in the paged pool with block-granular eviction: the caller
hands out only blocks that stay live, frees the blocks the library names dead after
every call (their table entries become -1 and the pool rows are refilled with NaN, as
another sequence reusing them would), and prefill, append and decode still match the
float64 oracle. A read or write of a dropped block would either trip the bad-block
error (table entry -1) or bring NaN into the outputs."""

import numpy as np
import pytest
import torch

import duo_synth as ds
import oracle
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import assert_close, device_stream, host_stream, to_np

pytestmark = pytest.mark.gpu


class Allocator:
    """Host mirror of both block tables plus a free list of pool blocks."""

    def __init__(self, layer, num_blocks, seed):
        self.layer = layer
        self.free = [int(x) for x in np.random.default_rng(seed).permutation(num_blocks)]
        self.ret = np.full(tuple(layer.block_table.shape), -1, np.int64) if layer.block_table is not None else None
        self.str = np.full(tuple(layer.stream_table.shape), -1, np.int64)
        self.freed = 0

    def upload(self):
        if self.ret is not None:
            self.layer.block_table.copy_(torch.from_numpy(self.ret.astype(np.int32)))
        self.layer.stream_table.copy_(torch.from_numpy(self.str.astype(np.int32)))

    def before_append(self, n, T):
        """Blocks that hold rows [n, n + T) and are still live after the call."""
        bs = self.layer.block_size
        lo, hi = self.layer.dead_blocks(n + T)
        for k in range(n // bs, -(-(n + T) // bs)):
            if self.ret is not None:
                for idx in np.ndindex(self.ret.shape[:2]):
                    if self.ret[idx + (k,)] < 0:
                        self.ret[idx + (k,)] = self.free.pop()
            if lo <= k < hi:
                continue  # dead by the end of the call: never written
            for idx in np.ndindex(self.str.shape[:2]):
                if self.str[idx + (k,)] < 0:
                    self.str[idx + (k,)] = self.free.pop()
        self.upload()

    def after_append(self, n):
        lo, hi = self.layer.dead_blocks(n)
        for k in range(lo, hi):
            for idx in np.ndindex(self.str.shape[:2]):
                blk = self.str[idx + (k,)]
                if blk >= 0:
                    self.layer.k_full[blk].fill_(float("nan"))
                    self.layer.v_full[blk].fill_(float("nan"))
                    self.free.append(int(blk))
                    self.str[idx + (k,)] = -1
                    self.freed += 1
        self.upload()


def _layer(B, Hq, Hkv, D, S, R, kinds, block_size, max_blocks, num_blocks):
    from streaming_kv_cache_duo_gb300 import DuoPagedLayer
    n_ret = sum(kinds)
    n_str = len(kinds) - n_ret
    ret = torch.full((B, n_ret, max_blocks), -1, dtype=torch.int32, device="cuda") if n_ret else None
    st = torch.full((B, n_str, max_blocks), -1, dtype=torch.int32, device="cuda")
    layer = DuoPagedLayer(B, Hq, Hkv, D, S, R, block_size, max_blocks, num_blocks, ret, kinds, stream_table=st)
    layer.k_full.fill_(float("nan"))
    layer.v_full.fill_(float("nan"))
    return layer


CASES = [
    # B, Hq, Hkv, D, S, R, kinds, block_size, chunks, decode steps
    (2, 8, 4, 128, 4, 200, [1, 0, 1, 0], 128, [300, 100, 37, 400, 5], 4),
    (1, 8, 2, 64, 130, 129, [0, 1], 128, [700, 1, 260], 3),        # sinks span two blocks
    (1, 4, 4, 128, 0, 1, [0, 0, 1, 0], 256, [129, 512], 2),        # window of one, no sinks
    (1, 8, 2, 128, 64, 256, [0, 0], 128, [1000, 300], 3),          # no retrieval head at all
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_paged_stream_matches_oracle(case):
    from streaming_kv_cache_duo_gb300 import duo_device_error
    B, Hq, Hkv, D, S, R, kinds, bs, chunks, steps = case
    total = sum(chunks) + steps
    max_blocks = -(-total // bs)
    num_blocks = B * len(kinds) * max_blocks + 4
    layer = _layer(B, Hq, Hkv, D, S, R, kinds, bs, max_blocks, num_blocks)
    alloc = Allocator(layer, num_blocks, seed=sum(chunks))
    seed = 41 + D
    Q = device_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D, "cuda")
    K = device_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    V = device_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D, "cuda")
    Qh = host_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D)
    Kh = host_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D)
    Vh = host_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D)
    t = 0
    for T in chunks:
        q, k, v = (x[:, t:t + T].contiguous() for x in (Q, K, V))
        o = layer.prefill(q, k, v)
        torch.cuda.synchronize()
        assert duo_device_error() == 0, f"prefill chunk at {t}"
        rows = np.arange(t, t + T)
        ref = np.stack([oracle.prefill(Qh[b, :t + T], Kh[b, :t + T], Vh[b, :t + T], kinds, S, R, rows=rows)
                        for b in range(B)])
        assert_close(to_np(o), ref, f"prefill chunk at {t}")
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
        assert duo_device_error() == 0, f"decode step {s}"
        for b in range(B):
            cache = OracleCache(kinds, S, R, D)
            cache.append(Kh[b, :t + 1], Vh[b, :t + 1])
            assert_close(to_np(o[b]), decode_from_cache(Qh[b, t], t, cache), f"decode step {s} sequence {b}")
        t += 1
    # blocks were dropped along the way, and a streaming head never held more than the
    # sink blocks plus the blocks reaching back R tokens (plus the one being filled)
    if total - R > -(-S // bs) * bs + bs:
        assert alloc.freed > 0
    held = (alloc.str >= 0).sum(axis=-1)
    assert held.max() <= -(-S // bs) + -(-R // bs) + 1


def test_dropped_block_is_reported_not_read():
    from streaming_kv_cache_duo_gb300 import _lib
    B, Hq, Hkv, D, S, R, bs = 1, 4, 2, 64, 4, 100, 128
    kinds = [1, 0]
    layer = _layer(B, Hq, Hkv, D, S, R, kinds, bs, 4, 16)
    alloc = Allocator(layer, 16, seed=7)
    K = device_stream(3, ds.STREAM_K, B, 0, 400, Hkv, D, "cuda")
    alloc.before_append(0, 300)
    layer.append(K[:, :300].contiguous(), K[:, :300].contiguous())
    alloc.after_append(300)
    assert _lib.duo_device_error() == 0
    # the caller wrongly drops a live block (the one holding the window)
    alloc.str[0, 0, 2] = -1
    alloc.upload()
    q = device_stream(3, ds.STREAM_Q, B, 299, 1, Hq, D, "cuda")[:, 0].contiguous()
    layer.decode(q)
    assert _lib.duo_device_error() & (1 << 21)
    layer.prefill(device_stream(3, ds.STREAM_Q, B, 300, 8, Hq, D, "cuda"), K[:, 300:308].contiguous(),
                  K[:, 300:308].contiguous())
    assert _lib.duo_device_error() & (1 << 21)
    assert _lib.duo_device_error() == 0
