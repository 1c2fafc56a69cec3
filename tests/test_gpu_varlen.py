"""Per-sequence lengths held on the device, and a decode step captured in a CUDA graph:
appends and decodes read each sequence's length from device memory, so one captured
step replays for every later token. Outputs are checked against the float64 oracle
run per sequence on its own length."""

import numpy as np
import pytest
import torch

import duo_synth as ds
from oracle import RingCacheSim
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import assert_close, device_stream, host_stream, to_np

pytestmark = pytest.mark.gpu


def _ragged_layer(seed, B, Hq, Hkv, D, S, R, kinds, lens, extra):
    """A layer whose sequence b holds exactly tokens [0, lens[b]) (retrieval rows and
    sink + ring slots as after lens[b] appends)."""
    from streaming_kv_cache_duo_gb300 import DuoLayer
    n0 = max(lens)
    total = n0 + extra
    layer = DuoLayer(B, Hq, Hkv, D, S, R, total, kinds)
    K = device_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    V = device_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D, "cuda")
    Q = device_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D, "cuda")
    if n0:
        layer.append(K[:, :n0].contiguous(), V[:, :n0].contiguous())
    strh = [h for h in range(Hkv) if not kinds[h]]
    for b in range(B):
        sim = RingCacheSim(S, R)
        sim.append(lens[b])
        pos = sim.positions()
        layer.pos[b] = torch.tensor(pos, dtype=torch.int32)
        for slot, t in enumerate(pos):
            if t >= 0:
                for si, h in enumerate(strh):
                    layer.k_sr[b, si, slot] = K[b, t, h]
                    layer.v_sr[b, si, slot] = V[b, t, h]
    seq_lens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return layer, seq_lens, Q, K, V


def _token(X, positions):
    """[B, 1, H, D] gathered at each sequence's own position."""
    return torch.stack([X[b, p] for b, p in enumerate(positions)])[:, None].contiguous()


def _oracle_step(seed, B, Hq, Hkv, D, S, R, kinds, lens, step):
    total = max(lens) + step + 1
    Qh = host_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D)
    Kh = host_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D)
    Vh = host_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D)
    out = []
    for b in range(B):
        p = lens[b] + step
        cache = OracleCache(kinds, S, R, D)
        cache.append(Kh[b, :p + 1], Vh[b, :p + 1])
        out.append(decode_from_cache(Qh[b, p], p, cache))
    return np.stack(out)


CASES = [
    # B, Hq, Hkv, D, S, R, kinds, lens
    (5, 8, 4, 128, 4, 64, [1, 0, 0, 1], [1, 37, 300, 4097, 64]),
    (3, 8, 2, 64, 2, 20, [0, 1], [0, 19, 500]),
    (4, 16, 2, 128, 64, 256, [1, 0], [2000, 1, 320, 321]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_ragged_decode_matches_oracle(case):
    from streaming_kv_cache_duo_gb300 import duo_device_error
    B, Hq, Hkv, D, S, R, kinds, lens = case
    seed = 300 + D
    steps = 3
    layer, seq_lens, Q, K, V = _ragged_layer(seed, B, Hq, Hkv, D, S, R, kinds, lens, steps)
    max_len = max(lens) + steps
    for s in range(steps):
        posn = [l + s for l in lens]
        layer.append_varlen(_token(K, posn), _token(V, posn), seq_lens)
        o = layer.decode_varlen(_token(Q, posn)[:, 0].contiguous(), seq_lens, max_len)
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        assert seq_lens.tolist() == [l + s + 1 for l in lens]
        ref = _oracle_step(seed, B, Hq, Hkv, D, S, R, kinds, lens, s)
        for b in range(B):
            assert_close(to_np(o[b]), ref[b], f"step {s} sequence {b}")


def test_uniform_lengths_match_the_uniform_decode_bitwise():
    B, Hq, Hkv, D, S, R = 3, 8, 2, 128, 4, 32
    kinds = [1, 0]
    n = 700
    layer, seq_lens, Q, K, V = _ragged_layer(9, B, Hq, Hkv, D, S, R, kinds, [n] * B, 1)
    layer.append(K[:, n:n + 1].contiguous(), V[:, n:n + 1].contiguous())
    seq_lens += 1
    q = Q[:, n].contiguous()
    a = layer.decode(q)
    b = layer.decode_varlen(q, seq_lens, n + 1)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_zero_length_sequence_gives_zero_output():
    B, Hq, Hkv, D, S, R = 2, 4, 2, 64, 2, 8
    layer, seq_lens, Q, K, V = _ragged_layer(4, B, Hq, Hkv, D, S, R, [1, 0], [0, 5], 1)
    o = layer.decode_varlen(Q[:, 4].contiguous(), seq_lens, 6)
    torch.cuda.synchronize()
    assert bool((o[0] == 0).all())
    assert torch.isfinite(o[1].float()).all()


def test_decode_step_captured_in_a_cuda_graph():
    from streaming_kv_cache_duo_gb300 import duo_device_error
    B, Hq, Hkv, D, S, R = 4, 8, 2, 128, 4, 64
    kinds = [0, 1]
    lens = [10, 1000, 64, 257]
    steps = 6
    seed = 77
    layer, seq_lens, Q, K, V = _ragged_layer(seed, B, Hq, Hkv, D, S, R, kinds, lens, steps)
    max_len = max(lens) + steps
    sq = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    sk = torch.empty((B, 1, Hkv, D), dtype=torch.bfloat16, device="cuda")
    sv = torch.empty_like(sk)
    so = torch.empty_like(sq)

    def feed(s):
        posn = [l + s for l in lens]
        sq.copy_(_token(Q, posn)[:, 0])
        sk.copy_(_token(K, posn))
        sv.copy_(_token(V, posn))

    # step 0 eagerly (the kernels are loaded before capture)
    feed(0)
    layer.append_varlen(sk, sv, seq_lens)
    layer.decode_varlen(sq, seq_lens, max_len, out=so)
    torch.cuda.synchronize()
    outs = [so.clone()]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.append_varlen(sk, sv, seq_lens)
        layer.decode_varlen(sq, seq_lens, max_len, out=so)
    for s in range(1, steps):
        feed(s)
        graph.replay()
        outs.append(so.clone())
    torch.cuda.synchronize()
    assert duo_device_error() == 0
    assert seq_lens.tolist() == [l + steps for l in lens]
    for s in range(steps):
        ref = _oracle_step(seed, B, Hq, Hkv, D, S, R, kinds, lens, s)
        assert_close(to_np(outs[s]), ref, f"graph step {s}")


def test_device_append_into_a_full_cache_reports_capacity():
    from streaming_kv_cache_duo_gb300 import DuoLayer, _lib
    layer = DuoLayer(2, 2, 2, 64, 2, 6, 4, [1, 0])
    seq_lens = torch.tensor([3, 4], dtype=torch.int32, device="cuda")
    k = torch.zeros((2, 1, 2, 64), dtype=torch.bfloat16, device="cuda")
    layer.append_varlen(k, k, seq_lens)
    code = _lib.duo_device_error()
    assert code & (1 << 20)
    assert seq_lens.tolist() == [4, 4]  # the full sequence did not move
    assert _lib.duo_device_error() == 0
