"""duo_kv_append on the GPU against the oracle's cache model: bit-exact cache rows,
ring slots and positions."""

import numpy as np
import pytest
import torch

import duo_synth as ds
from oracle import RingCacheSim

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _check_cache(layer, seed, kinds, S, R):
    n = layer.n
    B, Hkv, D = layer.B, layer.Hkv, layer.D
    kb = ds.stream_bits(seed, ds.STREAM_K, B, 0, n, Hkv, D)
    vb = ds.stream_bits(seed, ds.STREAM_V, B, 0, n, Hkv, D)
    sim = RingCacheSim(S, R)
    sim.append(n)
    want_pos = np.array(sim.positions(), dtype=np.int32)
    pos = layer.pos.cpu().numpy()
    if layer.n_str:  # pos[] serves the streaming heads only
        for b in range(B):
            np.testing.assert_array_equal(pos[b], want_pos)
    kf, vf = _bits(layer.k_full), _bits(layer.v_full)
    ks, vs = _bits(layer.k_sr), _bits(layer.v_sr)
    ri = si = 0
    for h in range(Hkv):
        if kinds[h]:
            np.testing.assert_array_equal(kf[:, ri, :n], kb[:, :, h])
            np.testing.assert_array_equal(vf[:, ri, :n], vb[:, :, h])
            ri += 1
        else:
            for slot, p in enumerate(want_pos):
                if p >= 0:
                    np.testing.assert_array_equal(ks[:, si, slot], kb[:, p, h])
                    np.testing.assert_array_equal(vs[:, si, slot], vb[:, p, h])
            si += 1


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S,R", [(4, 32), (0, 5), (3, 1), (64, 256)])
def test_append_sequences_bit_exact(D, S, R):
    from streaming_kv_cache_duo_gb300 import DuoLayer
    seed, B, Hkv, Hq = 11, 2, 4, 8
    kinds = [1, 0, 0, 1]
    chunks = [1, 5, 37, 1, 130, 2 * (S + R) + 3, 1, 1, 64]
    total = sum(chunks)
    layer = DuoLayer(B, Hq, Hkv, D, S, R, total + 8, kinds)
    k = ds.stream_torch(seed, ds.STREAM_K, B, 0, total, Hkv, D).cuda()
    v = ds.stream_torch(seed, ds.STREAM_V, B, 0, total, Hkv, D).cuda()
    t = 0
    for T in chunks:
        layer.append(k[:, t:t + T].contiguous(), v[:, t:t + T].contiguous())
        t += T
        assert layer.n == t
        _check_cache(layer, seed, kinds, S, R)


def test_all_streaming_and_all_retrieval():
    from streaming_kv_cache_duo_gb300 import DuoLayer
    for kinds in ([0, 0], [1, 1]):
        layer = DuoLayer(1, 2, 2, 128, 2, 6, 64, kinds)
        k = ds.stream_torch(3, ds.STREAM_K, 1, 0, 40, 2, 128).cuda()
        v = ds.stream_torch(3, ds.STREAM_V, 1, 0, 40, 2, 128).cuda()
        layer.append(k[:, :17].contiguous(), v[:, :17].contiguous())
        layer.append(k[:, 17:].contiguous(), v[:, 17:].contiguous())
        _check_cache(layer, 3, kinds, 2, 6)


def test_capacity_error_writes_nothing():
    from streaming_kv_cache_duo_gb300 import DuoError, DuoLayer
    layer = DuoLayer(1, 2, 2, 64, 2, 6, 16, [1, 0])
    k = ds.stream_torch(3, ds.STREAM_K, 1, 0, 17, 2, 64).cuda()
    layer.append(k[:, :10].contiguous(), k[:, :10].contiguous())
    before = layer.k_full.clone()
    with pytest.raises(DuoError, match="DUO_ERR_CAPACITY"):
        layer.append(k[:, 10:17].contiguous(), k[:, 10:17].contiguous())
    torch.cuda.synchronize()
    assert layer.n == 10
    assert torch.equal(before, layer.k_full)


def test_full_size_context_append_sampled():
    """The 131072-token context of the batched-decode workload (B = 8), appended in
    chunks of 65536 as the decode benchmark does; sampled rows compared bit for bit."""
    from streaming_kv_cache_duo_gb300 import DuoLayer
    w = ds.WORKLOADS["batched_decode_ctx128k"]
    kinds = w.is_retrieval
    layer = DuoLayer(w.B, w.Hq, w.Hkv, w.D, w.S, w.R, w.context + 8, kinds)
    chunk = 65536
    for c0 in range(0, w.context, chunk):
        k = ds.stream_torch(w.seed, ds.STREAM_K, w.B, c0, chunk, w.Hkv, w.D, device="cuda")
        v = ds.stream_torch(w.seed, ds.STREAM_V, w.B, c0, chunk, w.Hkv, w.D, device="cuda")
        layer.append(k, v)
    torch.cuda.synchronize()
    n = layer.n
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, chunk - 1, chunk, n - 1], rng.integers(0, n, 64)]))
    ret = [h for h in range(w.Hkv) if kinds[h]]
    strh = [h for h in range(w.Hkv) if not kinds[h]]
    for b in (0, w.B - 1):
        for ri, h in enumerate(ret):
            got = _bits(layer.k_full[b, ri, rows])
            want = np.stack([ds.stream_bits(w.seed, ds.STREAM_K, w.B, int(r), 1, w.Hkv, w.D)[b, 0, h] for r in rows])
            np.testing.assert_array_equal(got, want)
        sim = RingCacheSim(w.S, w.R)
        sim.append(n)
        pos = layer.pos[b].cpu().numpy()
        np.testing.assert_array_equal(pos, np.array(sim.positions(), dtype=np.int32))
        for si, h in enumerate(strh):
            got = _bits(layer.v_sr[b, si])
            want = np.stack([ds.stream_bits(w.seed, ds.STREAM_V, w.B, int(p), 1, w.Hkv, w.D)[b, 0, h] for p in pos])
            np.testing.assert_array_equal(got, want)
