"""Dual Chunk Attention on the GPU (duo_dca_prefill, duo_dca_decode) against the float64
oracle (oracle.dca, pinned against the pull request's brute-force schedule), on sampled
query rows of every head: the first and last rows of each chunk, their neighbours, the
ragged tail, and random rows. With q_succ = q_inter = q and no mscale the method is
plain causal attention, and the DCA kernel must then give exactly the plain kernel's
bits."""

import numpy as np
import pytest
import torch

import duo_synth as ds
import oracle.dca as dca
from gpu_util import assert_close, device_stream, host_stream, to_np

pytestmark = pytest.mark.gpu


def _inputs(seed, B, Hq, Hkv, D, T, dev=True):
    f = (lambda s, H: device_stream(seed, s, B, 0, T, H, D, "cuda")) if dev else \
        (lambda s, H: host_stream(seed, s, B, 0, T, H, D))
    return (f(ds.STREAM_Q, Hq), f(ds.STREAM_Q_SUCC, Hq), f(ds.STREAM_Q_INTER, Hq), f(ds.STREAM_K, Hkv),
            f(ds.STREAM_V, Hkv))


def _rows(T, chunk_len, seed):
    rows = {0, 1, T - 1, T - 2}
    for c0 in range(0, T, chunk_len):
        rows |= {c0, c0 + 1, c0 - 1, c0 + chunk_len - 1, c0 + 255, c0 + 256}
    rng = np.random.default_rng(seed)
    rows |= set(rng.integers(0, T, 12).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < T))


CASES = [
    # B, Hq, Hkv, D, T, chunk_len
    (1, 4, 2, 128, 1100, 256),   # five chunks, ragged last chunk and block
    (2, 8, 8, 64, 700, 256),     # MHA, D 64
    (1, 4, 4, 128, 300, 512),    # one chunk: query only
    (1, 8, 2, 128, 1536, 512),   # three whole chunks, GQA 4
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_dca_prefill_and_decode_match_oracle(case):
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    B, Hq, Hkv, D, T, chunk_len = case
    steps = 3
    seed = 500 + T
    total = T + steps
    Q, QS, QI, K, V = _inputs(seed, B, Hq, Hkv, D, total)
    Qh, QSh, QIh, Kh, Vh = _inputs(seed, B, Hq, Hkv, D, total, dev=False)
    ms = ds.dca_mscale(B, total, chunk_len)
    msd = torch.from_numpy(ms).cuda()
    layer = DuoLayer(B, Hq, Hkv, D, 0, 1, total, [1] * Hkv)
    sl = slice(0, T)
    o = layer.dca_prefill(*(x[:, sl].contiguous() for x in (Q, QS, QI, K, V)), chunk_len,
                          mscale=msd[:, sl].contiguous())
    torch.cuda.synchronize()
    assert duo_device_error() == 0
    rows = _rows(T, chunk_len, seed)
    got = to_np(o)
    for b in range(B):
        ref = dca.attention(Qh[b, :T], QSh[b, :T], QIh[b, :T], Kh[b, :T], Vh[b, :T], ms[b, :T], chunk_len, rows=rows)
        assert_close(got[b, rows], ref, f"prefill b{b}")
    # decode the next tokens over the cache the prefill's keys went into
    layer.append(K[:, sl].contiguous(), V[:, sl].contiguous())
    for s in range(steps):
        p = T + s
        layer.append(K[:, p:p + 1].contiguous(), V[:, p:p + 1].contiguous())
        od = layer.dca_decode(Q[:, p].contiguous(), QS[:, p].contiguous(), QI[:, p].contiguous(), chunk_len,
                              mscale=msd[:, p].contiguous())
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        g = Hq // Hkv
        for b in range(B):
            ref = np.stack([dca.decode(Qh[b, p, h], QSh[b, p, h], QIh[b, p, h], Kh[b, :p + 1, h // g],
                                       Vh[b, :p + 1, h // g], ms[b, p], p, chunk_len) for h in range(Hq)])
            assert_close(to_np(od[b]), ref, f"decode step {s} b{b}")


def test_one_query_vector_is_the_plain_kernel_bit_for_bit():
    from streaming_kv_cache_duo_gb300 import DuoLayer
    B, Hq, Hkv, D, T = 1, 8, 2, 128, 1300
    Q, _, _, K, V = _inputs(9, B, Hq, Hkv, D, T)
    layer = DuoLayer(B, Hq, Hkv, D, 0, 1, T, [1, 1])
    a = layer.dca_prefill(Q, Q, Q, K, V, 256)
    b = layer.prefill(Q, K, V)
    layer.append(K, V)
    q1 = Q[:, T - 1].contiguous()
    c = layer.dca_decode(q1, q1, q1, 256)
    d = layer.decode(q1)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(c, d)


def test_dca_argument_checks():
    from streaming_kv_cache_duo_gb300 import DuoError, DuoLayer
    Q, QS, QI, K, V = _inputs(2, 1, 2, 2, 64, 300)
    mixed = DuoLayer(1, 2, 2, 64, 4, 16, 300, [1, 0])
    with pytest.raises(DuoError, match="DUO_ERR_UNSUPPORTED"):
        mixed.dca_prefill(Q, QS, QI, K, V, 256)
    full = DuoLayer(1, 2, 2, 64, 0, 1, 300, [1, 1])
    with pytest.raises(DuoError, match="DUO_ERR_UNSUPPORTED"):
        full.dca_prefill(Q, QS, QI, K, V, 384)
    with pytest.raises(DuoError, match="DUO_ERR_UNSUPPORTED"):
        full.dca_prefill(Q, QS, QI, K, V, 128)


@pytest.mark.parametrize("chunks,chunk_len", [([512, 768, 300], 256), ([1024, 256, 517], 512)])
def test_dca_chunked_prefill_matches_oracle(chunks, chunk_len):
    """Dual Chunk Attention prefill chunk by chunk against the growing cache (the pull
    request's demo runs with chunked prefill): every chunk's rows equal the one-shot
    definition at their absolute positions."""
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    B, Hq, Hkv, D = 1, 8, 2, 128
    total = sum(chunks)
    seed = 901
    Q, QS, QI, K, V = _inputs(seed, B, Hq, Hkv, D, total)
    Qh, QSh, QIh, Kh, Vh = _inputs(seed, B, Hq, Hkv, D, total, dev=False)
    ms = ds.dca_mscale(B, total, chunk_len)
    msd = torch.from_numpy(ms).cuda()
    layer = DuoLayer(B, Hq, Hkv, D, 0, 1, total, [1] * Hkv)
    t = 0
    for T in chunks:
        sl = slice(t, t + T)
        o = layer.dca_prefill(*(x[:, sl].contiguous() for x in (Q, QS, QI, K, V)), chunk_len,
                              mscale=msd[:, sl].contiguous())
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        rows = np.array(sorted({0, 1, T // 2, T - 2, T - 1} | {r for r in range(0, T, 97)}))
        ref = dca.attention(Qh[0, :t + T], QSh[0, :t + T], QIh[0, :t + T], Kh[0, :t + T], Vh[0, :t + T],
                            ms[0, :t + T], chunk_len, rows=rows + t)
        assert_close(to_np(o)[0, rows], ref, f"chunk at {t}")
        layer.append(K[:, sl].contiguous(), V[:, sl].contiguous())
        t += T


def test_dca_chunked_prefill_needs_an_aligned_cache():
    from streaming_kv_cache_duo_gb300 import DuoError, DuoLayer
    Q, QS, QI, K, V = _inputs(3, 1, 2, 2, 64, 400)
    layer = DuoLayer(1, 2, 2, 64, 0, 1, 400, [1, 1])
    layer.append(K[:, :100].contiguous(), V[:, :100].contiguous())
    sl = slice(100, 400)
    with pytest.raises(DuoError, match="DUO_ERR_UNSUPPORTED"):
        layer.dca_prefill(*(x[:, sl].contiguous() for x in (Q, QS, QI, K, V)), 256)


def _row_ref(q, qs, qi, K, V, ms_i, i, chunk_len):
    """Oracle prefill row i of one query head: the three query vectors broadcast to [i + 1,
    1, D] views (only row i is read), the head's keys and values [i + 1, 1, D]."""
    D = q.shape[-1]
    Q3 = [np.broadcast_to(np.asarray(x, np.float64), (i + 1, 1, D)) for x in (q, qs, qi)]
    ms = np.full(i + 1, ms_i, np.float64)
    return dca.attention(*Q3, K[:i + 1, None], V[:i + 1, None], ms, chunk_len, rows=[i], heads=[0])[0, 0]


def _check_rows(w, o, rows, heads, pos0, ms, keys):
    """Sampled rows (absolute positions) of the output o [B, T, Hq, D] of a call that
    started at position pos0, for the given query heads."""
    g = w.Hq // w.Hkv
    got = to_np(o[0, [r - pos0 for r in rows]][:, heads])
    ref = np.empty_like(got)
    for a, i in enumerate(rows):
        q, qs, qi = (host_stream(w.seed, s, 1, i, 1, w.Hq, w.D)[0, 0]
                     for s in (ds.STREAM_Q, ds.STREAM_Q_SUCC, ds.STREAM_Q_INTER))
        for c, h in enumerate(heads):
            K, V = keys[h // g]
            ref[a, c] = _row_ref(q[h], qs[h], qi[h], K, V, ms[0, i], i, w.dca_chunk)
    assert_close(got, ref, f"{w.name} rows {rows} heads {heads}")


def test_full_size_dca_prefill128k_and_decode_sampled():
    """The 131072-token Qwen2-72B-shaped layer (64 query / 8 KV heads, chunk 32768) in the
    benchmark's launch: one-shot prefill, then the prompt appended and decode steps from
    position 131072 (the first token of a new chunk); sampled rows at every chunk
    boundary and sampled heads of three KV heads against the oracle."""
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    from gpu_util import head_keys
    w = ds.WORKLOADS["qwen2_72b_dca_prefill128k"]
    L, CL, steps = w.prefill_len, w.dca_chunk, 2
    total = L + steps
    gen = lambda s, pos0, T, H: device_stream(w.seed, s, 1, pos0, T, H, w.D, "cuda")
    q, qs, qi = (gen(s, 0, L, w.Hq) for s in (ds.STREAM_Q, ds.STREAM_Q_SUCC, ds.STREAM_Q_INTER))
    k, v = gen(ds.STREAM_K, 0, L, w.Hkv), gen(ds.STREAM_V, 0, L, w.Hkv)
    ms = ds.dca_mscale(1, total, CL)
    msd = torch.from_numpy(ms).cuda()
    layer = DuoLayer(1, w.Hq, w.Hkv, w.D, w.S, w.R, total, [1] * w.Hkv)
    o = layer.dca_prefill(q, qs, qi, k, v, CL, mscale=msd[:, :L].contiguous())
    torch.cuda.synchronize()
    assert duo_device_error() == 0
    del q, qs, qi
    heads = [0, 37, 63]
    g = w.Hq // w.Hkv
    keys = {h // g: head_keys(w.seed, 0, h // g, 0, total, w.D) for h in heads + [5]}
    rng = np.random.default_rng(6)
    rows = sorted({0, 255, 256, L - 2, L - 1} | {c + d for c in range(CL, L, CL) for d in (-1, 0)}
                  | set(rng.integers(0, L, 3).tolist()))
    _check_rows(w, o, rows, heads, 0, ms, keys)
    del o
    layer.append(k, v)
    for s in range(steps):
        p = L + s
        layer.append(gen(ds.STREAM_K, p, 1, w.Hkv), gen(ds.STREAM_V, p, 1, w.Hkv))
        qd = [gen(x, p, 1, w.Hq)[:, 0].contiguous() for x in (ds.STREAM_Q, ds.STREAM_Q_SUCC, ds.STREAM_Q_INTER)]
        od = layer.dca_decode(*qd, CL, mscale=msd[:, p].contiguous())
        torch.cuda.synchronize()
        assert duo_device_error() == 0
    p = total - 1
    qh = [host_stream(w.seed, x, 1, p, 1, w.Hq, w.D)[0, 0] for x in (ds.STREAM_Q, ds.STREAM_Q_SUCC, ds.STREAM_Q_INTER)]
    dh = [5, 63]
    ref = np.stack([dca.decode(qh[0][h], qh[1][h], qh[2][h], keys[h // g][0][:p + 1], keys[h // g][1][:p + 1],
                               ms[0, p], p, CL) for h in dh])
    assert_close(to_np(od[0, dh]), ref, "decode at 131073")


def test_full_size_dca_prefill32k_chunked_sampled():
    """The 32768-token layer (chunk 8192) prefilled in calls of 12288, 12288 and 8192
    tokens against the growing cache, so that calls start and end inside DCA chunks;
    sampled rows of each call against the one-shot definition."""
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    from gpu_util import head_keys
    w = ds.WORKLOADS["qwen2_72b_dca_prefill32k"]
    L, CL = w.prefill_len, w.dca_chunk
    gen = lambda s, pos0, T, H: device_stream(w.seed, s, 1, pos0, T, H, w.D, "cuda")
    ms = ds.dca_mscale(1, L, CL)
    msd = torch.from_numpy(ms).cuda()
    layer = DuoLayer(1, w.Hq, w.Hkv, w.D, w.S, w.R, L, [1] * w.Hkv)
    heads = [3, 30, 60]
    g = w.Hq // w.Hkv
    keys = {h // g: head_keys(w.seed, 0, h // g, 0, L, w.D) for h in heads}
    t = 0
    for T in (12288, 12288, 8192):
        q, qs, qi = (gen(s, t, T, w.Hq) for s in (ds.STREAM_Q, ds.STREAM_Q_SUCC, ds.STREAM_Q_INTER))
        k, v = gen(ds.STREAM_K, t, T, w.Hkv), gen(ds.STREAM_V, t, T, w.Hkv)
        o = layer.dca_prefill(q, qs, qi, k, v, CL, mscale=msd[:, t:t + T].contiguous())
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        rows = sorted(r for r in {t, t + 1, t + T - 1} | {c + d for c in range(CL, L, CL) for d in (-1, 0)}
                      if t <= r < t + T)
        _check_rows(w, o, rows, heads, t, ms, keys)
        layer.append(k, v)
        t += T
