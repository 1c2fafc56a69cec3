"""duo_attn_decode on the GPU against the float64 oracle reading the oracle's cache model."""

import numpy as np
import pytest
import torch

import duo_synth as ds
import oracle
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import assert_close, device_stream, head_keys, host_stream, to_np

pytestmark = pytest.mark.gpu


def _decode_run(seed, B, Hq, Hkv, D, S, R, kinds, ctx, steps, poison=False, prefill_chunk=None):
    """Append a context of ctx tokens, then `steps` decode steps (append, then attend)."""
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    total = ctx + steps
    layer = DuoLayer(B, Hq, Hkv, D, S, R, total, kinds)
    if poison:
        for t in (layer.k_full, layer.v_full, layer.k_sr, layer.v_sr):
            t.fill_(float("nan"))
    chunk = prefill_chunk or 65536
    for c0 in range(0, ctx, chunk):
        T = min(chunk, ctx - c0)
        layer.append(device_stream(seed, ds.STREAM_K, B, c0, T, Hkv, D, "cuda"),
                     device_stream(seed, ds.STREAM_V, B, c0, T, Hkv, D, "cuda"))
    q = device_stream(seed, ds.STREAM_Q, B, ctx, steps, Hq, D, "cuda")
    kn = device_stream(seed, ds.STREAM_K, B, ctx, steps, Hkv, D, "cuda")
    vn = device_stream(seed, ds.STREAM_V, B, ctx, steps, Hkv, D, "cuda")
    outs = []
    for s in range(steps):
        layer.append(kn[:, s:s + 1].contiguous(), vn[:, s:s + 1].contiguous())
        outs.append(layer.decode(q[:, s].contiguous()))
    torch.cuda.synchronize()
    assert duo_device_error() == 0
    return torch.stack(outs, dim=1), layer  # [B, steps, Hq, D]


CASES = [
    # B, Hq, Hkv, D, S, R, kinds, ctx, steps
    (1, 4, 4, 64, 4, 32, [1, 0, 1, 0], 256, 16),     # the tiny workload
    (2, 8, 2, 128, 4, 64, [1, 0], 300, 5),
    (3, 16, 2, 128, 64, 256, [0, 1], 1000, 3),       # GQA 8
    (1, 4, 2, 64, 0, 1, [0, 1], 70, 4),              # window of one, no sinks
    (2, 2, 2, 128, 3, 5, [1, 1], 5, 4),              # all retrieval, tiny context
    (1, 4, 4, 128, 2, 9, [0, 0, 0, 0], 1, 20),       # all streaming, ring fills during decode
    (1, 8, 4, 64, 8, 40, [1, 0, 0, 1], 0, 30),       # decode from an empty cache
    (4, 8, 4, 128, 16, 100, [0, 1, 0, 0], 5000, 2),  # several tiles per unit
    # fewer retrieval tiles than CTAs (streaming units add CTAs): a unit's tiles must
    # not be cut over CTAs with empty shares, whose parts would never arrive
    (1, 4, 4, 128, 4, 32, [0, 0, 1, 0], 641, 2),
    (1, 8, 4, 64, 0, 1, [0, 0, 1, 0], 200, 2),
    (2, 16, 8, 128, 4, 32, [0, 0, 1, 0, 0, 0, 0, 1], 1000, 2),
]


@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_decode_matches_oracle(case):
    B, Hq, Hkv, D, S, R, kinds, ctx, steps = case
    seed = 200 + ctx % 97
    out, _ = _decode_run(seed, B, Hq, Hkv, D, S, R, kinds, ctx, steps)
    total = ctx + steps
    Q = host_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D)
    K = host_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D)
    V = host_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D)
    got = to_np(out)
    for b in range(B):
        cache = OracleCache(kinds, S, R, D)
        if ctx:
            cache.append(K[b, :ctx], V[b, :ctx])
        for s in range(steps):
            p = ctx + s
            cache.append(K[b, p:p + 1], V[b, p:p + 1])
            ref = decode_from_cache(Q[b, p], p, cache)
            assert_close(got[b, s], ref, f"b{b} step {s}")


@pytest.mark.parametrize("case", [
    (2, 8, 4, 128, 4, 64, [0, 1, 1, 0], 150, 6),     # g = 2: CUDA-core consumer
    (2, 16, 4, 128, 4, 64, [0, 1, 1, 0], 150, 6),    # g = 4: tensor-core slices
    (1, 16, 2, 64, 5, 27, [1, 0], 333, 4),           # g = 8, D 64, partial tiles
], ids=["g2", "g4", "g8"])
def test_poisoned_cache_tail_is_never_read(case):
    clean, _ = _decode_run(3, *case)
    dirty, _ = _decode_run(3, *case, poison=True)
    assert torch.isfinite(dirty.float()).all()
    assert torch.equal(clean, dirty)


def test_decode_equals_prefill_last_row():
    from streaming_kv_cache_duo_gb300 import DuoLayer
    B, Hq, Hkv, D, S, R, L = 1, 8, 2, 128, 4, 64, 700
    kinds = [1, 0]
    dec, _ = _decode_run(4, B, Hq, Hkv, D, S, R, kinds, L - 1, 1)
    layer = DuoLayer(B, Hq, Hkv, D, S, R, L, kinds)
    q = device_stream(4, ds.STREAM_Q, B, 0, L, Hq, D, "cuda")
    k = device_stream(4, ds.STREAM_K, B, 0, L, Hkv, D, "cuda")
    v = device_stream(4, ds.STREAM_V, B, 0, L, Hkv, D, "cuda")
    pre = layer.prefill(q, k, v)
    assert_close(to_np(dec[:, 0]), to_np(pre[:, L - 1]), "decode vs prefill row", atol=1e-2, mean_rel=3e-3)


def test_workspace_errors():
    from streaming_kv_cache_duo_gb300 import DuoError, DuoLayer, duo_attn_decode
    layer = DuoLayer(1, 4, 2, 64, 2, 8, 64, [1, 0])
    k = device_stream(1, ds.STREAM_K, 1, 0, 3, 2, 64, "cuda")
    layer.append(k, k)
    q = device_stream(1, ds.STREAM_Q, 1, 0, 1, 4, 64, "cuda")[:, 0].contiguous()
    o = torch.empty_like(q)
    with pytest.raises(DuoError, match="DUO_ERR_WORKSPACE"):
        duo_attn_decode(layer.handle, layer.cache, q, o, layer.workspace[:16])
    with pytest.raises(DuoError, match="DUO_ERR_INVALID_ARG"):
        duo_attn_decode(layer.handle, layer.cache, q, o, layer.workspace[8:])


def _check_sampled(w, out, steps_to_check, batches, heads_kv):
    g = w.Hq // w.Hkv
    got = to_np(out)
    for s in steps_to_check:
        p = w.context + s
        for b in batches:
            Qp = ds.stream_f64(w.seed, ds.STREAM_Q, w.B, p, 1, w.Hq, w.D)[b, 0]
            for h in heads_kv:
                if w.is_retrieval[h]:
                    K, V = head_keys(w.seed, b, h, 0, p + 1, w.D)
                    kpos = np.arange(p + 1)
                else:
                    sim = oracle.RingCacheSim(w.S, w.R)
                    sim.append(p + 1)
                    kpos = np.array([x for x in sim.positions() if x >= 0])
                    K = np.stack([ds.stream_f64(w.seed, ds.STREAM_K, w.B, int(t), 1, w.Hkv, w.D)[b, 0, h] for t in kpos])
                    V = np.stack([ds.stream_f64(w.seed, ds.STREAM_V, w.B, int(t), 1, w.Hkv, w.D)[b, 0, h] for t in kpos])
                ref = oracle.attend_rows(Qp[h * g:(h + 1) * g], [p] * g, K, V, kpos, w.is_retrieval[h], w.S, w.R)
                assert_close(got[b, s, h * g:(h + 1) * g], ref, f"step {s} b {b} kv head {h}")


def test_full_size_batched_decode_128k_sampled():
    """B = 8 sequences of 131072 context tokens, 32 / 8 heads, 2 retrieval KV heads,
    256 decode steps: sampled (step, sequence, head) outputs against the oracle."""
    w = ds.WORKLOADS["batched_decode_ctx128k"]
    out, _ = _decode_run(w.seed, w.B, w.Hq, w.Hkv, w.D, w.S, w.R, w.is_retrieval, w.context, w.decode_steps)
    _check_sampled(w, out, [0, w.decode_steps - 1], [0, w.B - 1], range(w.Hkv))
    _check_sampled(w, out, [100], [3], [h for h in range(w.Hkv) if w.is_retrieval[h]][:1])


def test_full_size_decode_1m_sampled():
    """One sequence of 1,048,576 context tokens, 2 retrieval KV heads, 64 decode steps."""
    w = ds.WORKLOADS["decode_ctx1m"]
    out, _ = _decode_run(w.seed, w.B, w.Hq, w.Hkv, w.D, w.S, w.R, w.is_retrieval, w.context, w.decode_steps)
    ret = [h for h in range(w.Hkv) if w.is_retrieval[h]]
    strh = [h for h in range(w.Hkv) if not w.is_retrieval[h]]
    _check_sampled(w, out, [w.decode_steps - 1], [0], ret[:1] + strh)
    _check_sampled(w, out, [0], [0], strh[:2])


@pytest.mark.parametrize("Hq", [4, 8], ids=["g2", "g4"])
def test_workspace_holding_other_data_between_calls(Hq):
    """A caller may lend the workspace's memory to other data between decode calls (a
    caching allocator does): with the same handle and address, a workspace filled with
    0xFF bytes between two steps still gives the oracle's output (nothing in it has to
    survive between calls). The context is long enough that one unit spans many CTAs."""
    from streaming_kv_cache_duo_gb300 import DuoLayer, duo_device_error
    B, Hkv, D, S, R, kinds, ctx = 1, 2, 128, 4, 64, [1, 0], 20000
    seed = 41
    layer = DuoLayer(B, Hq, Hkv, D, S, R, ctx + 2, kinds)
    layer.append(device_stream(seed, ds.STREAM_K, B, 0, ctx, Hkv, D, "cuda"),
                 device_stream(seed, ds.STREAM_V, B, 0, ctx, Hkv, D, "cuda"))
    K = host_stream(seed, ds.STREAM_K, B, 0, ctx + 2, Hkv, D)
    V = host_stream(seed, ds.STREAM_V, B, 0, ctx + 2, Hkv, D)
    cache = OracleCache(kinds, S, R, D)
    cache.append(K[0, :ctx], V[0, :ctx])
    addr = layer.workspace.data_ptr()
    for step in range(2):
        p = ctx + step
        layer.append(device_stream(seed, ds.STREAM_K, B, p, 1, Hkv, D, "cuda"),
                     device_stream(seed, ds.STREAM_V, B, p, 1, Hkv, D, "cuda"))
        q = device_stream(seed, ds.STREAM_Q, B, p, 1, Hq, D, "cuda")[:, 0].contiguous()
        o = layer.decode(q)
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        cache.append(K[0, p:p + 1], V[0, p:p + 1])
        ref = decode_from_cache(host_stream(seed, ds.STREAM_Q, B, p, 1, Hq, D)[0, 0], p, cache)
        assert_close(to_np(o[0]), ref, f"step {step}")
        layer.workspace.fill_(0xFF)  # the memory used for something else until the next call
    assert layer.workspace.data_ptr() == addr
