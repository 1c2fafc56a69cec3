"""Chunked prefill against 4-bit caches (duo_attn_prefill_kv4): each chunk attends to
the cache as it was before the chunk, read as 4-bit rows and dequantized inside the
kernel, and to its own bf16 keys and values; then the chunk is appended with
duo_kv_append_kv4. Checked against the float64 oracle attending over exactly that key
set (the dequantized rows of earlier positions, the exact rows of the chunk), every row
of every head, then a decode step over the caches the chunks left behind."""

import numpy as np
import pytest
import torch

import duo_synth as ds
import oracle
import oracle.kv4 as kv4
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import assert_close, device_stream, host_stream, to_np

pytestmark = pytest.mark.gpu

CASES = [
    # B, Hq, Hkv, D, S, R, kinds, chunks
    (1, 8, 2, 128, 4, 64, [1, 0], [300, 200, 129]),          # ragged chunks, partial cache tiles
    (2, 8, 4, 64, 8, 100, [1, 0, 0, 1], [256, 256, 40]),      # D 64, two sequences
    (1, 16, 2, 128, 64, 256, [0, 1], [512, 700, 333]),        # GQA 8, window spans chunks
    (1, 32, 32, 128, 64, 256, [1] * 8 + [0] * 24, [1024, 1024, 1024]),  # MHA, 8 retrieval heads
    (1, 4, 4, 128, 70, 90, [0, 1, 0, 1], [50, 40, 300]),      # sinks spread over chunks
    (1, 8, 2, 128, 16, 200, [0, 0], [333, 444]),              # streaming heads only
    (2, 4, 4, 64, 0, 1, [1, 1, 1, 1], [128, 129, 255]),       # retrieval heads only, D 64
]


def _bf16(x):
    """Round to bf16 (nearest even), back to float64: the tensor cores' operand type."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("qscale", [1, 16], ids=["plain", "q16"])
@pytest.mark.parametrize("case", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_prefill_against_kv4_cache_matches_oracle(case, qscale):
    """qscale 16: queries times 16 (exact in bf16), so rows take the kernel's lazy rescale of
    the running output after their first tile, here with dequantized cache tiles.

    The products run on bf16 tensor-core operands, so a dequantized cache row enters them
    rounded to bf16 (relative error up to 2^-9 per element, against 2^-11 for the fp16
    rows of the 4-bit decode). That error scales with the logits: with plain queries the
    float64 oracle over the bf16-rounded rows and over the exact rows differ by about
    2e-3, with queries times 16 by about 0.1, far above the bf16 output tolerance. So every
    case is checked against the oracle over the rows as the operands hold them (dequantized,
    then rounded to bf16), and plain queries also against the exact dequantized rows."""
    from streaming_kv_cache_duo_gb300 import DuoKv4Layer, duo_device_error
    B, Hq, Hkv, D, S, R, kinds, chunks = case
    total = sum(chunks) + 1
    seed = 1700 + total % 89
    layer = DuoKv4Layer(B, Hq, Hkv, D, S, R, total, kinds)
    q = device_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D, "cuda") * qscale
    k = device_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D, "cuda")
    v = device_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D, "cuda")
    outs, t = [], 0
    for c in chunks:
        qs, ks, vs = (x[:, t:t + c].contiguous() for x in (q, k, v))
        outs.append(to_np(layer.prefill(qs, ks, vs)))
        layer.append(ks, vs)
        t += c
    p = t  # one decode step over what the chunks left in the 4-bit caches
    layer.append(k[:, p:p + 1].contiguous(), v[:, p:p + 1].contiguous())
    dec = to_np(layer.decode(q[:, p].contiguous()))
    torch.cuda.synchronize()
    assert duo_device_error() == 0

    Qh = host_stream(seed, ds.STREAM_Q, B, 0, total, Hq, D) * qscale
    Kh = host_stream(seed, ds.STREAM_K, B, 0, total, Hkv, D)
    Vh = host_stream(seed, ds.STREAM_V, B, 0, total, Hkv, D)
    Kq, Vq = kv4.roundtrip(Kh.astype(np.float32)), kv4.roundtrip(Vh.astype(np.float32))
    Kb, Vb = _bf16(Kq), _bf16(Vq)
    for b in range(B):
        n0 = 0
        for ci, c in enumerate(chunks):
            # keys before the chunk as the cache holds them, the chunk's own exactly
            rows = np.arange(n0, n0 + c)
            K = np.concatenate([Kb[b, :n0], Kh[b, n0:n0 + c]])
            V = np.concatenate([Vb[b, :n0], Vh[b, n0:n0 + c]])
            ref = oracle.prefill(Qh[b, :n0 + c], K, V, kinds, S, R, rows=rows)
            assert_close(outs[ci][b], ref, f"b{b} chunk {ci}")
            if qscale == 1:
                K = np.concatenate([Kq[b, :n0], Kh[b, n0:n0 + c]])
                V = np.concatenate([Vq[b, :n0], Vh[b, n0:n0 + c]])
                ref = oracle.prefill(Qh[b, :n0 + c], K, V, kinds, S, R, rows=rows)
                assert_close(outs[ci][b], ref, f"b{b} chunk {ci}, exact rows")
            n0 += c
        cache = OracleCache(kinds, S, R, D)
        cache.append(Kq[b, :p + 1], Vq[b, :p + 1])
        assert_close(dec[b], decode_from_cache(Qh[b, p], p, cache), f"b{b} decode")


def test_prefill_kv4_equals_prefill_over_the_dequantized_cache():
    """The fused dequantization gives the same attention as the bf16 prefill over a bf16
    cache holding the dequantized rows (rounded to bf16, as the kernel rounds them)."""
    from streaming_kv_cache_duo_gb300 import DuoKv4Layer, DuoLayer
    B, Hq, Hkv, D, S, R, kinds = 1, 8, 4, 128, 4, 64, [1, 0, 1, 0]
    n0, T = 700, 300
    seed = 1777
    k = host_stream(seed, ds.STREAM_K, B, 0, n0 + T, Hkv, D)
    v = host_stream(seed, ds.STREAM_V, B, 0, n0 + T, Hkv, D)
    q = device_stream(seed, ds.STREAM_Q, B, n0, T, Hq, D, "cuda")
    kd = torch.from_numpy(k.astype(np.float32)).to(torch.bfloat16).cuda()
    vd = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).cuda()
    kq = torch.from_numpy(kv4.roundtrip(k.astype(np.float32)).astype(np.float32)).to(torch.bfloat16).cuda()
    vq = torch.from_numpy(kv4.roundtrip(v.astype(np.float32)).astype(np.float32)).to(torch.bfloat16).cuda()
    a = DuoKv4Layer(B, Hq, Hkv, D, S, R, n0 + T, kinds)
    a.append(kd[:, :n0].contiguous(), vd[:, :n0].contiguous())
    b = DuoLayer(B, Hq, Hkv, D, S, R, n0 + T, kinds)
    b.append(kq[:, :n0].contiguous(), vq[:, :n0].contiguous())
    kc, vc = kd[:, n0:].contiguous(), vd[:, n0:].contiguous()
    oa = a.prefill(q, kc, vc)
    ob = b.prefill(q, kc, vc)
    torch.cuda.synchronize()
    # fp32 code * scale + zero, then bf16: equal to the bf16 rounding of the exact value
    # except where an fp32 product straddles a bf16 rounding boundary
    assert_close(to_np(oa), to_np(ob), "kv4 prefill vs bf16 prefill", atol=4e-3, mean_rel=1e-3)
