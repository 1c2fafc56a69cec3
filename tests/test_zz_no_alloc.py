"""duo_attn_decode_static: decode for callers that cannot allocate device scratch.

Some callers cannot give the library a workspace: an engine that handed all device
memory to its own pool, or a loop that must not call cudaMalloc/cudaFree because
they may synchronise the device. This entry point keeps its scratch in a fixed
array inside the library instead. It is checked here, through the C ABI, against
the workspace-taking duo_attn_decode and against the float64 oracle, on two decode
calls in a row, for both head dims, every consumer of the decode kernel and a shape
whose scratch need lies just under the array's size (one sequence more is
rejected). The file is named so that pytest collects it last.
"""

import pytest
import torch

import duo_synth as ds
from oracle.attention import OracleCache, decode_from_cache
from gpu_util import assert_close, device_stream, host_stream, to_np

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 2 << 20  # the array's size, as include/duo_attn.h states it


def _scratch_need(B, Hq, Hkv, D, num_sms):
    """Decode scratch of a shape as the header defines it: (SMs + units) partial slots of
    g x (D + 4) floats."""
    U = B * Hkv
    return (num_sms + U) * (Hq // Hkv) * (D + 4) * 4


def _run(B, Hq, Hkv, D, S, R, kinds, ctx, seed, check_batches=None):
    from streaming_kv_cache_duo_gb300 import DuoLayer, _lib, duo_device_error
    layer = DuoLayer(B, Hq, Hkv, D, S, R, ctx + 2, kinds)
    layer.append(device_stream(seed, ds.STREAM_K, B, 0, ctx, Hkv, D, "cuda"),
                 device_stream(seed, ds.STREAM_V, B, 0, ctx, Hkv, D, "cuda"))
    K = host_stream(seed, ds.STREAM_K, B, 0, ctx + 2, Hkv, D)
    V = host_stream(seed, ds.STREAM_V, B, 0, ctx + 2, Hkv, D)
    batches = range(B) if check_batches is None else check_batches
    caches = {b: OracleCache(kinds, S, R, D) for b in batches}
    for b in batches:
        caches[b].append(K[b, :ctx], V[b, :ctx])
    for step in range(2):  # two calls in a row share the library's one scratch array
        p = ctx + step
        layer.append(device_stream(seed, ds.STREAM_K, B, p, 1, Hkv, D, "cuda"),
                     device_stream(seed, ds.STREAM_V, B, p, 1, Hkv, D, "cuda"))
        q = device_stream(seed, ds.STREAM_Q, B, p, 1, Hq, D, "cuda")[:, 0].contiguous()
        o_ws = torch.empty_like(q)
        o_static = torch.full_like(q, float("nan"))
        _lib.duo_attn_decode(layer.handle, layer.cache, q, o_ws, layer.workspace)
        _lib.duo_attn_decode_static(layer.handle, layer.cache, q, o_static)
        torch.cuda.synchronize()
        assert duo_device_error() == 0
        assert_close(to_np(o_static), to_np(o_ws), f"call {step}: static vs workspace")
        Q = host_stream(seed, ds.STREAM_Q, B, p, 1, Hq, D)[:, 0]
        got = to_np(o_static)
        for b in batches:
            caches[b].append(K[b, p:p + 1], V[b, p:p + 1])
            assert_close(got[b], decode_from_cache(Q[b], p, caches[b]), f"call {step}: static vs oracle, b{b}")
    layer.close()


@pytest.mark.parametrize("B,Hq,Hkv,D,kinds", [
    (2, 8, 4, 128, [1, 0, 0, 1]),               # g = 2: CUDA-core consumer
    (1, 32, 8, 128, [1, 0, 0, 0, 0, 0, 1, 0]),  # g = 4: tensor-core slices
    (2, 16, 2, 128, [0, 1]),                    # g = 8
    (2, 8, 8, 64, [1, 0, 1, 0, 0, 0, 0, 1]),    # g = 1, D = 64
    (1, 16, 4, 64, [0, 1, 1, 0]),               # g = 4, D = 64
], ids=["g2", "g4", "g8", "g1-d64", "g4-d64"])
def test_static_scratch_decode_matches_workspace_decode_and_oracle(B, Hq, Hkv, D, kinds):
    _run(B, Hq, Hkv, D, 4, 64, kinds, 3000, 31)


def test_static_scratch_just_under_its_size():
    """The largest batch of a 64 / 8-head, D = 128 layer whose scratch fits the array
    runs and matches; one sequence more is rejected."""
    from streaming_kv_cache_duo_gb300 import DuoError, DuoLayer, _lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hq, Hkv, D = 64, 8, 128
    B = 1
    while _scratch_need(B + 1, Hq, Hkv, D, sms) <= STATIC_SCRATCH_BYTES:
        B += 1
    assert _scratch_need(B, Hq, Hkv, D, sms) > STATIC_SCRATCH_BYTES - 8 * (D + 4) * 4 * 8
    kinds = [1, 0, 0, 1, 0, 0, 0, 1]
    _run(B, Hq, Hkv, D, 4, 60, kinds, 300, 37, check_batches=[0, B // 2, B - 1])
    layer = DuoLayer(B + 1, Hq, Hkv, D, 4, 60, 8, kinds)
    k = torch.zeros((B + 1, 1, Hkv, D), dtype=torch.bfloat16, device="cuda")
    layer.append(k, k)
    q = torch.zeros((B + 1, Hq, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(DuoError, match="DUO_ERR_WORKSPACE"):
        _lib.duo_attn_decode_static(layer.handle, layer.cache, q, torch.empty_like(q))
    layer.close()


def test_static_scratch_rejects_shapes_beyond_its_size():
    from streaming_kv_cache_duo_gb300 import DuoError, DuoLayer, _lib
    # 64 sequences x 32 KV heads x 8 query heads each need ~9 MB of scratch (> 2 MiB)
    layer = DuoLayer(64, 256, 32, 128, 4, 60, 8, [1] * 32)
    k = torch.zeros((64, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    layer.append(k, k)
    q = torch.zeros((64, 256, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    with pytest.raises(DuoError, match="DUO_ERR_WORKSPACE"):
        _lib.duo_attn_decode_static(layer.handle, layer.cache, q, o)
    layer.close()
