"""duo_attn_decode_static: decode for callers that cannot allocate device scratch.

Some callers cannot give the library a workspace: an engine that handed all device
memory to its own pool, or a loop that must not call cudaMalloc/cudaFree because
they may synchronise the device. This entry point keeps its scratch in a fixed
array inside the library instead. It is checked here, through the C ABI, against
the workspace-taking duo_attn_decode on two decode calls in a row. The file is
named so that pytest collects it last.
"""

import pytest
import torch

import duo_synth as ds
from gpu_util import assert_close, device_stream, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,Hq,Hkv,kinds", [
    (2, 8, 4, [1, 0, 0, 1]),             # g = 2: CUDA-core consumer
    (1, 32, 8, [1, 0, 0, 0, 0, 0, 1, 0]),  # g = 4: tensor-core slices
    (2, 16, 2, [0, 1]),                  # g = 8
], ids=["g2", "g4", "g8"])
def test_static_scratch_decode_matches_workspace_decode(B, Hq, Hkv, kinds):
    from streaming_kv_cache_duo_gb300 import DuoLayer, _lib, duo_device_error
    D, S, R, ctx = 128, 4, 64, 3000
    layer = DuoLayer(B, Hq, Hkv, D, S, R, ctx + 2, kinds)
    seed = 31
    layer.append(device_stream(seed, ds.STREAM_K, B, 0, ctx, Hkv, D, "cuda"),
                 device_stream(seed, ds.STREAM_V, B, 0, ctx, Hkv, D, "cuda"))
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
        assert_close(to_np(o_static), to_np(o_ws), f"call {step}")
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
