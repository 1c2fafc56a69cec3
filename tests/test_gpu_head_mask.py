"""duo_set_head_mask: re-classifying the heads of an existing handle gives exactly
what a handle created with the new mask gives (same caches, reset and refilled)."""

import pytest
import torch

import duo_synth as ds
from gpu_util import device_stream

pytestmark = pytest.mark.gpu


def _run(layer, Q, K, V, L):
    layer.reset()
    o = layer.prefill(Q[:, :L].contiguous(), K[:, :L].contiguous(), V[:, :L].contiguous())
    layer.append(K[:, :L + 1].contiguous(), V[:, :L + 1].contiguous())
    d = layer.decode(Q[:, L].contiguous())
    torch.cuda.synchronize()
    return o, d


def test_set_head_mask_equals_a_new_handle():
    from streaming_kv_cache_duo_gb300 import DuoLayer, _lib
    B, Hq, Hkv, D, S, R, L = 2, 8, 4, 128, 4, 64, 500
    Q = device_stream(5, ds.STREAM_Q, B, 0, L + 1, Hq, D, "cuda")
    K = device_stream(5, ds.STREAM_K, B, 0, L + 1, Hkv, D, "cuda")
    V = device_stream(5, ds.STREAM_V, B, 0, L + 1, Hkv, D, "cuda")
    old, new = [1, 0, 1, 0], [0, 1, 1, 0]  # same counts, so the cache tensors fit both
    layer = DuoLayer(B, Hq, Hkv, D, S, R, L + 1, old)
    _run(layer, Q, K, V, L)
    _lib.duo_set_head_mask(layer.handle, new)
    got = _run(layer, Q, K, V, L)
    want = _run(DuoLayer(B, Hq, Hkv, D, S, R, L + 1, new), Q, K, V, L)
    assert torch.equal(got[0], want[0]) and torch.equal(got[1], want[1])
