"""Failure detection without a GPU fault: a kernel's bounded wait runs out (an
mbarrier that nothing completes), the host reads DUO_ERR_DEVICE_TIMEOUT through
duo_device_error(), and the context keeps working afterwards."""

import pytest
import torch

import duo_synth as ds
from gpu_util import device_stream

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    from streaming_kv_cache_duo_gb300 import DuoLayer, _lib
    assert _lib.duo_device_error() == 0
    _lib.duo_selftest_bounded_wait(20000)  # 20 ms
    code = _lib.duo_device_error()
    assert code & (1 << 16)
    assert _lib.duo_device_error() == 0  # read-and-clear
    # the context is still usable: a small decode runs and is finite
    layer = DuoLayer(1, 4, 2, 64, 2, 8, 32, [1, 0])
    k = device_stream(1, ds.STREAM_K, 1, 0, 5, 2, 64, "cuda")
    layer.append(k, k)
    q = device_stream(1, ds.STREAM_Q, 1, 4, 1, 4, 64, "cuda")[:, 0].contiguous()
    o = layer.decode(q)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    assert _lib.duo_device_error() == 0


def test_selftest_limit_is_validated():
    from streaming_kv_cache_duo_gb300 import DuoError, _lib
    with pytest.raises(DuoError, match="DUO_ERR_INVALID_ARG"):
        _lib.duo_selftest_bounded_wait(0)
