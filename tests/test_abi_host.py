"""The C ABI on the host (no GPU needed): the library loads, exports every function
include/duo_attn.h declares, and rejects bad arguments before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from streaming_kv_cache_duo_gb300 import _lib
    return _lib


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "duo_attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(duo_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 10
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in names:
        assert hasattr(raw, name), name
    assert sorted(lib.EXPORTS) == names


def test_classify_heads(lib):
    kidx, nr = lib.duo_classify_heads([1, 0, 1, 0, 0])
    assert nr == 2 and kidx == [0, 0, 1, 1, 2]
    kidx, nr = lib.duo_classify_heads([0, 0])
    assert nr == 0 and kidx == [0, 1]


@pytest.mark.parametrize("args,status", [
    (dict(head_dim=96), "DUO_ERR_UNSUPPORTED"),
    (dict(num_q_heads=6, num_kv_heads=4), "DUO_ERR_INVALID_ARG"),
    (dict(num_q_heads=48, num_kv_heads=3), "DUO_ERR_UNSUPPORTED"),
    (dict(recent_size=0), "DUO_ERR_INVALID_ARG"),
    (dict(sink_size=-1), "DUO_ERR_INVALID_ARG"),
    (dict(batch=0), "DUO_ERR_INVALID_ARG"),
    (dict(max_seq_len=0), "DUO_ERR_INVALID_ARG"),
])
def test_create_rejects_bad_config(lib, args, status):
    cfg = dict(batch=1, num_q_heads=8, num_kv_heads=4, head_dim=128, sink_size=4, recent_size=32,
               max_seq_len=1024)
    cfg.update(args)
    with pytest.raises(lib.DuoError) as e:
        lib.duo_create(cfg["batch"], cfg["num_q_heads"], cfg["num_kv_heads"], cfg["head_dim"], cfg["sink_size"],
                       cfg["recent_size"], cfg["max_seq_len"], [1] * cfg["num_kv_heads"])
    assert status in str(e.value)
    assert lib.duo_last_error() != ""


def test_null_handle_is_rejected(lib):
    cache = lib.duo_kv_cache()
    with pytest.raises(lib.DuoError) as e:
        lib.duo_kv_append(None, cache, None, None, 1, stream=0)
    assert "DUO_ERR_INVALID_ARG" in str(e.value)
    assert lib.duo_decode_workspace_size(None, 10) == 0


def test_status_strings(lib):
    assert lib.status_string(0) == "DUO_OK"
    assert lib.status_string(3) == "DUO_ERR_CAPACITY"


def test_paged_stream_dead_blocks_match_the_oracle(lib):
    from oracle.ring_cache import paged_stream_dead_blocks
    for S, R, bs in ((0, 1, 128), (4, 64, 128), (64, 256, 128), (200, 100, 256), (1, 1000, 384)):
        for n in list(range(0, 1200, 7)) + [4096, 65536 + 3]:
            lo, hi = lib.duo_paged_stream_dead_blocks(S, R, bs, n)
            if n < 5000:
                assert list(range(lo, hi)) == paged_stream_dead_blocks(n, S, R, bs), (S, R, bs, n)
            assert lo == -(-S // bs) and hi >= lo


@pytest.mark.parametrize("args,status", [((4, 0, 128, 10), "DUO_ERR_INVALID_ARG"),
                                         ((-1, 4, 128, 10), "DUO_ERR_INVALID_ARG"),
                                         ((4, 4, 100, 10), "DUO_ERR_UNSUPPORTED"),
                                         ((4, 4, 128, -1), "DUO_ERR_INVALID_ARG")])
def test_paged_stream_dead_blocks_rejects_bad_arguments(lib, args, status):
    with pytest.raises(lib.DuoError, match=status):
        lib.duo_paged_stream_dead_blocks(*args)


def test_set_head_mask_rejects_a_null_handle(lib):
    with pytest.raises(lib.DuoError, match="DUO_ERR_INVALID_ARG"):
        lib.duo_set_head_mask(None, [1, 0])
