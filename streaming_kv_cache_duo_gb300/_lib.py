"""ctypes binding of include/duo_attn.h: the same entry points, argument marshalling only.

Every function here checks the torch tensors it is handed (device, dtype, shape,
contiguity), passes raw pointers and sizes to the C ABI and raises ``DuoError``
on a non-OK status. All computation happens in the CUDA kernels of
``libduo_attn.so``; if the library is missing, importing it raises. There is no
CPU fallback.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_int32, c_int64, c_size_t, c_uint8, c_uint32, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libduo_attn.so")

DUO_OK = 0
DUO_ERR_INVALID_ARG = 1
DUO_ERR_UNSUPPORTED = 2
DUO_ERR_CAPACITY = 3
DUO_ERR_CUDA = 4
DUO_ERR_DEVICE_TIMEOUT = 5
DUO_ERR_WORKSPACE = 6

DUO_STREAMING = 0
DUO_RETRIEVAL = 1

# exported names of include/duo_attn.h (checked against the library by the tests)
EXPORTS = (
    "duo_classify_heads", "duo_create", "duo_destroy", "duo_set_head_mask", "duo_cache_reset", "duo_kv_append",
    "duo_attn_prefill", "duo_attn_prefill_select", "duo_decode_workspace_size", "duo_attn_decode",
    "duo_attn_decode_static", "duo_kv_append_paged", "duo_attn_prefill_paged", "duo_attn_decode_paged",
    "duo_paged_stream_dead_blocks", "duo_dca_prefill", "duo_dca_decode", "duo_kv_append_kv4",
    "duo_attn_decode_kv4", "duo_kv_append_kv4_paged", "duo_attn_decode_kv4_paged", "duo_attn_prefill_kv4",
    "duo_kv_append_varlen", "duo_attn_decode_varlen", "duo_device_error", "duo_selftest_bounded_wait",
    "duo_last_error", "duo_status_string",
)


class DuoError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


class duo_config(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("num_q_heads", c_int32), ("num_kv_heads", c_int32),
                ("head_dim", c_int32), ("sink_size", c_int32), ("recent_size", c_int32),
                ("max_seq_len", c_int64)]


class duo_paged(ctypes.Structure):
    _fields_ = [("block_table", c_void_p), ("block_size", c_int32), ("max_blocks", c_int32),
                ("num_blocks", c_int64), ("stream_table", c_void_p)]


class duo_kv4_cache(ctypes.Structure):
    _fields_ = [(name, c_void_p) for name in ("k_codes", "v_codes", "k_sz", "v_sz", "ks_codes", "vs_codes", "ks_sz",
                                              "vs_sz")]


class duo_kv_cache(ctypes.Structure):
    _fields_ = [("k_full", c_void_p), ("v_full", c_void_p), ("k_sr", c_void_p), ("v_sr", c_void_p),
                ("pos", c_void_p), ("n", c_int64)]


_LIB = None


def library() -> ctypes.CDLL:
    """Load libduo_attn.so (built in-tree by __graft_entry__.build())."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "duo_classify_heads": (c_int32, [POINTER(c_uint8), c_int32, POINTER(c_int32), POINTER(c_int32)]),
        "duo_create": (c_int32, [POINTER(duo_config), POINTER(c_uint8), POINTER(c_void_p)]),
        "duo_destroy": (None, [c_void_p]),
        "duo_set_head_mask": (c_int32, [c_void_p, POINTER(c_uint8)]),
        "duo_cache_reset": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p]),
        "duo_kv_append": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p, c_void_p, c_int32, c_void_p]),
        "duo_attn_prefill": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p, c_void_p, c_void_p, c_int32,
                                       c_void_p, c_void_p]),
        "duo_attn_prefill_select": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p, c_void_p, c_void_p,
                                              c_int32, c_void_p, c_int32, c_void_p]),
        "duo_decode_workspace_size": (c_size_t, [c_void_p, c_int64]),
        "duo_attn_decode": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p, c_void_p, c_void_p, c_size_t,
                                      c_void_p]),
        "duo_attn_decode_static": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p, c_void_p, c_void_p]),
        "duo_kv_append_paged": (c_int32, [c_void_p, POINTER(duo_kv_cache), POINTER(duo_paged), c_void_p, c_void_p,
                                          c_int32, c_void_p]),
        "duo_attn_prefill_paged": (c_int32, [c_void_p, POINTER(duo_kv_cache), POINTER(duo_paged), c_void_p,
                                             c_void_p, c_void_p, c_int32, c_void_p, c_void_p]),
        "duo_attn_decode_paged": (c_int32, [c_void_p, POINTER(duo_kv_cache), POINTER(duo_paged), c_void_p,
                                            c_void_p, c_void_p, c_size_t, c_void_p]),
        "duo_paged_stream_dead_blocks": (c_int32, [c_int32, c_int32, c_int32, c_int64, POINTER(c_int64),
                                                   POINTER(c_int64)]),
        "duo_kv_append_kv4": (c_int32, [c_void_p, POINTER(duo_kv_cache), POINTER(duo_kv4_cache), c_void_p, c_void_p,
                                        c_int32, c_void_p]),
        "duo_attn_decode_kv4": (c_int32, [c_void_p, POINTER(duo_kv_cache), POINTER(duo_kv4_cache), c_void_p,
                                          c_void_p, c_void_p, c_size_t, c_void_p]),
        "duo_attn_prefill_kv4": (c_int32, [c_void_p, POINTER(duo_kv_cache), POINTER(duo_kv4_cache), c_void_p,
                                           c_void_p, c_void_p, c_int32, c_void_p, c_void_p]),
        "duo_kv_append_kv4_paged": (c_int32, [c_void_p, POINTER(duo_kv_cache), POINTER(duo_paged),
                                              POINTER(duo_kv4_cache), c_void_p, c_void_p, c_int32, c_void_p]),
        "duo_attn_decode_kv4_paged": (c_int32, [c_void_p, POINTER(duo_kv_cache), POINTER(duo_paged),
                                                POINTER(duo_kv4_cache), c_void_p, c_void_p, c_void_p, c_size_t,
                                                c_void_p]),
        "duo_dca_prefill": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_int32, c_int32, c_void_p, c_void_p]),
        "duo_dca_decode": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_int32, c_void_p, c_void_p, c_size_t, c_void_p]),
        "duo_kv_append_varlen": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p, c_void_p, c_void_p,
                                           c_void_p]),
        "duo_attn_decode_varlen": (c_int32, [c_void_p, POINTER(duo_kv_cache), c_void_p, c_int64, c_void_p, c_void_p,
                                             c_void_p, c_size_t, c_void_p]),
        "duo_device_error": (c_int32, [POINTER(c_uint32)]),
        "duo_selftest_bounded_wait": (c_int32, [c_uint32, c_void_p]),
        "duo_last_error": (c_char_p, []),
        "duo_status_string": (c_char_p, [c_int32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    try:
        return library().duo_status_string(status).decode()
    except Exception:  # the library itself is missing
        return f"status {status}"


def _check(status: int) -> None:
    if status != DUO_OK:
        raise DuoError(status, library().duo_last_error().decode())


def _stream_ptr(stream) -> c_void_p:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t) -> c_void_p:
    return c_void_p(0 if t is None else t.data_ptr())


def _bf16(t, shape, name):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: need a contiguous CUDA bfloat16 tensor of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


# ---------------------------------------------------------------------- entry points
def duo_classify_heads(is_retrieval):
    """Per-head retrieval/streaming mask -> (kind_index list, n_retrieval)."""
    H = len(is_retrieval)
    arr = (c_uint8 * H)(*[1 if x else 0 for x in is_retrieval])
    kidx = (c_int32 * H)()
    nr = c_int32()
    _check(library().duo_classify_heads(arr, H, kidx, ctypes.byref(nr)))
    return list(kidx), nr.value


def duo_create(batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, max_seq_len, is_retrieval):
    cfg = duo_config(batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, max_seq_len)
    arr = (c_uint8 * num_kv_heads)(*[1 if x else 0 for x in is_retrieval])
    h = c_void_p()
    _check(library().duo_create(ctypes.byref(cfg), arr, ctypes.byref(h)))
    return h


def duo_destroy(handle) -> None:
    library().duo_destroy(handle)


def duo_set_head_mask(handle, is_retrieval) -> None:
    mask = (c_uint8 * len(is_retrieval))(*[1 if x else 0 for x in is_retrieval])
    _check(library().duo_set_head_mask(handle, mask))


def duo_cache_reset(handle, cache: "duo_kv_cache", stream=None) -> None:
    _check(library().duo_cache_reset(handle, ctypes.byref(cache), _stream_ptr(stream)))


def duo_kv_append(handle, cache: "duo_kv_cache", k_new, v_new, T: int, stream=None) -> None:
    _check(library().duo_kv_append(handle, ctypes.byref(cache), _ptr(k_new), _ptr(v_new), T, _stream_ptr(stream)))


def duo_attn_prefill(handle, cache: "duo_kv_cache", q, k, v, T: int, o, stream=None) -> None:
    _check(library().duo_attn_prefill(handle, ctypes.byref(cache), _ptr(q), _ptr(k), _ptr(v), T, _ptr(o),
                                      _stream_ptr(stream)))


def duo_attn_prefill_select(handle, cache: "duo_kv_cache", q, k, v, T: int, o, kind_mask: int,
                            stream=None) -> None:
    _check(library().duo_attn_prefill_select(handle, ctypes.byref(cache), _ptr(q), _ptr(k), _ptr(v), T, _ptr(o),
                                             kind_mask, _stream_ptr(stream)))


def duo_decode_workspace_size(handle, n: int) -> int:
    return int(library().duo_decode_workspace_size(handle, n))


def duo_attn_decode(handle, cache: "duo_kv_cache", q, o, workspace, stream=None) -> None:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().duo_attn_decode(handle, ctypes.byref(cache), _ptr(q), _ptr(o), _ptr(workspace), nbytes,
                                     _stream_ptr(stream)))


def duo_attn_decode_static(handle, cache: "duo_kv_cache", q, o, stream=None) -> None:
    """Decode with the library's built-in scratch array instead of a caller workspace,
    for callers that cannot allocate device memory (see include/duo_attn.h)."""
    _check(library().duo_attn_decode_static(handle, ctypes.byref(cache), _ptr(q), _ptr(o), _stream_ptr(stream)))


def duo_kv_append_paged(handle, cache: "duo_kv_cache", paged: "duo_paged", k_new, v_new, T: int,
                        stream=None) -> None:
    _check(library().duo_kv_append_paged(handle, ctypes.byref(cache), ctypes.byref(paged), _ptr(k_new), _ptr(v_new),
                                         T, _stream_ptr(stream)))


def duo_attn_prefill_paged(handle, cache: "duo_kv_cache", paged: "duo_paged", q, k, v, T: int, o,
                           stream=None) -> None:
    _check(library().duo_attn_prefill_paged(handle, ctypes.byref(cache), ctypes.byref(paged), _ptr(q), _ptr(k),
                                            _ptr(v), T, _ptr(o), _stream_ptr(stream)))


def duo_attn_decode_paged(handle, cache: "duo_kv_cache", paged: "duo_paged", q, o, workspace, stream=None) -> None:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().duo_attn_decode_paged(handle, ctypes.byref(cache), ctypes.byref(paged), _ptr(q), _ptr(o),
                                           _ptr(workspace), nbytes, _stream_ptr(stream)))


def duo_kv_append_kv4(handle, cache: "duo_kv_cache", kv4: "duo_kv4_cache", k_new, v_new, T: int,
                      stream=None) -> None:
    _check(library().duo_kv_append_kv4(handle, ctypes.byref(cache), ctypes.byref(kv4), _ptr(k_new), _ptr(v_new), T,
                                       _stream_ptr(stream)))


def duo_attn_decode_kv4(handle, cache: "duo_kv_cache", kv4: "duo_kv4_cache", q, o, workspace, stream=None) -> None:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().duo_attn_decode_kv4(handle, ctypes.byref(cache), ctypes.byref(kv4), _ptr(q), _ptr(o),
                                         _ptr(workspace), nbytes, _stream_ptr(stream)))


def duo_attn_prefill_kv4(handle, cache: "duo_kv_cache", kv4: "duo_kv4_cache", q, k, v, T: int, o,
                         stream=None) -> None:
    _check(library().duo_attn_prefill_kv4(handle, ctypes.byref(cache), ctypes.byref(kv4), _ptr(q), _ptr(k), _ptr(v),
                                          T, _ptr(o), _stream_ptr(stream)))


def duo_kv_append_kv4_paged(handle, cache: "duo_kv_cache", paged: "duo_paged", kv4: "duo_kv4_cache", k_new, v_new,
                            T: int, stream=None) -> None:
    _check(library().duo_kv_append_kv4_paged(handle, ctypes.byref(cache), ctypes.byref(paged), ctypes.byref(kv4),
                                             _ptr(k_new), _ptr(v_new), T, _stream_ptr(stream)))


def duo_attn_decode_kv4_paged(handle, cache: "duo_kv_cache", paged: "duo_paged", kv4: "duo_kv4_cache", q, o,
                              workspace, stream=None) -> None:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().duo_attn_decode_kv4_paged(handle, ctypes.byref(cache), ctypes.byref(paged), ctypes.byref(kv4),
                                               _ptr(q), _ptr(o), _ptr(workspace), nbytes, _stream_ptr(stream)))


def duo_dca_prefill(handle, cache, q, q_succ, q_inter, k, v, mscale, T: int, chunk_len: int, o,
                    stream=None) -> None:
    _check(library().duo_dca_prefill(handle, None if cache is None else ctypes.byref(cache), _ptr(q), _ptr(q_succ),
                                     _ptr(q_inter), _ptr(k), _ptr(v), _ptr(mscale), T, chunk_len, _ptr(o),
                                     _stream_ptr(stream)))


def duo_dca_decode(handle, cache: "duo_kv_cache", q, q_succ, q_inter, mscale, chunk_len: int, o, workspace,
                   stream=None) -> None:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().duo_dca_decode(handle, ctypes.byref(cache), _ptr(q), _ptr(q_succ), _ptr(q_inter), _ptr(mscale),
                                    chunk_len, _ptr(o), _ptr(workspace), nbytes, _stream_ptr(stream)))


def duo_paged_stream_dead_blocks(sink_size: int, recent_size: int, block_size: int, n: int) -> tuple:
    """(lo, hi): logical blocks of a paged streaming head no later query can see."""
    lo, hi = c_int64(0), c_int64(0)
    _check(library().duo_paged_stream_dead_blocks(sink_size, recent_size, block_size, n, ctypes.byref(lo),
                                                  ctypes.byref(hi)))
    return int(lo.value), int(hi.value)


def duo_kv_append_varlen(handle, cache: "duo_kv_cache", seq_lens, k_new, v_new, stream=None) -> None:
    """One token per sequence at the device-held positions seq_lens (int32 [B]), then seq_lens += 1."""
    _check(library().duo_kv_append_varlen(handle, ctypes.byref(cache), _ptr(seq_lens), _ptr(k_new), _ptr(v_new),
                                          _stream_ptr(stream)))


def duo_attn_decode_varlen(handle, cache: "duo_kv_cache", seq_lens, max_len: int, q, o, workspace,
                           stream=None) -> None:
    """Decode with per-sequence lengths read on the device (launch shape planned for max_len)."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(library().duo_attn_decode_varlen(handle, ctypes.byref(cache), _ptr(seq_lens), max_len, _ptr(q), _ptr(o),
                                            _ptr(workspace), nbytes, _stream_ptr(stream)))


def duo_device_error() -> int:
    """Synchronise; return the kernels' recorded error code (0 = none)."""
    code = c_uint32()
    st = library().duo_device_error(ctypes.byref(code))
    if code.value == 0:
        _check(st)
    return code.value


def duo_selftest_bounded_wait(limit_us: int, stream=None) -> None:
    """Launch a kernel whose bounded wait must run out (failure-detection self-test)."""
    _check(library().duo_selftest_bounded_wait(limit_us, _stream_ptr(stream)))


def duo_last_error() -> str:
    return library().duo_last_error().decode()
