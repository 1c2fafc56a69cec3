"""GB300-native mixed-head causal attention (retrieval + streaming heads) for long-context serving.

The product is the C ABI in ``include/duo_attn.h``, implemented by
``libduo_attn.so`` (hand-written sm_103a kernels). This package holds its thin
ctypes binding (``_lib``, the same entry-point names), ``DuoLayer`` -- a small
owner of the torch tensors one layer's caches live in -- and the algorithmic
work counters used to report throughput (``workload``).
"""

from __future__ import annotations

from . import _lib
from ._lib import (DUO_RETRIEVAL, DUO_STREAMING, DuoError, duo_attn_decode, duo_attn_decode_varlen,  # noqa: F401
                   duo_attn_prefill, duo_attn_prefill_select, duo_cache_reset, duo_classify_heads, duo_create,
                   duo_decode_workspace_size, duo_destroy, duo_device_error, duo_kv_append, duo_kv_append_varlen,
                   duo_last_error, duo_paged_stream_dead_blocks)


class DuoLayer:
    """Caches of one attention layer in torch device memory plus a library handle.

    k_full/v_full: bf16 [B, n_ret, max_seq_len, D]; k_sr/v_sr: bf16 [B, n_str, S+R, D];
    pos: int32 [B, S+R]; ``n`` tokens appended so far. ``workspace`` is the decode
    workspace (zero-filled once)."""

    def __init__(self, batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, max_seq_len,
                 is_retrieval, device="cuda"):
        import torch
        self.B, self.Hq, self.Hkv, self.D = batch, num_q_heads, num_kv_heads, head_dim
        self.S, self.R, self.cap = sink_size, recent_size, max_seq_len
        self.is_retrieval = [1 if x else 0 for x in is_retrieval]
        self.kind_index, self.n_ret = duo_classify_heads(self.is_retrieval)
        self.n_str = num_kv_heads - self.n_ret
        self.device = torch.device(device)
        with torch.cuda.device(self.device):
            self.handle = duo_create(batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size,
                                     max_seq_len, self.is_retrieval)
        bf = dict(dtype=torch.bfloat16, device=self.device)
        SR = sink_size + recent_size
        self.k_full = torch.empty((batch, self.n_ret, max_seq_len if self.n_ret else 0, head_dim), **bf)
        self.v_full = torch.empty_like(self.k_full)
        self.k_sr = torch.empty((batch, self.n_str, SR, head_dim), **bf)
        self.v_sr = torch.empty_like(self.k_sr)
        self.pos = torch.empty((batch, SR), dtype=torch.int32, device=self.device)
        ws = duo_decode_workspace_size(self.handle, 1)
        self.workspace = torch.zeros(((ws + 255) // 256) * 256, dtype=torch.uint8, device=self.device)
        self.cache = _lib.duo_kv_cache(self.k_full.data_ptr() if self.n_ret else None,
                                       self.v_full.data_ptr() if self.n_ret else None,
                                       self.k_sr.data_ptr() if self.n_str else None,
                                       self.v_sr.data_ptr() if self.n_str else None,
                                       self.pos.data_ptr(), 0)
        self.reset()

    @property
    def n(self) -> int:
        return int(self.cache.n)

    def reset(self, stream=None) -> None:
        duo_cache_reset(self.handle, self.cache, stream)

    def append(self, k_new, v_new, stream=None) -> None:
        T = k_new.shape[1]
        _lib._bf16(k_new, (self.B, T, self.Hkv, self.D), "k_new")
        _lib._bf16(v_new, (self.B, T, self.Hkv, self.D), "v_new")
        duo_kv_append(self.handle, self.cache, k_new, v_new, T, stream)

    def prefill(self, q, k, v, out=None, kind_mask=3, stream=None):
        import torch
        T = q.shape[1]
        _lib._bf16(q, (self.B, T, self.Hq, self.D), "q")
        _lib._bf16(k, (self.B, T, self.Hkv, self.D), "k")
        _lib._bf16(v, (self.B, T, self.Hkv, self.D), "v")
        if out is None:
            out = torch.empty_like(q)
        _lib._bf16(out, (self.B, T, self.Hq, self.D), "o")
        duo_attn_prefill_select(self.handle, self.cache, q, k, v, T, out, kind_mask, stream)
        return out

    def decode(self, q, out=None, stream=None):
        import torch
        _lib._bf16(q, (self.B, self.Hq, self.D), "q")
        if out is None:
            out = torch.empty_like(q)
        _lib._bf16(out, (self.B, self.Hq, self.D), "o")
        duo_attn_decode(self.handle, self.cache, q, out, self.workspace, stream)
        return out

    def dca_prefill(self, q, q_succ, q_inter, k, v, chunk_len, mscale=None, out=None, stream=None):
        """Dual Chunk Attention prefill of T tokens at positions n ... n+T-1 against the cache
        (n = tokens appended so far, a multiple of 256; every head full attention); mscale:
        fp32 [B, T] on the device or None."""
        import torch
        T = q.shape[1]
        for name, t in (("q", q), ("q_succ", q_succ), ("q_inter", q_inter)):
            _lib._bf16(t, (self.B, T, self.Hq, self.D), name)
        _lib._bf16(k, (self.B, T, self.Hkv, self.D), "k")
        _lib._bf16(v, (self.B, T, self.Hkv, self.D), "v")
        _check_mscale(mscale, (self.B, T))
        if out is None:
            out = torch.empty_like(q)
        _lib._bf16(out, (self.B, T, self.Hq, self.D), "o")
        _lib.duo_dca_prefill(self.handle, self.cache, q, q_succ, q_inter, k, v, mscale, T, chunk_len, out, stream)
        return out

    def dca_decode(self, q, q_succ, q_inter, chunk_len, mscale=None, out=None, stream=None):
        """Dual Chunk Attention decode of the token at position n - 1; mscale fp32 [B] or None."""
        import torch
        for name, t in (("q", q), ("q_succ", q_succ), ("q_inter", q_inter)):
            _lib._bf16(t, (self.B, self.Hq, self.D), name)
        _check_mscale(mscale, (self.B,))
        if out is None:
            out = torch.empty_like(q)
        _lib._bf16(out, (self.B, self.Hq, self.D), "o")
        _lib.duo_dca_decode(self.handle, self.cache, q, q_succ, q_inter, mscale, chunk_len, out, self.workspace, stream)
        return out

    def append_varlen(self, k_new, v_new, seq_lens, stream=None) -> None:
        """One token per sequence at positions seq_lens (device int32 [B]), which advance by one."""
        _lib._bf16(k_new, (self.B, 1, self.Hkv, self.D), "k_new")
        _lib._bf16(v_new, (self.B, 1, self.Hkv, self.D), "v_new")
        _check_lens(seq_lens, self.B)
        duo_kv_append_varlen(self.handle, self.cache, seq_lens, k_new, v_new, stream)

    def decode_varlen(self, q, seq_lens, max_len, out=None, stream=None):
        """Decode where sequence b holds seq_lens[b] tokens (device int32 [B], <= max_len)."""
        import torch
        _lib._bf16(q, (self.B, self.Hq, self.D), "q")
        _check_lens(seq_lens, self.B)
        if out is None:
            out = torch.empty_like(q)
        _lib._bf16(out, (self.B, self.Hq, self.D), "o")
        duo_attn_decode_varlen(self.handle, self.cache, seq_lens, max_len, q, out, self.workspace, stream)
        return out

    def close(self) -> None:
        if getattr(self, "handle", None) is not None:
            duo_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DuoPagedLayer(DuoLayer):
    """A layer whose caches live in a shared pool of blocks addressed through block
    tables (device int32): retrieval heads through ``block_table`` [B, n_ret,
    max_blocks]; streaming heads through ``stream_table`` [B, n_str, max_blocks] when
    given (block-granular eviction: ``dead_blocks()`` names the blocks the caller may
    free), else they keep the sink + ring cache."""

    def __init__(self, batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, block_size,
                 max_blocks, num_blocks, block_table, is_retrieval, device="cuda", stream_table=None):
        import torch
        super().__init__(batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, 1, is_retrieval,
                         device=device)
        bf = dict(dtype=torch.bfloat16, device=self.device)
        self.block_size = block_size
        self.k_full = torch.empty((num_blocks, block_size, head_dim), **bf)
        self.v_full = torch.empty_like(self.k_full)
        self.cache.k_full = self.k_full.data_ptr()
        self.cache.v_full = self.v_full.data_ptr()
        for name, t, rows in (("block_table", block_table, self.n_ret), ("stream_table", stream_table, self.n_str)):
            if t is not None:
                assert t.dtype == torch.int32 and t.is_cuda and t.is_contiguous(), name
                assert tuple(t.shape) == (batch, rows, max_blocks), name
        self.block_table = block_table
        self.stream_table = stream_table
        self.paged = _lib.duo_paged(block_table.data_ptr() if block_table is not None else None, block_size,
                                    max_blocks, num_blocks,
                                    stream_table.data_ptr() if stream_table is not None else None)

    def dead_blocks(self, n=None) -> tuple:
        """Logical blocks [lo, hi) of every streaming head that no query can see any more."""
        return _lib.duo_paged_stream_dead_blocks(self.S, self.R, self.block_size, self.n if n is None else n)

    def append(self, k_new, v_new, stream=None) -> None:
        T = k_new.shape[1]
        _lib._bf16(k_new, (self.B, T, self.Hkv, self.D), "k_new")
        _lib._bf16(v_new, (self.B, T, self.Hkv, self.D), "v_new")
        _lib.duo_kv_append_paged(self.handle, self.cache, self.paged, k_new, v_new, T, stream)

    def prefill(self, q, k, v, out=None, kind_mask=3, stream=None):
        import torch
        assert kind_mask == 3
        T = q.shape[1]
        _lib._bf16(q, (self.B, T, self.Hq, self.D), "q")
        if out is None:
            out = torch.empty_like(q)
        _lib.duo_attn_prefill_paged(self.handle, self.cache, self.paged, q, k, v, T, out, stream)
        return out

    def decode(self, q, out=None, stream=None):
        import torch
        _lib._bf16(q, (self.B, self.Hq, self.D), "q")
        if out is None:
            out = torch.empty_like(q)
        _lib.duo_attn_decode_paged(self.handle, self.cache, self.paged, q, out, self.workspace, stream)
        return out


class DuoKv4Layer(DuoLayer):
    """A layer whose caches hold 4-bit codes with an fp16 (scale, zero) pair per row
    (layout in include/duo_attn.h): codes u8 [B, planes, pitch, D/2] and pairs int32
    [B, planes, pitch], pitch = capacity rounded up to 16 rows. Prefill attention is
    computed from bf16 inputs as usual; appends quantize; decode reads the codes."""

    def __init__(self, batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, max_seq_len,
                 is_retrieval, device="cuda"):
        import torch
        super().__init__(batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, 1, is_retrieval,
                         device=device)
        self.cap = max_seq_len
        cap16 = -(-max_seq_len // 16) * 16
        sr16 = -(-(sink_size + recent_size) // 16) * 16
        u8 = dict(dtype=torch.uint8, device=self.device)
        i32 = dict(dtype=torch.int32, device=self.device)
        self.k_codes = torch.zeros((batch, self.n_ret, cap16 if self.n_ret else 0, head_dim // 2), **u8)
        self.v_codes = torch.zeros_like(self.k_codes)
        self.k_sz = torch.zeros((batch, self.n_ret, cap16 if self.n_ret else 0), **i32)
        self.v_sz = torch.zeros_like(self.k_sz)
        self.ks_codes = torch.zeros((batch, self.n_str, sr16, head_dim // 2), **u8)
        self.vs_codes = torch.zeros_like(self.ks_codes)
        self.ks_sz = torch.zeros((batch, self.n_str, sr16), **i32)
        self.vs_sz = torch.zeros_like(self.ks_sz)
        # the handle's capacity is max_seq_len: recreate it with the real value
        duo_destroy(self.handle)
        with torch.cuda.device(self.device):
            self.handle = duo_create(batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, max_seq_len,
                                     self.is_retrieval)
        ptr = lambda t: t.data_ptr() if t.numel() else None
        self.kv4 = _lib.duo_kv4_cache(ptr(self.k_codes), ptr(self.v_codes), ptr(self.k_sz), ptr(self.v_sz),
                                      ptr(self.ks_codes), ptr(self.vs_codes), ptr(self.ks_sz), ptr(self.vs_sz))
        self.reset()

    def append(self, k_new, v_new, stream=None) -> None:
        T = k_new.shape[1]
        _lib._bf16(k_new, (self.B, T, self.Hkv, self.D), "k_new")
        _lib._bf16(v_new, (self.B, T, self.Hkv, self.D), "v_new")
        _lib.duo_kv_append_kv4(self.handle, self.cache, self.kv4, k_new, v_new, T, stream)

    def decode(self, q, out=None, stream=None):
        import torch
        _lib._bf16(q, (self.B, self.Hq, self.D), "q")
        if out is None:
            out = torch.empty_like(q)
        _lib._bf16(out, (self.B, self.Hq, self.D), "o")
        _lib.duo_attn_decode_kv4(self.handle, self.cache, self.kv4, q, out, self.workspace, stream)
        return out

    def prefill(self, q, k, v, out=None, kind_mask=3, stream=None):
        """A chunk of T new tokens against the 4-bit caches (dequantized in the kernel)."""
        import torch
        assert kind_mask == 3
        T = q.shape[1]
        _lib._bf16(q, (self.B, T, self.Hq, self.D), "q")
        _lib._bf16(k, (self.B, T, self.Hkv, self.D), "k")
        _lib._bf16(v, (self.B, T, self.Hkv, self.D), "v")
        if out is None:
            out = torch.empty_like(q)
        _lib._bf16(out, (self.B, T, self.Hq, self.D), "o")
        _lib.duo_attn_prefill_kv4(self.handle, self.cache, self.kv4, q, k, v, T, out, stream)
        return out


class DuoKv4PagedLayer(DuoKv4Layer):
    """4-bit caches whose retrieval rows live in a pool of blocks shared by every sequence
    and head: codes u8 [num_blocks, block_size, D/2] and (scale, zero) pairs int32
    [num_blocks, block_size], row t of retrieval head r of sequence b at row t %
    block_size of block block_table[b, r, t // block_size] (block_table: device int32
    [B, n_ret, max_blocks]; block_size a multiple of 128). Streaming heads keep their 4-bit
    sink + ring arrays."""

    def __init__(self, batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, block_size,
                 max_blocks, num_blocks, block_table, is_retrieval, device="cuda"):
        import torch
        super().__init__(batch, num_q_heads, num_kv_heads, head_dim, sink_size, recent_size, 16, is_retrieval,
                         device=device)
        u8 = dict(dtype=torch.uint8, device=self.device)
        i32 = dict(dtype=torch.int32, device=self.device)
        rows = num_blocks * block_size if self.n_ret else 0
        self.k_codes = torch.zeros((rows, head_dim // 2), **u8)
        self.v_codes = torch.zeros_like(self.k_codes)
        self.k_sz = torch.zeros((rows,), **i32)
        self.v_sz = torch.zeros_like(self.k_sz)
        if block_table is not None:
            assert block_table.dtype == torch.int32 and block_table.is_cuda and block_table.is_contiguous()
            assert tuple(block_table.shape) == (batch, self.n_ret, max_blocks)
        self.block_size = block_size
        self.block_table = block_table
        self.paged = _lib.duo_paged(block_table.data_ptr() if block_table is not None else None, block_size,
                                    max_blocks, num_blocks, None)
        ptr = lambda t: t.data_ptr() if t.numel() else None
        self.kv4 = _lib.duo_kv4_cache(ptr(self.k_codes), ptr(self.v_codes), ptr(self.k_sz), ptr(self.v_sz),
                                      ptr(self.ks_codes), ptr(self.vs_codes), ptr(self.ks_sz), ptr(self.vs_sz))

    def append(self, k_new, v_new, stream=None) -> None:
        T = k_new.shape[1]
        _lib._bf16(k_new, (self.B, T, self.Hkv, self.D), "k_new")
        _lib._bf16(v_new, (self.B, T, self.Hkv, self.D), "v_new")
        _lib.duo_kv_append_kv4_paged(self.handle, self.cache, self.paged, self.kv4, k_new, v_new, T, stream)

    def prefill(self, *args, **kwargs):
        raise NotImplementedError("prefill against 4-bit rows in a paged pool is not provided")

    def decode(self, q, out=None, stream=None):
        import torch
        _lib._bf16(q, (self.B, self.Hq, self.D), "q")
        if out is None:
            out = torch.empty_like(q)
        _lib._bf16(out, (self.B, self.Hq, self.D), "o")
        _lib.duo_attn_decode_kv4_paged(self.handle, self.cache, self.paged, self.kv4, q, out, self.workspace, stream)
        return out


def _check_mscale(mscale, shape):
    import torch
    if mscale is None:
        return
    if (mscale.dtype != torch.float32 or not mscale.is_cuda or not mscale.is_contiguous()
            or tuple(mscale.shape) != tuple(shape)):
        raise ValueError(f"mscale: need a contiguous CUDA float32 tensor of shape {tuple(shape)}")


def _check_lens(seq_lens, B):
    import torch
    if seq_lens.dtype != torch.int32 or not seq_lens.is_cuda or not seq_lens.is_contiguous() or seq_lens.numel() != B:
        raise ValueError(f"seq_lens: need a contiguous CUDA int32 tensor of {B} elements")
