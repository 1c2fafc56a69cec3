"""Seeded synthetic inputs shared by the CUDA path's tests and bench and by the CPU oracle.

This module holds no attention, mask or cache arithmetic. It defines one
counter-based generator, so that any element of any input stream can be
regenerated on its own (the CPU oracle regenerates only the tokens it needs,
for example the keys of one head of a million-token context), plus the
workload shapes (five mixed-head, two Dual Chunk Attention) and the seeded
retrieval/streaming head choice.

Generator definition (one value per element, no state carried between elements):

    key   = seed << 51 | stream << 47 | b << 39 | pos << 15 | head << 8 | d
    z     = splitmix64_mix(key + 0x9E3779B97F4A7C15)       (one SplitMix64 output
                                                            for state ``key``)
    u     = sum of the eight bytes of z                      (0 ... 2040)
    x32   = float32(u - 1020) * float32(sqrt(1.5) / 256)   (one IEEE multiply)
    value = bfloat16(x32), round to nearest even

``u`` is an Irwin-Hall sum of eight uniform bytes, so ``x32`` has mean 0 and
variance 1 (to 1e-5) and lies in [-4.9, 4.9]: a bounded stand-in for N(0, 1).
Only integer arithmetic and one correctly rounded float32 multiply are used, so
the numpy version (CPU, used by the oracle) and the CUDA version (used to fill
device buffers quickly) give identical bits; a GPU test checks this.

Streams: 0 = Q, 1 = K, 2 = V. ``pos`` is the absolute token position, so the
query and key/value of a decode step at position p are the same values a
prefill over p + 1 tokens would see.
"""

from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass, field

import numpy as np

STREAM_Q = 0
STREAM_K = 1
STREAM_V = 2
STREAM_Q_SUCC = 3   # Dual Chunk Attention: query vectors for the previous chunk
STREAM_Q_INTER = 4  # and for earlier chunks
STREAM_HEADS = 15  # the seeded head permutation

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BYTE_MASK = np.uint64(0x00FF00FF00FF00FF)
_LANE_SUM = np.uint64(0x0001000100010001)
SCALE_F32 = np.float32(math.sqrt(1.5) / 256.0)

MAX_POS = 1 << 24
MAX_HEAD = 1 << 7
MAX_D = 1 << 8
MAX_B = 1 << 8


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (Steele, Lea and Flood, OOPSLA 2014)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def element_keys(seed: int, stream: int, b, pos, head, d) -> np.ndarray:
    """Counter of every element; arguments broadcast like numpy arrays."""
    u = np.uint64
    return ((u(seed) << u(51)) | (u(stream) << u(47))
            | (np.asarray(b, dtype=np.uint64) << u(39))
            | (np.asarray(pos, dtype=np.uint64) << u(15))
            | (np.asarray(head, dtype=np.uint64) << u(8))
            | np.asarray(d, dtype=np.uint64))


def keys_to_f32(keys: np.ndarray) -> np.ndarray:
    """float32 value of each counter before rounding to bfloat16."""
    with np.errstate(over="ignore"):
        z = _mix64(keys + _GAMMA)
        t = (z & _BYTE_MASK) + ((z >> np.uint64(8)) & _BYTE_MASK)
        s = (t * _LANE_SUM) >> np.uint64(48)
    return (s.astype(np.int32) - 1020).astype(np.float32) * SCALE_F32


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16, nearest even; finite inputs only."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def stream_bits(seed: int, stream: int, B: int, pos0: int, T: int, H: int, D: int,
                heads=None, batches=None) -> np.ndarray:
    """bf16 bits of a token-major block [B, T, H, D] at positions pos0 ... pos0+T-1.

    ``heads`` / ``batches`` restrict the block to a subset (the result then has
    len(heads) / len(batches) in those axes)."""
    _check(B, pos0 + T, H, D)
    bs = np.arange(B) if batches is None else np.asarray(batches)
    hs = np.arange(H) if heads is None else np.asarray(heads)
    keys = element_keys(seed, stream,
                        bs[:, None, None, None],
                        (pos0 + np.arange(T))[None, :, None, None],
                        hs[None, None, :, None],
                        np.arange(D)[None, None, None, :])
    return f32_to_bf16_bits(keys_to_f32(keys))


def stream_f64(seed, stream, B, pos0, T, H, D, heads=None, batches=None) -> np.ndarray:
    """Exact float64 values of the bf16 inputs (the oracle's view)."""
    return bf16_bits_to_f64(stream_bits(seed, stream, B, pos0, T, H, D, heads, batches))


def head_stream_f64(seed, stream, b, head, pos0, T, D, chunk=1 << 16, workers=1) -> np.ndarray:
    """float64 [T, D] of one (batch, head), generated chunk by chunk (long contexts).

    ``workers`` > 1 generates chunks on that many threads (numpy releases the GIL)."""
    out = np.empty((T, D), dtype=np.float64)

    def one(c0):
        c1 = min(T, c0 + chunk)
        keys = element_keys(seed, stream, b, (pos0 + np.arange(c0, c1))[:, None], head,
                            np.arange(D)[None, :])
        out[c0:c1] = bf16_bits_to_f64(f32_to_bf16_bits(keys_to_f32(keys)))

    starts = list(range(0, T, chunk))
    if workers > 1 and len(starts) > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, starts))
    else:
        for c0 in starts:
            one(c0)
    return out


def _check(B, P, H, D):
    if not (0 < B <= MAX_B and 0 <= P <= MAX_POS and 0 < H <= MAX_HEAD and 0 < D <= MAX_D):
        raise ValueError(f"generator counter out of range: B={B} P={P} H={H} D={D}")


def stream_torch(seed, stream, B, pos0, T, H, D, device="cpu"):
    """A torch.bfloat16 tensor [B, T, H, D]. On a CUDA device the CUDA generator fills it."""
    import torch
    dev = torch.device(device)
    if dev.type == "cuda":
        out = torch.empty((B, T, H, D), dtype=torch.bfloat16, device=dev)
        fill_cuda(out, seed, stream, pos0)
        return out
    bits = stream_bits(seed, stream, B, pos0, T, H, D)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


# --------------------------------------------------------------------- CUDA generator
_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libduo_synth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        lib.synth_fill_bf16.restype = ctypes.c_int
        lib.synth_fill_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_float, ctypes.c_void_p]
        _LIB = lib
    return _LIB


def fill_cuda(out, seed: int, stream: int, pos0: int) -> None:
    """Fill a contiguous CUDA bf16 tensor [B, T, H, D] with the generator's values."""
    import torch
    assert out.is_cuda and out.dtype == torch.bfloat16 and out.is_contiguous() and out.dim() == 4
    B, T, H, D = out.shape
    _check(B, pos0 + T, H, D)
    st = torch.cuda.current_stream(out.device).cuda_stream
    rc = _lib().synth_fill_bf16(out.data_ptr(), seed, stream, B, pos0, T, H, D,
                                float(SCALE_F32), ctypes.c_void_p(st))
    if rc != 0:
        raise RuntimeError(f"synth_fill_bf16 failed: CUDA error {rc}")


# --------------------------------------------------------------------- workloads
def seeded_head_permutation(seed: int, H: int) -> list:
    """A permutation of range(H), ordered by the generator's hash of each head."""
    with np.errstate(over="ignore"):
        z = _mix64(element_keys(seed, STREAM_HEADS, 0, 0, np.arange(H), 0) + _GAMMA)
    return [int(h) for h in np.argsort(z, kind="stable")]


def retrieval_mask(seed: int, H_kv: int, n_retrieval: int, fixed=None) -> list:
    """Per-KV-head flags (1 = retrieval, 0 = streaming)."""
    chosen = list(fixed) if fixed is not None else seeded_head_permutation(seed, H_kv)[:n_retrieval]
    return [1 if h in chosen else 0 for h in range(H_kv)]


@dataclass(frozen=True)
class Workload:
    """One synthetic workload (shapes, head kinds, schedule)."""
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    S: int
    R: int
    n_retrieval: int
    prefill_len: int = 0          # tokens prefilled by attention (0 = none)
    chunk: int = 0                # chunk size of a chunked prefill (0 = one shot)
    context: int = 0              # tokens appended without attention before decoding
    decode_steps: int = 0
    fixed_retrieval: tuple = field(default=None)
    dca_chunk: int = 0            # Dual Chunk Attention chunk length (0 = not DCA)

    @property
    def is_retrieval(self) -> list:
        return retrieval_mask(self.seed, self.Hkv, self.n_retrieval, self.fixed_retrieval)

    @property
    def total_tokens(self) -> int:
        return self.prefill_len + self.context + self.decode_steps


WORKLOADS = {
    "tiny_prefill256_decode16": Workload("tiny_prefill256_decode16", 1, 1, 4, 4, 64, 4, 32, 2,
                                         prefill_len=256, decode_steps=16, fixed_retrieval=(0, 2)),
    "llama3_8b_prefill32k": Workload("llama3_8b_prefill32k", 2, 1, 32, 8, 128, 64, 256, 4,
                                     prefill_len=32768),
    "batched_decode_ctx128k": Workload("batched_decode_ctx128k", 3, 8, 32, 8, 128, 64, 256, 2,
                                       context=131072, decode_steps=256),
    "llama2_7b_chunked_prefill32k": Workload("llama2_7b_chunked_prefill32k", 4, 1, 32, 32, 128, 64, 256, 8,
                                             prefill_len=32768, chunk=4096),
    "decode_ctx1m": Workload("decode_ctx1m", 5, 1, 32, 8, 128, 64, 256, 2,
                             context=1 << 20, decode_steps=64),
    # Dual Chunk Attention (Qwen2-72B-shaped layer: 64 query / 8 KV heads, all full
    # attention), 131072-token prompt in chunks of 32768, then decode steps
    "qwen2_72b_dca_prefill128k": Workload("qwen2_72b_dca_prefill128k", 6, 1, 64, 8, 128, 0, 1, 8,
                                          prefill_len=131072, decode_steps=16, dca_chunk=32768),
    # the same layer at 32768 tokens in chunks of 8192 (a size ncu can capture in full)
    "qwen2_72b_dca_prefill32k": Workload("qwen2_72b_dca_prefill32k", 7, 1, 64, 8, 128, 0, 1, 8,
                                         prefill_len=32768, decode_steps=16, dca_chunk=8192),
}


def dca_mscale(B: int, T: int, chunk_len: int, pos0: int = 0) -> np.ndarray:
    """A smooth per-position fp32 scale for Dual Chunk Attention inputs (an input of
    the method, not part of it): 1 + 0.1 ln(1 + position / chunk_len), the same row
    for every sequence, float32 [B, T]."""
    pos = np.arange(pos0, pos0 + T, dtype=np.float64)
    row = (1.0 + 0.1 * np.log1p(pos / chunk_len)).astype(np.float32)
    return np.broadcast_to(row, (B, T)).copy()
