"""4-bit KV cache rows, the encoding restated plainly. TEST INFRASTRUCTURE ONLY.

Source: the DuoAttention README (quick-start demo and Efficiency section) combines
DuoAttention with 8-bit weights and a 4-bit KV cache to decode 3.3M tokens on one
GPU, but gives no format. The reading used here (the plainest asymmetric 4-bit
encoding of one cached row):

* a row is the D values of one token of one head, as stored in bf16;
* mn, mx = min and max of the row (fp32, exact for bf16 inputs);
* scale = fp16(round-to-nearest((mx - mn) / 15) in fp32); zero = fp16(mn);
* code_d = clamp(rint((x_d - zero) / scale), 0, 15), every operation in fp32 with
  round-to-nearest-even (the subtraction, the division, the rounding to an
  integer), with fp16 scale and zero widened exactly to fp32; a zero scale gives
  all codes 0;
* the row is stored as D / 2 bytes (element 2i in the low nibble of byte i, 2i + 1
  in the high nibble) plus the fp16 pair (scale, zero);
* its value is code * scale + zero.

Floating point decides the integer codes here, so the oracle takes those decisions
in fp32 exactly as the kernel does (numpy float32 arithmetic is IEEE round-to-
nearest like the GPU's); everything after decoding is float64.
"""

from __future__ import annotations

import numpy as np


def quantize_rows(x) -> tuple:
    """x: [..., D] values exactly representable in bf16. Returns (codes uint8 [..., D],
    scale float16 [...], zero float16 [...])."""
    x = np.asarray(x, np.float32)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    scale = ((mx - mn) / np.float32(15.0)).astype(np.float32).astype(np.float16)
    zero = mn.astype(np.float16)
    s32 = scale.astype(np.float32)[..., None]
    z32 = zero.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        c = np.rint((x - z32) / np.where(s32 == 0, np.float32(1), s32)).astype(np.float32)
    c = np.clip(c, 0, 15)
    c = np.where(s32 == 0, 0, c)
    return c.astype(np.uint8), scale, zero


def pack_codes(codes) -> np.ndarray:
    """uint8 codes [..., D] -> bytes [..., D / 2] (even element in the low nibble)."""
    codes = np.asarray(codes, np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    packed = np.asarray(packed, np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = packed & 15
    out[..., 1::2] = packed >> 4
    return out


def dequantize(codes, scale, zero) -> np.ndarray:
    """float64 values code * scale + zero."""
    return (np.asarray(codes, np.float64) * np.asarray(scale, np.float64)[..., None]
            + np.asarray(zero, np.float64)[..., None])


def roundtrip(x) -> np.ndarray:
    """What a 4-bit cache holds for rows x, as float64."""
    return dequantize(*quantize_rows(x))
