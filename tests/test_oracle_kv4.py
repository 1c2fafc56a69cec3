"""Pins of the oracle's 4-bit KV row encoding (CPU only): hand-worked rows, the
nearest-grid-point property checked by brute force, a closed-form error bound, the
degenerate constant row and the nibble order."""

import numpy as np
import pytest

import oracle.kv4 as kv4


def _bf16_rows(rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    # round to bf16 (keep the top 16 bits, round to nearest even)
    u = x.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def test_worked_row_half_steps():
    # 0, 0.5, ..., 7.5: scale (7.5 - 0) / 15 = 0.5 exactly, zero 0, codes 0 ... 15
    x = np.arange(16, dtype=np.float32) * 0.5
    c, s, z = kv4.quantize_rows(x)
    assert float(s) == 0.5 and float(z) == 0.0
    assert c.tolist() == list(range(16))
    assert np.array_equal(kv4.dequantize(c, s, z), x.astype(np.float64))


def test_worked_row_ties_round_to_even():
    # scale 0.5: 0.25 / 0.5 = 0.5 -> 0, 0.75 / 0.5 = 1.5 -> 2, 1.25 / 0.5 = 2.5 -> 2
    x = np.array([0.0, 0.25, 0.75, 1.25, 7.5], np.float32)
    c, s, z = kv4.quantize_rows(x)
    assert float(s) == 0.5
    assert c.tolist() == [0, 0, 2, 2, 15]


def test_constant_row():
    x = np.full(8, 1.5, np.float32)
    c, s, z = kv4.quantize_rows(x)
    assert float(s) == 0.0 and float(z) == 1.5 and c.tolist() == [0] * 8
    assert np.array_equal(kv4.roundtrip(x), np.full(8, 1.5))


def test_nibble_order_and_packing():
    assert kv4.pack_codes(np.array([1, 2], np.uint8)).tolist() == [0x21]
    rng = np.random.default_rng(0)
    c = rng.integers(0, 16, (3, 64)).astype(np.uint8)
    assert np.array_equal(kv4.unpack_codes(kv4.pack_codes(c)), c)


def test_codes_are_the_nearest_grid_point_by_brute_force():
    rng = np.random.default_rng(1)
    x = _bf16_rows(rng, (50, 32))
    c, s, z = kv4.quantize_rows(x)
    grid = np.arange(16)[None, None, :] * s.astype(np.float64)[:, None, None] + z.astype(np.float64)[:, None, None]
    best = np.abs(x.astype(np.float64)[..., None] - grid).min(axis=-1)
    got = np.abs(x.astype(np.float64) - kv4.dequantize(c, s, z))
    assert (got <= best + 1e-6 * s.astype(np.float64)[:, None] + 1e-12).all()


def test_error_bound():
    rng = np.random.default_rng(2)
    x = _bf16_rows(rng, (200, 128))
    c, s, z = kv4.quantize_rows(x)
    mn, mx = x.min(-1).astype(np.float64), x.max(-1).astype(np.float64)
    s64, z64 = s.astype(np.float64), z.astype(np.float64)
    # fp16 rounding: zero within 2^-11 |mn| of the row min, 15 scale within 2^-10 of the range
    bound = 0.5 * s64 + 2 * (2.0 ** -11 * np.abs(mn) + 2.0 ** -24 + 2.0 ** -10 * (mx - mn)) \
        + 1e-6 * (np.abs(mx) + np.abs(mn))
    assert (np.abs(z64 - mn) <= 2.0 ** -11 * np.abs(mn) + 2.0 ** -24).all()
    err = np.abs(x.astype(np.float64) - kv4.dequantize(c, s, z)).max(-1)
    assert (err <= bound).all()
    # and the codes span the row: its min takes code 0, its max code 14 or 15
    assert (c.min(-1) == 0).all() and (c.max(-1) >= 14).all()


def test_planted_zero_from_the_max_fails(monkeypatch):
    real = kv4.quantize_rows

    def wrong(x):
        c, s, z = real(x)
        return c, s, np.asarray(x, np.float32).max(-1).astype(np.float16)

    monkeypatch.setattr(kv4, "quantize_rows", wrong)
    with pytest.raises(AssertionError):
        test_worked_row_half_steps()
    with pytest.raises(AssertionError):
        test_error_bound()
