"""Helpers of the GPU parity tests: inputs from the seeded generator, oracle views, tolerances."""

from __future__ import annotations

import numpy as np

import duo_synth as ds

# bf16 outputs against the float64 oracle: max |err| and mean |err| / mean |ref|
ATOL = 2e-2
MEAN_REL = 1e-2


def assert_close(got, ref, what="", atol=ATOL, mean_rel=MEAN_REL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    rel = err.mean() / max(np.abs(ref).mean(), 1e-30)
    assert err.max() <= atol and rel <= mean_rel, f"{what}: max|err| {err.max():.3e} mean rel {rel:.3e}"
    return float(err.max()), float(rel)


def to_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def device_stream(seed, stream, B, pos0, T, H, D, dev):
    """bf16 [B, T, H, D] on the device; large blocks come from the CUDA generator."""
    import torch
    if B * T * H * D >= (1 << 22):
        return ds.stream_torch(seed, stream, B, pos0, T, H, D, device=dev)
    return ds.stream_torch(seed, stream, B, pos0, T, H, D).to(dev)


def host_stream(seed, stream, B, pos0, T, H, D, heads=None, batches=None):
    return ds.stream_f64(seed, stream, B, pos0, T, H, D, heads=heads, batches=batches)


def head_keys(seed, b, h, pos0, T, D):
    """float64 K and V [T, D] of one (sequence, KV head)."""
    return (ds.head_stream_f64(seed, ds.STREAM_K, b, h, pos0, T, D, workers=8),
            ds.head_stream_f64(seed, ds.STREAM_V, b, h, pos0, T, D, workers=8))
