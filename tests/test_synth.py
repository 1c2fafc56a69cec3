"""The seeded input generator (CPU side): counter-based, exact rounding, N(0,1)-like."""

import numpy as np
import torch

import duo_synth as ds


def test_splitmix64_reference_outputs():
    # First outputs of SplitMix64 seeded with state 0 (Vigna's splitmix64.c):
    # state k * gamma, output mix(state).
    z = ds._mix64(np.array([1, 2, 3], dtype=np.uint64) * ds._GAMMA)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_block_equals_concatenated_chunks():
    a = ds.stream_bits(3, ds.STREAM_K, 2, 100, 50, 4, 16)
    b = np.concatenate([ds.stream_bits(3, ds.STREAM_K, 2, 100 + s, 10, 4, 16) for s in range(0, 50, 10)], axis=1)
    np.testing.assert_array_equal(a, b)
    c = ds.stream_bits(3, ds.STREAM_K, 2, 100, 50, 4, 16, heads=[1, 3], batches=[1])
    np.testing.assert_array_equal(a[[1]][:, :, [1, 3]], c)
    h = ds.head_stream_f64(3, ds.STREAM_K, 1, 3, 100, 50, 16, chunk=7)
    np.testing.assert_array_equal(ds.bf16_bits_to_f64(a[1, :, 3]), h)


def test_streams_and_seeds_differ():
    a = ds.stream_bits(1, ds.STREAM_Q, 1, 0, 64, 2, 32)
    b = ds.stream_bits(1, ds.STREAM_K, 1, 0, 64, 2, 32)
    c = ds.stream_bits(2, ds.STREAM_Q, 1, 0, 64, 2, 32)
    assert (a != b).mean() > 0.9 and (a != c).mean() > 0.9


def test_rounding_matches_torch_bf16():
    x = ds.keys_to_f32(np.arange(200000, dtype=np.uint64))
    rng = np.random.default_rng(0)
    y = (rng.standard_normal(200000) * 10).astype(np.float32)
    for v in (x, y):
        mine = ds.f32_to_bf16_bits(v)
        ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(mine, ref)


def test_distribution_is_standardised():
    v = ds.keys_to_f32(ds.element_keys(7, 1, 0, np.arange(4096)[:, None], 0, np.arange(256)[None, :]))
    assert abs(float(v.mean())) < 0.01
    assert abs(float(v.var()) - 1.0) < 0.01
    assert float(np.abs(v).max()) <= 1020 * float(ds.SCALE_F32) + 1e-6


def test_workloads_and_head_masks():
    w = ds.WORKLOADS
    assert w["tiny_prefill256_decode16"].is_retrieval == [1, 0, 1, 0]
    for name, n in [("llama3_8b_prefill32k", 4), ("batched_decode_ctx128k", 2),
                    ("llama2_7b_chunked_prefill32k", 8), ("decode_ctx1m", 2)]:
        m = w[name].is_retrieval
        assert sum(m) == n and len(m) == w[name].Hkv
    p = ds.seeded_head_permutation(2, 8)
    assert sorted(p) == list(range(8))
