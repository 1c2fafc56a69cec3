"""The CUDA half of the input generator gives the same bits as the numpy half."""

import numpy as np
import pytest
import torch

import duo_synth as ds

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,pos0", [((1, 300, 4, 64), 0), ((3, 77, 8, 128), 131000), ((2, 5, 32, 128), 1 << 20)])
def test_cuda_generator_equals_numpy(shape, pos0):
    B, T, H, D = shape
    for stream in (ds.STREAM_Q, ds.STREAM_K, ds.STREAM_V):
        g = ds.stream_torch(5, stream, B, pos0, T, H, D, device="cuda")
        c = ds.stream_bits(5, stream, B, pos0, T, H, D)
        np.testing.assert_array_equal(g.view(torch.int16).cpu().numpy().view(np.uint16), c)
