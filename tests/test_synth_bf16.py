"""The input generators' bf16 storage format (dflash2_synth.to_bf16_bits and
bf16_bits_to_f32), which both the CUDA path and the oracle read: round to
nearest, ties to even, against torch's float32 -> bfloat16 conversion, on
values that include exact ties, subnormals, signed zeros and the largest
finite magnitudes."""

import numpy as np
import torch

import dflash2_synth as S


def _torch_bits(x):
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_bits_match_torch_on_random_and_edge_values():
    g = np.random.default_rng(31)
    x = np.concatenate([
        g.standard_normal(50000).astype(np.float32) * np.float32(10.0) ** g.integers(-30, 30, 50000),
        # exact ties: the 16 dropped bits are 0x8000, with an even and an odd kept bit
        (np.arange(1, 2001, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        # subnormals, zeros, the largest finite float32 values that stay finite in bf16
        np.array([1e-40, -1e-40, 1e-45, 0.0, -0.0, 3.38e38, -3.38e38], dtype=np.float32),
    ]).astype(np.float32)
    np.testing.assert_array_equal(S.to_bf16_bits(x), _torch_bits(x))


def test_bf16_round_trip_is_exact_and_idempotent():
    g = np.random.default_rng(32)
    x = g.standard_normal(20000).astype(np.float32)
    y = S.bf16_bits_to_f32(S.to_bf16_bits(x))
    np.testing.assert_array_equal(S.to_bf16_bits(y), S.to_bf16_bits(x))   # bf16 values map to themselves
    np.testing.assert_array_equal(y, torch.from_numpy(x).to(torch.bfloat16).float().numpy())
    # at most half a unit in the last kept place away
    rel = np.abs(y.astype(np.float64) - x) / np.abs(x.astype(np.float64))
    assert np.max(rel[np.abs(x) > 1e-30]) <= 2.0 ** -8
