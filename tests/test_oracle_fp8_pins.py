"""Pins of the oracle's E4M3 block quantization (a byte-exact reference for the GPU quantizer)."""

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(7)


def test_e4m3_table_matches_the_format():
    vals = oracle.e4m3_values()
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF]) and vals[0x80] == 0.0
    # torch's float8_e4m3fn decodes the same 256 codes
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(np.nan_to_num(t, nan=1234.5), np.nan_to_num(vals, nan=1234.5))


def test_rounding_is_nearest_even_and_matches_torch():
    x = np.concatenate([RNG.standard_normal(20000) * 50, RNG.standard_normal(2000) * 0.01,
                        np.array([0.0, -0.0, 448.0, -448.0, 447.9, 2.0 ** -10, 3 * 2.0 ** -10])]).astype(np.float32)
    codes = oracle.round_to_e4m3(x)
    vals = oracle.e4m3_values()[codes.astype(np.int64)]
    # brute force: no code is strictly closer
    table = oracle.e4m3_values()[:0x7F]
    best = np.abs(np.abs(x.astype(np.float64))[:, None] - table[None, :]).min(axis=1)
    np.testing.assert_array_equal(np.abs(np.abs(vals) - np.abs(x)), best)
    # torch's conversion (round to nearest even) agrees on every in-range value
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, t)


def test_saturation_and_ties():
    assert oracle.round_to_e4m3(np.float32(1e6)) == 0x7E
    assert oracle.round_to_e4m3(np.float32(-1e6)) == 0xFE
    # 1 + 1/16 lies halfway between 1 (code 0x38, even) and 1.125 (0x39): ties go to the even code
    assert oracle.round_to_e4m3(np.float32(1.0625)) == 0x38
    assert oracle.round_to_e4m3(np.float32(1.1875)) == 0x3A


def test_block_quantization_round_trip_and_amax():
    x = RNG.standard_normal((2, 3, 300, 16)).astype(np.float32)
    x[1, 2, 128:256] = 0.0
    codes, scales = oracle.quantize_e4m3_blocks(x)
    assert scales.shape == (2, 3, 3) and scales[1, 2, 1] == 1.0
    back = oracle.dequantize_blocks(codes, scales)
    # each element within half an E4M3 spacing (relative 2^-4) of the original, or exact zero
    rel = np.abs(back - x) / np.maximum(np.abs(x), 1e-30)
    big = np.abs(x) / np.repeat(scales, 128, axis=2)[:, :, :300, None] >= 2.0 ** -6
    assert np.all(rel[big] <= 2.0 ** -4 + 1e-7)
    # the block's amax element maps to exactly +-448
    blk = x[0, 0, :128]
    i = np.unravel_index(np.abs(blk).argmax(), blk.shape)
    assert abs(oracle.e4m3_values()[codes[0, 0, :128][i]]) == 448.0
