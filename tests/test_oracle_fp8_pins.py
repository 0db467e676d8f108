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


# ---------------------------------------------------------------- the FP8 forward (attention_fp8)

def _codes(shape, rng, lo=0x20, hi=0x4F):
    """Random E4M3 codes of either sign with magnitudes between 2^-3 and 3.75."""
    mag = rng.integers(lo, hi, size=shape)
    return (mag | (rng.integers(0, 2, size=shape) << 7)).astype(np.uint8)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_without_p_quantization_is_sdpa_on_dequantized_inputs(causal):
    # quantize_p=False reduces the FP8 forward to the plain definition on value(code) * scale;
    # torch's CPU scaled_dot_product_attention in fp64 is the library routine it must match.
    rng = np.random.default_rng(11)
    n, d = 300, 16
    q8, k8, v8 = (_codes((1, 2, n, d), rng) for _ in range(3))
    sq, sk, sv = (rng.uniform(0.01, 0.2, size=(1, 2, 3)).astype(np.float32) for _ in range(3))
    scale = 0.3
    o, lse = oracle.attention_fp8(q8, sq, k8, sk, v8, sv, scale, causal, quantize_p=False)
    qd, kd, vd = (torch.from_numpy(oracle.dequantize_blocks(c, s)) for c, s in ((q8, sq), (k8, sk), (v8, sv)))
    ref = torch.nn.functional.scaled_dot_product_attention(qd, kd, vd, is_causal=causal, scale=scale).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    s = scale * (qd @ kd.transpose(-1, -2))
    if causal:
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_uniform_scores_give_the_mean_of_v(causal):
    # Every key has the same score, so p = 1 for every admissible key and P~ = 256 s_v[j] / max(s_v):
    # 256 or 128 here, both exact in E4M3.  O is then the mean of the dequantized V rows exactly.
    rng = np.random.default_rng(12)
    n, d = 384, 8
    q8 = _codes((1, 1, n, d), rng)
    k8 = np.broadcast_to(_codes((1, 1, 1, d), rng), (1, 1, n, d)).copy()
    v8 = _codes((1, 1, n, d), rng)
    sq = np.full((1, 1, 3), 0.05, np.float32)
    sk = np.full((1, 1, 3), 0.07, np.float32)
    sv = np.array([[[0.25, 0.125, 0.25]]], np.float32)  # ratios 1, 1/2, 1
    o, lse = oracle.attention_fp8(q8, sq, k8, sk, v8, sv, 1.0, causal)
    vd = oracle.dequantize_blocks(v8, sv)[0, 0]
    s = (oracle.dequantize_blocks(q8, sq)[0, 0] @ oracle.dequantize_blocks(k8[:, :, :1], sk[:, :, :1])[0, 0].T)[:, 0]
    for i in range(n):
        m = i + 1 if causal else n
        np.testing.assert_allclose(o[0, 0, i], vd[:m].mean(axis=0), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0, i], s[i] + np.log(m), rtol=0, atol=1e-12)


def test_fp8_two_keys_half_weight_closed_form():
    # Two keys whose scores differ by ln 2: p = (1, 1/2), P~ = (256, 128) exactly, so
    # O = (v0 + v1 / 2) / 1.5 and lse = s0 + ln 1.5.
    vals = oracle.e4m3_values()
    q8 = np.array([[[[0x38, 0x00]]]], np.uint8)           # q = (1, 0)
    k8 = np.array([[[[0x40, 0x00], [0x38, 0x00]]]], np.uint8)  # k0 = (2, 0), k1 = (1, 0): q.k = 2, 1
    v8 = np.array([[[[0x44, 0xB8], [0x30, 0x48]]]], np.uint8)
    sq = sk = sv = np.ones((1, 1, 1), np.float32)
    scale = float(np.log(2.0))
    o, lse = oracle.attention_fp8(q8, sq, k8, sk, v8, sv, scale)
    v0, v1 = vals[v8[0, 0, 0].astype(int)], vals[v8[0, 0, 1].astype(int)]
    np.testing.assert_allclose(o[0, 0, 0], (v0 + v1 / 2) / 1.5, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0, 0], 2 * scale + np.log(1.5), rtol=0, atol=1e-15)


def test_fp8_p_quantization_error_within_its_bound():
    # P~ s_p differs from p by at most half an E4M3 spacing: 2^-4 p for normal codes, 2^-10 s_p
    # below 2^-6 (subnormal spacing 2^-9).  So per row |O - O_exact| <= sum_k max(2^-4 p_k,
    # 2^-10 s_p) |v_k| / l with p relative to the running max (<= 1): bounded by
    # 2^-4 max|v| + n 2^-10 max(s_p) max|v| / l, l >= 1.
    rng = np.random.default_rng(13)
    n, d = 520, 32
    q8, k8, v8 = (_codes((1, 1, n, d), rng) for _ in range(3))
    sq, sk = (rng.uniform(0.05, 0.1, size=(1, 1, 5)).astype(np.float32) for _ in range(2))
    sv = rng.uniform(0.1, 0.3, size=(1, 1, 5)).astype(np.float32)
    for causal in (False, True):
        o_q, _ = oracle.attention_fp8(q8, sq, k8, sk, v8, sv, 0.5, causal)
        o_x, lse = oracle.attention_fp8(q8, sq, k8, sk, v8, sv, 0.5, causal, quantize_p=False)
        vmax = np.abs(oracle.dequantize_blocks(v8, sv)).max()
        sp_max = sv.max() / (256.0 * sv.min())
        bound = 2.0 ** -4 * vmax + n * 2.0 ** -10 * sp_max * vmax  # l >= 1 (the max key has p = 1)
        err = np.abs(o_q - o_x).max()
        assert 0 < err <= bound + 1e-9
        # and the error is real: the quantized result is not the exact one
        assert err > 1e-6
