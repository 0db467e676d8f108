"""Pins of the fp64 oracle against what the pages and mathematics fix.

No expected value here comes from the oracle itself or from the CUDA path:
each is a number the pages print (``tests/golden``), a closed form evaluated
with ``math`` in independent code, an invariant, a library routine (torch fp64
softmax) or brute force over tiny inputs.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# cnblogs worked example (section 二): S11, S12 as printed, scale 1
# ----------------------------------------------------------------------------

def _worked(golden_dir):
    g = _golden(golden_dir, "worked_example_cnblogs.json")
    s11 = np.array(g["S11"])
    s12 = np.array(g["S12"])
    v = RNG.standard_normal((4, 3))
    return g, s11, s12, v


def _closed_form_row(scores, v):
    """softmax(scores) @ v and log-sum-exp, written out with math.exp."""
    m = max(scores)
    ex = [math.exp(s - m) for s in scores]
    l = sum(ex)
    o = [sum(ex[j] * v[j][c] for j in range(len(scores))) / l for c in range(len(v[0]))]
    return np.array(o), m + math.log(l), l


def test_worked_example_max_after_block1(golden_dir):
    g, s11, s12, v = _worked(golden_dir)
    trace = []
    oracle.online_merge_scores([s11, s12], [v[:2], v[2:]], trace=trace)
    assert trace[0]["m_new"].tolist() == g["m_after_block1"]
    assert np.maximum(trace[0]["m_new"], s12.max(axis=1)).tolist() == [30.0, 10.0]
    assert s12.max(axis=1).tolist() == g["block2_local_max"]


def test_worked_example_rescale_factor(golden_dir):
    g, s11, s12, v = _worked(golden_dir)
    trace = []
    oracle.online_merge_scores([s11, s12], [v[:2], v[2:]], trace=trace)
    r = g["row0_rescale_exponent"]
    # row 0: max 20 -> 30, old terms scaled by e^(20-30); row 1 keeps max 10 -> factor 1
    assert trace[1]["alpha"][0] == pytest.approx(math.exp(r["m_old"] - r["m_new"]), rel=1e-15)
    assert trace[1]["alpha"][1] == 1.0
    # first non-empty block: old contribution factor 0 (running max was -inf)
    assert trace[0]["alpha"].tolist() == [0.0, 0.0]


def test_worked_example_equals_global_softmax(golden_dir):
    g, s11, s12, v = _worked(golden_dir)
    o, lse = oracle.online_merge_scores([s11, s12], [v[:2], v[2:]])
    rows = np.concatenate([s11, s12], axis=1)
    for i in range(2):
        o_ref, lse_ref, _ = _closed_form_row(rows[i].tolist(), v.tolist())
        np.testing.assert_allclose(o[i], o_ref, rtol=1e-14, atol=1e-15)
        assert lse[i] == pytest.approx(lse_ref, rel=1e-15)
    # the printed row-0 scores give l = 1 + e^-10 + e^-20 + e^-25 relative to max 30
    _, lse0, l0 = _closed_form_row([10.0, 20.0, 30.0, 5.0], v.tolist())
    assert l0 == pytest.approx(1 + math.exp(-10) + math.exp(-20) + math.exp(-25), rel=1e-15)
    assert lse0 == pytest.approx(30 + math.log1p(math.exp(-10) + math.exp(-20) + math.exp(-25)), rel=1e-15)


def test_worked_example_through_plain_definition(golden_dir):
    """Q rows e0, e1 and K rows built so that Q K^T reproduces S11 | S12."""
    g, s11, s12, v = _worked(golden_dir)
    s = np.concatenate([s11, s12], axis=1)  # [2, 4]
    q = np.eye(2)
    k = s.T.copy()  # key j = (s_0j, s_1j)
    o, lse = oracle.attention_head(q, k, v, 1.0, causal=False)
    for i in range(2):
        o_ref, lse_ref, _ = _closed_form_row(s[i].tolist(), v.tolist())
        np.testing.assert_allclose(o[i], o_ref, rtol=1e-14, atol=1e-15)
        assert lse[i] == pytest.approx(lse_ref, rel=1e-15)


def test_worked_example_mutation_is_caught(golden_dir):
    """Planting the 'forgot to rescale U' bug (operatorworld page) breaks the pin."""
    g, s11, s12, v = _worked(golden_dir)
    o_bad, _ = oracle.online_merge_scores([s11, s12], [v[:2], v[2:]], rescale_u=False)
    o_ref, _, _ = _closed_form_row([10.0, 20.0, 30.0, 5.0], v.tolist())
    assert np.max(np.abs(o_bad[0] - o_ref)) > 1e-3
    # row 1 never changes its max (alpha = 1), so the bug is invisible there
    o_ref1, _, _ = _closed_form_row([10.0, 10.0, 5.0, 5.0], v.tolist())
    np.testing.assert_allclose(o_bad[1], o_ref1, rtol=1e-14)


# ----------------------------------------------------------------------------
# degenerate checks (operatorworld page; xuesongtap §2.2; triton-tutorial exercise 2)
# ----------------------------------------------------------------------------

def test_single_block_is_standard_softmax():
    s = RNG.standard_normal((5, 7)) * 3
    v = RNG.standard_normal((7, 4))
    o, lse = oracle.online_merge_scores([s], [v])
    for i in range(5):
        o_ref, lse_ref, _ = _closed_form_row(s[i].tolist(), v.tolist())
        np.testing.assert_allclose(o[i], o_ref, rtol=1e-13, atol=1e-15)
        assert lse[i] == pytest.approx(lse_ref, rel=1e-15)


def test_nonincreasing_block_maxima_give_alpha_one():
    # block maxima per row: 5, then 4, then 5 -> the running max never grows
    b1 = np.array([[5.0, 1.0, -2.0], [0.5, -1.0, 5.0]])
    b2 = np.array([[4.0, 3.0], [4.0, -7.0]])
    b3 = np.array([[5.0, 0.0, 2.0, 1.0], [2.0, 5.0, 3.0, 0.0]])
    v = RNG.standard_normal((9, 3))
    trace = []
    o, _ = oracle.online_merge_scores([b1, b2, b3], [v[:3], v[3:5], v[5:]], trace=trace)
    assert trace[1]["alpha"].tolist() == [1.0, 1.0]
    assert trace[2]["alpha"].tolist() == [1.0, 1.0]
    s = np.concatenate([b1, b2, b3], axis=1)
    for i in range(2):
        o_ref, _, _ = _closed_form_row(s[i].tolist(), v.tolist())
        np.testing.assert_allclose(o[i], o_ref, rtol=1e-13)


def test_alpha_values_printed_on_the_pages(golden_dir):
    for case in _golden(golden_dir, "alpha_cases.json")["cases"]:
        m_old, m_new = case["m_old"], case["m_new"]
        b1 = np.array([[m_old, m_old - 1.5]])
        b2 = np.array([[m_new - 0.25, m_new]])
        v = RNG.standard_normal((4, 2))
        trace = []
        oracle.online_merge_scores([b1, b2], [v[:2], v[2:]], trace=trace)
        assert trace[1]["alpha"][0] == pytest.approx(math.exp(case["alpha_exponent"]), rel=1e-15)
    # the two printed exponents, evaluated: e^-1 and e^-12
    assert math.exp(-1.0) == pytest.approx(0.36787944117144233, rel=1e-15)
    assert math.exp(-12.0) == pytest.approx(6.14421235332821e-06, rel=1e-14)


# ----------------------------------------------------------------------------
# closed forms and invariants of the plain definition
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_average_the_values(causal):
    n, d = 37, 8
    q = np.zeros((n, d))
    k = RNG.standard_normal((n, d))
    v = RNG.standard_normal((n, 5))
    o, lse = oracle.attention_head(q, k, v, 0.3, causal)
    for i in range(n):
        cnt = i + 1 if causal else n
        np.testing.assert_allclose(o[i], v[:cnt].mean(axis=0), rtol=1e-13, atol=1e-14)
        assert lse[i] == pytest.approx(math.log(cnt), rel=1e-14, abs=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_value_rows(causal):
    n, d = 23, 6
    q = RNG.standard_normal((n, d)) * 2
    k = RNG.standard_normal((n, d)) * 2
    vbar = RNG.standard_normal(4)
    v = np.tile(vbar, (n, 1))
    o, _ = oracle.attention_head(q, k, v, 0.7, causal)
    np.testing.assert_allclose(o, np.tile(vbar, (n, 1)), rtol=1e-13, atol=1e-14)


def test_causal_row_zero_sees_only_key_zero():
    n, d = 9, 4
    q = RNG.standard_normal((n, d))
    k = RNG.standard_normal((n, d))
    v = RNG.standard_normal((n, 3))
    o, lse = oracle.attention_head(q, k, v, 0.5, True)
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=0)
    assert lse[0] == pytest.approx(0.5 * float(sum(q[0, c] * k[0, c] for c in range(d))), rel=1e-14)


def test_permutation_invariance():
    n, d = 17, 8
    q = RNG.standard_normal((n, d))
    k = RNG.standard_normal((n, d))
    v = RNG.standard_normal((n, 8))
    o, lse = oracle.attention_head(q, k, v, 0.35, False)
    perm = RNG.permutation(n)
    o2, lse2 = oracle.attention_head(q, k[perm], v[perm], 0.35, False)
    np.testing.assert_allclose(o2, o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-14)
    o3, lse3 = oracle.attention_head(q[perm], k, v, 0.35, False)
    np.testing.assert_allclose(o3, o[perm], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse3, lse[perm], rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_block_split_invariance_all_compositions(causal):
    for n in range(1, 9):
        q = RNG.standard_normal((n, 3)) * 2
        k = RNG.standard_normal((n, 3)) * 2
        v = RNG.standard_normal((n, 2))
        o_ref, lse_ref = oracle.attention_head(q, k, v, 0.9, causal)
        count = 0
        for sizes in oracle.compositions(n):
            o, lse = oracle.online_attention_head(q, k, v, 0.9, causal, sizes)
            np.testing.assert_allclose(o, o_ref, rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(lse, lse_ref, rtol=1e-14, atol=1e-14)
            count += 1
        assert count == 2 ** (n - 1)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_fp64_naive_attention(causal):
    """triton-tutorial §8.1 naive_attention, evaluated by torch in fp64."""
    b, h, n, d = 2, 3, 19, 16
    q = torch.randn(b, h, n, d, dtype=torch.float64, generator=torch.Generator().manual_seed(5))
    k = torch.randn(b, h, n, d, dtype=torch.float64, generator=torch.Generator().manual_seed(6))
    v = torch.randn(b, h, n, d + 3, dtype=torch.float64, generator=torch.Generator().manual_seed(7))
    scale = 1.0 / math.sqrt(d)
    s = torch.matmul(q, k.transpose(-2, -1)) * scale
    if causal:
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    p = torch.softmax(s, dim=-1)
    o_ref = torch.matmul(p, v).numpy()
    lse_ref = torch.logsumexp(s, dim=-1).numpy()
    o, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), scale, causal)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-13, atol=1e-13)
    rows = np.array([0, 4, 18])
    o_r, lse_r = oracle.attention(q.numpy(), k.numpy(), v.numpy(), scale, causal, rows=rows)
    np.testing.assert_allclose(o_r, o_ref[:, :, rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse_r, lse_ref[:, :, rows], rtol=1e-13, atol=1e-13)


def test_two_keys_one_dim_closed_form():
    q = np.array([[1.3]])
    k = np.array([[0.7], [-2.1]])
    v = np.array([[3.0], [-5.0]])
    scale = 0.8
    s0, s1 = scale * 1.3 * 0.7, scale * 1.3 * -2.1
    sig = 1.0 / (1.0 + math.exp(-(s0 - s1)))
    o, lse = oracle.attention_head(q, k, v, scale, False)
    assert o[0, 0] == pytest.approx(sig * 3.0 + (1 - sig) * -5.0, rel=1e-14)
    assert lse[0] == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))), rel=1e-14)


def test_brute_force_pure_python():
    n, d, dv = 4, 3, 2
    q = RNG.standard_normal((n, d))
    k = RNG.standard_normal((n, d))
    v = RNG.standard_normal((n, dv))
    scale = 0.6
    for causal in (False, True):
        o, lse = oracle.attention_head(q, k, v, scale, causal)
        for i in range(n):
            keys = range(i + 1) if causal else range(n)
            w = {j: math.exp(scale * sum(q[i][c] * k[j][c] for c in range(d))) for j in keys}
            z = sum(w.values())
            for c in range(dv):
                assert o[i][c] == pytest.approx(sum(w[j] * v[j][c] for j in keys) / z, rel=1e-12, abs=1e-14)
            assert lse[i] == pytest.approx(math.log(z), rel=1e-13, abs=1e-14)


def test_empty_row_reading():
    """Reading for a row with no admissible key: O = 0, lse = -inf."""
    q = RNG.standard_normal((3, 2))
    k = np.zeros((0, 2))
    v = np.zeros((0, 2))
    o, lse = oracle.attention_head(q, k, v, 1.0, False)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


# ----------------------------------------------------------------------------
# combine laws (iceferryling §6 merge; cnblogs §三 FlashDecoding reduce)
# ----------------------------------------------------------------------------

def _partials(r, s, dv, with_empty=False):
    u = RNG.standard_normal((r, s, dv))
    m = RNG.standard_normal((r, s)) * 4
    l = RNG.uniform(0.5, 3.0, (r, s))
    if with_empty:
        m[:, 0] = -np.inf
        l[:, 0] = 0.0
        u[:, 0] = 0.0
    return u, m, l


def test_combine_single_partial_is_identity():
    u, m, l = _partials(6, 1, 5)
    o, lse = oracle.combine(u, m, l)
    np.testing.assert_allclose(o, u[:, 0] / l[:, :1], rtol=1e-15)
    np.testing.assert_allclose(lse, m[:, 0] + np.log(l[:, 0]), rtol=1e-15)


def test_combine_is_order_invariant_and_ignores_empty():
    u, m, l = _partials(4, 7, 3, with_empty=True)
    o, lse = oracle.combine(u, m, l)
    perm = RNG.permutation(7)
    o2, lse2 = oracle.combine(u[:, perm], m[:, perm], l[:, perm])
    np.testing.assert_allclose(o2, o, rtol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-14)
    o3, lse3 = oracle.combine(u[:, 1:], m[:, 1:], l[:, 1:])
    np.testing.assert_allclose(o3, o, rtol=1e-13)
    np.testing.assert_allclose(lse3, lse, rtol=1e-14)
    o4, lse4 = oracle.combine(np.zeros((1, 3, 2)), np.full((1, 3), -np.inf), np.zeros((1, 3)))
    assert np.all(o4 == 0) and np.isneginf(lse4[0])


def test_combine_two_partials_closed_form():
    u = np.array([[[2.0], [6.0]]])
    m = np.array([[1.0, 3.0]])
    l = np.array([[4.0, 5.0]])
    o, lse = oracle.combine(u, m, l)
    w0 = math.exp(1.0 - 3.0)
    assert o[0, 0] == pytest.approx((w0 * 2.0 + 6.0) / (w0 * 4.0 + 5.0), rel=1e-15)
    assert lse[0] == pytest.approx(3.0 + math.log(w0 * 4.0 + 5.0), rel=1e-15)


@pytest.mark.parametrize("chunk", [1, 3, 16, 128, 1000])
def test_chunked_decode_equals_one_shot(chunk):
    n_keys, d = 777, 16
    q = RNG.standard_normal(d)
    k = RNG.standard_normal((n_keys, d))
    v = RNG.standard_normal((n_keys, d))
    scale = 1.0 / math.sqrt(d)
    u, m, l = oracle.chunk_partials(q, k, v, scale, chunk)
    assert u.shape[0] == -(-n_keys // chunk)
    o, lse = oracle.combine(u[None], m[None], l[None])
    o_ref, lse_ref = oracle.attention_head(q[None], k, v, scale, False)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-14)


def test_decode_is_one_row_attention():
    b, h, n_keys, d = 2, 3, 50, 8
    q = RNG.standard_normal((b, h, d))
    k = RNG.standard_normal((b, h, n_keys, d))
    v = RNG.standard_normal((b, h, n_keys, d))
    o, lse = oracle.decode(q, k, v, 0.25, pairs=[(1, 2), (0, 0)])
    for idx, (bb, hh) in enumerate([(1, 2), (0, 0)]):
        s = 0.25 * (k[bb, hh] @ q[bb, hh])
        w = np.exp(s - s.max())
        np.testing.assert_allclose(o[idx], (w @ v[bb, hh]) / w.sum(), rtol=1e-13)
        assert lse[idx] == pytest.approx(s.max() + math.log(w.sum()), rel=1e-14)


# ------------------------------------------------------------------ key-shard partials (Ring Attention merge)

@pytest.mark.parametrize("causal", [False, True])
def test_shard_partials_merge_to_the_full_definition(causal):
    # cutting the keys into shards anywhere and merging the partials with ``combine`` gives the
    # unsharded result (cnblogs §三 场景 A; checked against torch's fp64 SDPA)
    rng = np.random.default_rng(31)
    n, d = 45, 6
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    cuts = [0, 7, 8, 30, 45]
    parts = [oracle.shard_partials_head(q, k[a:b], v[a:b], 0.4, causal, a) for a, b in zip(cuts, cuts[1:])]
    u = np.stack([p[0] for p in parts], axis=1)
    m = np.stack([p[1] for p in parts], axis=1)
    l = np.stack([p[2] for p in parts], axis=1)
    o, lse = oracle.combine(u, m, l)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q)[None], torch.from_numpy(k)[None],
                                                           torch.from_numpy(v)[None], is_causal=causal,
                                                           scale=0.4)[0].numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-13)
    ro, rl = oracle.attention_head(q, k, v, 0.4, causal)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-13)
    if causal:
        # rows before a shard's first key get the empty partial (0, -inf, 0)
        u2, m2, l2 = parts[3]  # keys 30..44
        assert np.all(np.isneginf(m2[:30])) and np.all(l2[:30] == 0) and np.all(u2[:30] == 0)
        assert np.all(np.isfinite(m2[30:]))


def test_shard_partial_of_one_key_is_closed_form():
    # a shard holding the single key j: m = scale q.k_j, l = 1, U = v_j
    rng = np.random.default_rng(32)
    q, k, v = (rng.standard_normal((4, 3)) for _ in range(3))
    u, m, l = oracle.shard_partials_head(q, k[2:3], v[2:3], 0.5, False, 2)
    np.testing.assert_allclose(m, 0.5 * q @ k[2], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(l, 1.0)
    np.testing.assert_array_equal(u, np.broadcast_to(v[2], (4, 3)))
