"""Pins of the oracle's paged-KV decode (decode_paged, paged_rows)."""

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(21)


def _pool_from_contiguous(k, page_size, perm):
    """Write contiguous caches [B, H, L, d] into a pool [P, H, page_size, d], logical page i of
    sequence b going to pool page perm[b * n + i]; returns (pool, block_table)."""
    B, H, L, d = k.shape
    n = -(-L // page_size)
    pool = np.full((B * n, H, page_size, d), np.nan)
    table = np.zeros((B, n), dtype=np.int64)
    for b in range(B):
        for i in range(n):
            pid = perm[b * n + i]
            rows = k[b, :, i * page_size:(i + 1) * page_size]
            pool[pid, :, :rows.shape[1]] = rows
            table[b, i] = pid
    return pool, table


@pytest.mark.parametrize("page_size", [4, 16])
def test_paged_decode_equals_contiguous_decode(page_size):
    # any placement of the pages gives the contiguous decode (a pinned special case: it is the
    # plain one-row definition); the unused tail of the last page holds NaN and must not matter
    B, H, L, d = 3, 2, 37, 8
    q = RNG.standard_normal((B, H, d))
    k = RNG.standard_normal((B, H, L, d))
    v = RNG.standard_normal((B, H, L, d))
    n = -(-L // page_size)
    perm = RNG.permutation(B * n)
    kp, table = _pool_from_contiguous(k, page_size, perm)
    vp, _ = _pool_from_contiguous(v, page_size, perm)
    lens = np.full(B, L)
    o, lse = oracle.decode_paged(q, kp, vp, table, lens, 0.3)
    ro, rl = oracle.decode(q, k, v, 0.3)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-14)
    # and equals torch's fp64 SDPA with one query row per (b, h)
    t = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q)[:, :, None], torch.from_numpy(k),
                                                         torch.from_numpy(v), scale=0.3)[:, :, 0].numpy()
    np.testing.assert_allclose(o.reshape(B, H, d), t, rtol=0, atol=1e-13)


def test_ragged_lengths_use_only_their_keys():
    # sequence b sees only its first seq_lens[b] keys: equal to decoding the truncated cache
    B, H, L, d, ps = 4, 2, 40, 8, 8
    q = RNG.standard_normal((B, H, d))
    k = RNG.standard_normal((B, H, L, d))
    v = RNG.standard_normal((B, H, L, d))
    perm = RNG.permutation(B * (L // ps))
    kp, table = _pool_from_contiguous(k, ps, perm)
    vp, _ = _pool_from_contiguous(v, ps, perm)
    lens = np.array([1, 9, 40, 17])
    o, lse = oracle.decode_paged(q, kp, vp, table, lens, 0.5)
    for idx, (b, h) in enumerate([(b, h) for b in range(B) for h in range(H)]):
        ro, rl = oracle.decode(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1, :lens[b]], v[b:b + 1, h:h + 1, :lens[b]], 0.5)
        np.testing.assert_allclose(o[idx], ro[0], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[idx], rl[0], rtol=0, atol=1e-14)
    # closed form for a single key: O = v_0, lse = scale * q.k_0
    b = 0
    for h in range(H):
        np.testing.assert_allclose(o[b * H + h], v[b, h, 0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[b * H + h], 0.5 * q[b, h] @ k[b, h, 0], rtol=0, atol=1e-14)


def test_empty_sequence_and_foreign_page_ids():
    B, H, d, ps = 2, 1, 4, 4
    q = np.ones((B, H, d))
    kp = RNG.standard_normal((3, H, ps, d))
    vp = RNG.standard_normal((3, H, ps, d))
    table = np.array([[1, 7], [-1, 0]])  # page 7 and page -1 are outside the pool of 3
    o, lse = oracle.decode_paged(q, kp, vp, table, np.array([0, 6]), 1.0)
    assert np.all(o[0] == 0) and lse[0] == -np.inf  # no keys: O = 0, lse = -inf
    # sequence 1: keys 0-3 come from the foreign id -1 (zero rows: score 0, value 0), keys 4-5
    # from page 0
    kz = np.concatenate([np.zeros((ps, d)), kp[0, 0, :2]])
    vz = np.concatenate([np.zeros((ps, d)), vp[0, 0, :2]])
    ro, rl = oracle.attention_head(q[1, 0][None], kz, vz, 1.0)
    np.testing.assert_allclose(o[1], ro[0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[1], rl[0], rtol=0, atol=1e-14)
    rows = oracle.paged_rows(kp, table, 0, 0, 6)
    np.testing.assert_array_equal(rows[:4], kp[1, 0])
    np.testing.assert_array_equal(rows[4:], 0.0)
