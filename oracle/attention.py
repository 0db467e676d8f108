"""Plain fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, header, table or helper with the CUDA library; it receives the exact
bf16 input values (widened to fp64) and produces the values the GPU results are
compared against.

What it computes, and where the pages define it
-----------------------------------------------
* ``attention`` -- the plain definition S = scale * Q K^T, P = softmax(S),
  O = P V, one explicit score row per query (xuesongtap.github.io
  "flash-attention" page, §1 equation for S, P, O; triton-tutorial
  "8. FlashAttention 实战", §8.1 ``naive_attention``).  The log-sum-exp saved
  per row is m + log(l) in natural log of the *scaled* scores (xuesongtap §3,
  "前向额外保存逐行的 log-sum-exp"; triton-tutorial §8.8.2).  Causal keeps key
  j <= i (triton-tutorial §8.7.1, diagonal-block mask ``offs_m >= offs_n``),
  masked scores are -inf (xuesongtap §2.2, last paragraph).
* ``online_merge_scores`` / ``online_attention`` -- the blockwise algorithm in
  the pages' order: per key block, block row max, new running max m_new,
  alpha = exp(m_old - m_new), p = exp(s - m_new), l = alpha*l + rowsum(p),
  U = alpha*U + p V, and O = U / l only after the scan (xuesongtap §2.2,
  equation for U_i^new; operatorworld "在线 softmax：边算边修正" update
  equations; triton-tutorial §8.3.3).  Used to pin the worked example and the
  block-split invariance; the GPU path is compared against ``attention``.
* ``shard_partials_head`` -- one key shard's partial (U, m, l) per query row
  (Ring Attention's local step, cnblogs §三 场景 A), the plain definition
  restricted to the shard's admissible keys.
* ``combine`` -- merging partial (U, m, l) triples: m = max_w m_w,
  l = sum_w exp(m_w - m) l_w, O = sum_w exp(m_w - m) U_w / l (iceferryling
  "FlashAttention 1 和 FlashAttention 2 的区别", §6 cross-warp merge; the same
  rule reduces FlashDecoding partials, cnblogs jzssuanfa page, §三 场景 B).
* ``attention_backward_head`` / ``attention_backward`` -- gradients of the
  plain definition given dO: dV = P^T dO, dP = dO V^T, D_i = rowsum(dP_i * P_i)
  (= rowsum(O_i * dO_i)), dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q
  (triton-tutorial "8. FlashAttention 实战", §8.8.1 gradient formulas and
  §8.8.3 D_i and dS; operatorworld "反向传播：用重算换显存").  P is formed
  explicitly here; the blockwise recomputation from lse is the GPU's business.
* ``attention_backward_rows`` -- the same gradients at selected query rows (dQ)
  and key rows (dK, dV) of one head, forming only those rows and columns of
  P, dP and dS (plus every row's softmax normaliser and D_i), for heads too
  long for the full N x N matrices.
* ``e4m3_values`` / ``quantize_e4m3_blocks`` / ``dequantize_blocks`` -- FP8
  block quantization (triton-tutorial "8. FlashAttention 实战", §8.9.4: one
  scale per 128-row block, scale = max|x| / 448, E4M3 max 448): the scale and
  x / scale are fp32 operations, taken in the kernel's precision because they
  decide integer codes; the code is the nearest E4M3 value, ties to the even
  code, saturating at +-448.
* ``attention_fp8_head`` / ``attention_fp8`` -- the FP8 forward's mixed
  precision (triton-tutorial §8.9.3 and §8.9.6): S = (Q8 K8^T) * s_q * s_k *
  scale, the online softmax of ``online_merge_scores`` in fp64 with l summing
  the unquantized p, p quantized to E4M3 with a per-block scale before the
  second GEMM, and U += (P~ V8) * s_p * s_v.  With ``quantize_p=False`` it is
  ``attention`` on the dequantized values.
* ``paged_rows`` / ``decode_paged`` -- decode over a paged KV cache: key j of
  sequence b is row j % page_size of pool page block_table[b][j // page_size]
  (iceferryling §13 names the paged block table; the layout [P, H, page_size,
  d] and "an id outside the pool reads as zeros" are this library's reading),
  then the decode definition over seq_lens[b] keys.
* ``chunk_partials`` / ``decode`` -- FlashDecoding split-K: one query row, the
  KV sequence cut into chunks, one partial (U, m, l) per chunk by the plain
  definition restricted to the chunk (cnblogs §三 场景 B, step 2).

Readings where the pages are silent or disagree (each also listed in the
design notes):
* A query row with no admissible key has O = 0 and lse = -inf.
* FP8: the block scale of P~ for key tile j (the pages leave it open) is
  s_p = max(s_v) / (256 s_v[j]), so that P~ = E4M3(fp32(p) * 256 s_v[j] / max(s_v))
  never exceeds 256 (p <= 1) and s_p * s_v[j] = max(s_v) / 256 is the same for
  every tile.  The code is decided in fp32, as the pages compute p.
* When the running max is still -inf, 0 is used as the subtraction base so
  that alpha and p are 0 instead of NaN (xuesongtap §2.2: "首个非空块的旧贡献
  系数取 0"; rows that are fully masked skip the invalid exponent difference).
* U is kept unnormalised and divided by l once at the end (xuesongtap §2.2 and
  §4; triton-tutorial §8.4.5).  The cnblogs page's block-local normalisation
  gives the same result.

Every function here is pinned by ``tests/test_oracle_pins.py``,
``tests/test_oracle_backward_pins.py``, ``tests/test_oracle_fp8_pins.py`` and
``tests/test_oracle_paged_pins.py`` against values the pages print, closed
forms, invariants, library routines (torch's float8 conversion and fp64 SDPA)
and brute force.
"""

from __future__ import annotations

import itertools
from typing import Iterable, Sequence

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Widen any array-like (numpy, torch CPU tensor of bf16/fp32) to fp64."""
    if hasattr(x, "detach"):  # a torch tensor; bf16 has no numpy dtype
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def admissible_keys(i: int, n_keys: int, causal: bool) -> np.ndarray:
    """J(i): the keys query row i may attend to.

    Non-causal: all keys 0..n_keys-1.  Causal (top-left aligned, square):
    keys 0..i (triton-tutorial §8.7.1: a score survives when row >= column).
    """
    hi = min(i + 1, n_keys) if causal else n_keys
    return np.arange(max(hi, 0))


def attention_head(q, k, v, scale: float, causal: bool = False, rows=None):
    """Plain-definition attention for one (batch, head).

    q: [N, d], k: [Nk, d], v: [Nk, dv]; returns (O [R, dv], lse [R]) for the
    query rows ``rows`` (default: all N).  One explicit score row per query,
    the stable softmax of triton-tutorial §8.3.1 (max, exp, sum, divide)
    applied to S = scale * q k^T (xuesongtap §1; triton-tutorial §8.1).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n = q.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.shape[0], v.shape[1]), dtype=np.float64)
    lse = np.full(rows.shape[0], NEG_INF, dtype=np.float64)
    if rows.shape[0] == 0:
        return out, lse
    # the explicit N x N score matrix, one row per selected query
    s_all = float(scale) * (q[rows] @ k.T)
    for r, i in enumerate(rows):
        keys = admissible_keys(int(i), k.shape[0], causal)
        if keys.shape[0] == 0:
            continue  # reading: no admissible key -> O = 0, lse = -inf
        s = s_all[r, keys]
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        out[r] = (e @ v[keys]) / l
        lse[r] = m + np.log(l)
    return out, lse


def attention(q, k, v, scale: float, causal: bool = False, rows=None):
    """Attention over [B, H, N, d] tensors, head by head.

    ``rows`` selects query rows per head: None (all rows), a 1-D index array
    (same rows for every head) or a [B, H, R] integer array (rows per head).
    Returns O [B, H, R, dv] and lse [B, H, R] in fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    b_, h_, n = q.shape[0], q.shape[1], q.shape[2]
    if rows is None:
        rows_bh = None
        r = n
    else:
        rows = np.asarray(rows, dtype=np.int64)
        rows_bh = rows
        r = rows.shape[-1]
    out = np.zeros((b_, h_, r, v.shape[-1]))
    lse = np.zeros((b_, h_, r))
    for b in range(b_):
        for h in range(h_):
            sel = None
            if rows_bh is not None:
                sel = rows_bh if rows_bh.ndim == 1 else rows_bh[b, h]
            out[b, h], lse[b, h] = attention_head(q[b, h], k[b, h], v[b, h], scale, causal, sel)
    return out, lse


def online_merge_scores(score_blocks: Sequence, value_blocks: Sequence, *, rescale_u: bool = True,
                        trace: list | None = None):
    """Blockwise online softmax over given score blocks, in the pages' order.

    score_blocks[j]: [R, Bc_j] already-scaled scores (-inf where masked);
    value_blocks[j]: [Bc_j, dv].  State per row starts at m = -inf, l = 0,
    U = 0 (xuesongtap §2.2 "初始状态").  For each block (triton-tutorial
    §8.3.3):
        m_new = max(m_old, rowmax(S_block))
        alpha = exp(m_old - m_new)
        p     = exp(S_block - m_new)
        l     = alpha * l + rowsum(p)
        U     = alpha * U + p @ V_block
    and after the scan O = U / l, lse = m + log(l).

    ``rescale_u=False`` plants the bug the operatorworld page warns about
    (forgetting to rescale the old output); tests use it to show that the
    pins catch it.  When ``trace`` is a list, one dict per block with the
    block's m_new, alpha and l is appended to it.
    """
    first = _f64(score_blocks[0])
    r = first.shape[0]
    dv = _f64(value_blocks[0]).shape[1]
    m = np.full(r, NEG_INF)
    l = np.zeros(r)
    u = np.zeros((r, dv))
    for s_blk, v_blk in zip(score_blocks, value_blocks):
        s_blk = _f64(s_blk)
        v_blk = _f64(v_blk)
        if s_blk.shape[1] == 0:
            continue
        m_new = np.maximum(m, s_blk.max(axis=1))
        base = np.where(np.isneginf(m_new), 0.0, m_new)  # fully-masked guard
        alpha = np.exp(m - base)
        p = np.exp(s_blk - base[:, None])
        l = alpha * l + p.sum(axis=1)
        u = (alpha[:, None] * u if rescale_u else u) + p @ v_blk
        m = m_new
        if trace is not None:
            trace.append({"m_new": m_new.copy(), "alpha": alpha.copy(), "l": l.copy()})
    safe_l = np.where(l > 0, l, 1.0)
    o = np.where(l[:, None] > 0, u / safe_l[:, None], 0.0)
    lse = np.where(l > 0, m + np.log(safe_l), NEG_INF)
    return o, lse


def online_attention_head(q, k, v, scale: float, causal: bool, block_sizes: Iterable[int], *,
                          rescale_u: bool = True, trace: list | None = None):
    """One head through the blockwise algorithm with key blocks of the given sizes.

    Q_i stays whole (one query block), the key/value blocks K_j, V_j arrive
    in order (xuesongtap §2.1; cnblogs §一 inner loop).  Scores of masked
    pairs are -inf (xuesongtap §2.2, last paragraph).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n = q.shape[0]
    sizes = list(block_sizes)
    assert sum(sizes) == k.shape[0], "block sizes must cover the keys"
    s_blocks, v_blocks = [], []
    start = 0
    for bc in sizes:
        s = float(scale) * (q @ k[start:start + bc].T)
        if causal:
            cols = np.arange(start, start + bc)
            s = np.where(cols[None, :] > np.arange(n)[:, None], NEG_INF, s)
        s_blocks.append(s)
        v_blocks.append(v[start:start + bc])
        start += bc
    return online_merge_scores(s_blocks, v_blocks, rescale_u=rescale_u, trace=trace)


def compositions(n: int):
    """All ordered ways to cut n keys into consecutive non-empty blocks (2^(n-1))."""
    for cuts in itertools.product([0, 1], repeat=max(n - 1, 0)):
        sizes, run = [], 1
        for c in cuts:
            if c:
                sizes.append(run)
                run = 1
            else:
                run += 1
        sizes.append(run)
        yield sizes


def shard_partials_head(q, k_shard, v_shard, scale: float, causal: bool, key_offset: int, rows=None):
    """One query block against one key shard (Ring Attention's local step, cnblogs §三 场景 A):
    per row the plain definition restricted to the shard's admissible keys (global index
    key_offset + j, causal keeps those <= the row) -> (U [R, dv], m [R], l [R]) with
    m = max s, l = sum exp(s - m), U = sum exp(s - m) v; (0, -inf, 0) for a row without keys."""
    q, k, v = _f64(q), _f64(k_shard), _f64(v_shard)
    n = q.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    u = np.zeros((rows.shape[0], v.shape[1]))
    m = np.full(rows.shape[0], NEG_INF)
    l = np.zeros(rows.shape[0])
    s_all = float(scale) * (q[rows] @ k.T)
    for r, i in enumerate(rows):
        keys = np.arange(k.shape[0])
        if causal:
            keys = keys[key_offset + keys <= i]
        if keys.shape[0] == 0:
            continue
        s = s_all[r, keys]
        m[r] = s.max()
        e = np.exp(s - m[r])
        l[r] = e.sum()
        u[r] = e @ v[keys]
    return u, m, l


def combine(u_parts, m_parts, l_parts):
    """Merge partial (U, m, l) triples of the same query rows.

    u_parts [R, S, dv] unnormalised numerators, m_parts [R, S] maxima (natural
    log units of scaled scores), l_parts [R, S] denominators.  The merge of
    iceferryling §6: m = max_s m_s, l = sum_s exp(m_s - m) l_s,
    O = sum_s exp(m_s - m) U_s / l; lse = m + log(l).  An empty partial has
    m = -inf, l = 0, U = 0 and weight 0; a row whose partials are all empty
    gets O = 0, lse = -inf.
    """
    u, m_p, l_p = _f64(u_parts), _f64(m_parts), _f64(l_parts)
    m = m_p.max(axis=1)
    base = np.where(np.isneginf(m), 0.0, m)
    w = np.exp(m_p - base[:, None])
    l = (w * l_p).sum(axis=1)
    num = (w[:, :, None] * u).sum(axis=1)
    safe_l = np.where(l > 0, l, 1.0)
    o = np.where(l[:, None] > 0, num / safe_l[:, None], 0.0)
    lse = np.where(l > 0, m + np.log(safe_l), NEG_INF)
    return o, lse


def chunk_partials(q_row, k, v, scale: float, chunk: int):
    """FlashDecoding map step for one query row: a partial per KV chunk.

    q_row [d], k/v [L, d]; chunk c covers keys [c*chunk, min(L, (c+1)*chunk)).
    Each partial is the plain definition restricted to its chunk:
    m_c = max s, l_c = sum exp(s - m_c), U_c = sum exp(s - m_c) v
    (cnblogs §三 场景 B step 2: local O_partial with max m and normaliser l).
    Returns U [C, dv], m [C], l [C].
    """
    q_row, k, v = _f64(q_row), _f64(k), _f64(v)
    n_keys = k.shape[0]
    n_chunks = -(-n_keys // chunk)
    u = np.zeros((n_chunks, v.shape[1]))
    m = np.full(n_chunks, NEG_INF)
    l = np.zeros(n_chunks)
    s_all = float(scale) * (k @ q_row)
    for c in range(n_chunks):
        s = s_all[c * chunk:(c + 1) * chunk]
        m[c] = s.max()
        e = np.exp(s - m[c])
        l[c] = e.sum()
        u[c] = e @ v[c * chunk:(c + 1) * chunk]
    return u, m, l


def decode(q, k, v, scale: float, pairs=None):
    """Single-token decode: q [B, H, d], k/v [B, H, L, d] -> O [P, dv], lse [P].

    The plain definition with one query row and every key admissible.
    ``pairs`` is an optional [P, 2] array of (b, h) rows to evaluate
    (default: every (b, h) in order).
    """
    b_, h_ = q.shape[0], q.shape[1]
    if pairs is None:
        pairs = [(b, h) for b in range(b_) for h in range(h_)]
    pairs = [(int(b), int(h)) for b, h in pairs]
    dv = v.shape[-1]
    out = np.zeros((len(pairs), dv))
    lse = np.zeros(len(pairs))
    for idx, (b, h) in enumerate(pairs):
        o, ls = attention_head(_f64(q[b, h])[None, :], _f64(k[b, h]), _f64(v[b, h]), scale, False)
        out[idx], lse[idx] = o[0], ls[0]
    return out, lse


def paged_rows(pages, block_table, b: int, h: int, n_keys: int) -> np.ndarray:
    """Rows 0 .. n_keys-1 of sequence b, head h, read from a paged pool [P, H, page_size, d]:
    key j sits in row j % page_size of pool page block_table[b][j // page_size]; a page id
    outside [0, P) reads as zeros."""
    pages = _f64(pages)
    n_pages, _, page_size, d = pages.shape
    out = np.zeros((n_keys, d))
    for j in range(0, n_keys, page_size):
        pid = int(block_table[b][j // page_size])
        m = min(page_size, n_keys - j)
        if 0 <= pid < n_pages:
            out[j:j + m] = pages[pid, h, :m]
    return out


def decode_paged(q, k_pages, v_pages, block_table, seq_lens, scale: float, pairs=None):
    """Decode over a paged KV cache (iceferryling §13, paged block table): sequence b has
    seq_lens[b] keys, gathered through ``paged_rows``; then ``decode``'s plain definition.
    q [B, H, d] -> O [P, dv], lse [P] for ``pairs`` (default every (b, h))."""
    b_, h_ = q.shape[0], q.shape[1]
    if pairs is None:
        pairs = [(b, h) for b in range(b_) for h in range(h_)]
    pairs = [(int(b), int(h)) for b, h in pairs]
    table = np.asarray(block_table, dtype=np.int64)
    lens = np.asarray(seq_lens, dtype=np.int64)
    out = np.zeros((len(pairs), _f64(v_pages).shape[-1]))
    lse = np.zeros(len(pairs))
    for idx, (b, h) in enumerate(pairs):
        n = max(int(lens[b]), 0)
        kb = paged_rows(k_pages, table, b, h, n)
        vb = paged_rows(v_pages, table, b, h, n)
        o, ls = attention_head(_f64(q[b, h])[None, :], kb, vb, scale, False)
        out[idx], lse[idx] = o[0], ls[0]
    return out, lse


def attention_backward_head(q, k, v, do, scale: float, causal: bool = False):
    """Gradients of O = softmax(scale q k^T) v for one head, fp64.

    q [N, d], k/v [Nk, d], do [N, dv] -> (dq [N, d], dk [Nk, d], dv [Nk, dv]).
    Triton-tutorial §8.8.1: dV = P^T dO, dP = dO V^T; §8.8.3:
    D_i = sum_j P_ij dP_ij, dS_ij = P_ij (dP_ij - D_i); dQ = scale dS K,
    dK = scale dS^T Q.  Masked pairs have P = 0 and so dS = 0; a query row
    with no admissible key gets zero gradient.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    n, nk = q.shape[0], k.shape[0]
    s = float(scale) * (q @ k.T)
    if causal:
        s = np.where(np.arange(nk)[None, :] > np.arange(n)[:, None], NEG_INF, s)
    p = np.zeros_like(s)
    for i in range(n):
        row = s[i]
        if np.all(np.isneginf(row)):
            continue
        e = np.exp(row - row.max())
        p[i] = e / e.sum()
    dv = p.T @ do
    dp = do @ v.T
    dd = (dp * p).sum(axis=1)
    ds = p * (dp - dd[:, None])
    dq = float(scale) * (ds @ k)
    dk = float(scale) * (ds.T @ q)
    return dq, dk, dv


def attention_backward(q, k, v, do, scale: float, causal: bool = False):
    """attention_backward_head over [B, H, N, d] tensors; fp64 results."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            dq[b, h], dk[b, h], dv[b, h] = attention_backward_head(q[b, h], k[b, h], v[b, h], do[b, h], scale,
                                                                   causal)
    return dq, dk, dv


def attention_backward_rows(q, k, v, do, scale: float, causal: bool = False, q_rows=None, k_rows=None,
                            block: int = 512):
    """Gradients of one head at selected rows, fp64: dQ for the query rows ``q_rows``, dK and dV for
    the key rows ``k_rows`` (either may be None).

    The definitions of ``attention_backward_head`` (triton-tutorial §8.8.1: dV = P^T dO,
    dP = dO V^T; §8.8.3: D_i = sum_j P_ij dP_ij, dS = P (dP - D); dQ = scale dS K,
    dK = scale dS^T Q), restricted to those rows and columns so that a head of 8192 rows fits in
    memory.  dS_ij needs every query row's softmax normaliser and D_i, so the score rows of all
    queries are formed first (``block`` rows at a time) for m_i = max_j s_ij,
    l_i = sum_j exp(s_ij - m_i) and D_i; then the selected rows (dQ) or columns (dK, dV) of
    P = exp(s - m) / l, dP and dS are formed explicitly and contracted.  A query row with no
    admissible key has P = 0 and zero gradients.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    n, nk = q.shape[0], k.shape[0]
    scale = float(scale)
    m = np.full(n, NEG_INF)
    l = np.zeros(n)
    dd = np.zeros(n)

    def scores(rows, cols):
        s = scale * (q[rows] @ k[cols].T)
        if causal:
            s = np.where(cols[None, :] > rows[:, None], NEG_INF, s)
        return s

    def probs(rows, cols):
        s = scores(rows, cols)
        base = np.where(np.isfinite(m[rows]), m[rows], 0.0)
        e = np.exp(s - base[:, None])  # masked scores give exp(-inf) = 0
        return e / np.where(l[rows] > 0, l[rows], 1.0)[:, None]

    all_keys = np.arange(nk)
    for r0 in range(0, n, block):
        rows = np.arange(r0, min(n, r0 + block))
        s = scores(rows, all_keys)
        mx = s.max(axis=1) if nk > 0 else np.full(rows.shape[0], NEG_INF)
        base = np.where(np.isfinite(mx), mx, 0.0)
        e = np.exp(s - base[:, None])
        m[rows] = mx
        l[rows] = e.sum(axis=1)
        p = e / np.where(l[rows] > 0, l[rows], 1.0)[:, None]
        dd[rows] = (p * (do[rows] @ v.T)).sum(axis=1)

    dq = dk = dv = None
    if q_rows is not None:
        rows = np.asarray(q_rows, dtype=np.int64)
        p = probs(rows, all_keys)
        ds = p * ((do[rows] @ v.T) - dd[rows][:, None])
        dq = scale * (ds @ k)
    if k_rows is not None:
        cols = np.asarray(k_rows, dtype=np.int64)
        all_rows = np.arange(n)
        p = probs(all_rows, cols)  # column j of P for every query row
        ds = p * ((do @ v[cols].T) - dd[:, None])
        dv = p.T @ do
        dk = scale * (ds.T @ q)
    return dq, dk, dv


def backward_delta(o, do):
    """D_i = rowsum(O_i * dO_i) (triton-tutorial §8.8.3, the preprocess step)."""
    return (_f64(o) * _f64(do)).sum(axis=-1)


def e4m3_values() -> np.ndarray:
    """The 256 E4M3 (fn variant) codes as fp64: 1 sign, 4 exponent (bias 7), 3 mantissa bits;
    exponent 0 is subnormal (m/8 * 2^-6); code 0x7F/0xFF is NaN (no infinities)."""
    vals = np.empty(256)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def round_to_e4m3(x) -> np.ndarray:
    """Codes (uint8) of the nearest E4M3 values to fp32 x: ties to the even code, |x| > 448 -> +-448,
    the sign kept (also on zero)."""
    x = np.asarray(x, dtype=np.float64)
    vals = e4m3_values()
    pos_codes = np.arange(0, 0x7F)            # 0 .. 448 (0x7E), ascending values
    pos_vals = vals[pos_codes]
    a = np.minimum(np.abs(x), 448.0)
    idx = np.searchsorted(pos_vals, a)         # first code with value >= a
    idx = np.clip(idx, 1, len(pos_vals) - 1)
    lo, hi = pos_vals[idx - 1], pos_vals[idx]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & ((pos_codes[idx] & 1) == 0))
    code = np.where(pick_hi, pos_codes[idx], pos_codes[idx - 1])
    code = np.where(a == 0, 0, code)
    sign = np.signbit(x).astype(np.int64) << 7  # negative values that round to zero give -0 (0x80)
    return (code | sign).astype(np.uint8)


def quantize_e4m3_blocks(x, block: int = 128):
    """Block quantization of [B, H, N, d] values along N: returns (codes uint8 [B, H, N, d],
    scales fp32 [B, H, ceil(N/block)]).  scale = amax / 448 in fp32 (1 for an all-zero block) and
    the code of x / scale (fp32 division) rounded to nearest E4M3."""
    x32 = np.asarray(_f64(x), dtype=np.float32)
    b_, h_, n, d = x32.shape
    nb = -(-n // block)
    codes = np.zeros(x32.shape, dtype=np.uint8)
    scales = np.zeros((b_, h_, nb), dtype=np.float32)
    for b in range(b_):
        for h in range(h_):
            for t in range(nb):
                blk = x32[b, h, t * block:(t + 1) * block]
                amax = np.float32(np.abs(blk).max())
                sc = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
                scales[b, h, t] = sc
                codes[b, h, t * block:(t + 1) * block] = round_to_e4m3((blk / sc).astype(np.float32))
    return codes, scales


def dequantize_blocks(codes, scales, block: int = 128):
    """E4M3 codes [B, H, N, d] and per-block scales -> fp64 values."""
    vals = e4m3_values()[np.asarray(codes, dtype=np.int64)]
    sc = np.repeat(np.asarray(scales, dtype=np.float64), block, axis=2)[:, :, :vals.shape[2]]
    return vals * sc[..., None]



def attention_fp8_head(q8, sq, k8, sk, v8, sv, scale: float, causal: bool = False, rows=None, block: int = 128,
                       quantize_p: bool = True, trace: list | None = None):
    """FP8 forward for one head, in the order of triton-tutorial §8.9.3 / §8.9.6.

    q8, k8, v8: [N, d] E4M3 codes; sq, sk, sv: [ceil(N/block)] fp32 block scales (row r of
    a tensor dequantizes as value(code) * s[r // block]).  Key tiles of ``block`` keys, one
    per V block, in order; per tile:
        S     = (Q8 K8_j^T) * s_q[i] * s_k[j] * scale
        m_new = max(m, rowmax S);  alpha = exp(m - m_new);  p = exp(S - m_new)
        l     = alpha * l + rowsum(p)                    (the unquantized p)
        P~    = E4M3(fp32(p) / s_p),  s_p = max(s_v) / (256 s_v[j])
        U     = alpha * U + (P~ V8_j) * (s_p * s_v[j])
    then O = U / l and lse = m + log(l).  ``quantize_p=False`` uses p itself in the second
    GEMM.  Returns (O [R, d], lse [R]) for ``rows`` (default all).  When ``trace`` is a list,
    one dict per key tile is appended: its key indices ``cols``, the fp32 values ``x`` that
    are rounded to P~ codes, and the running max ``m`` after the tile.
    """
    vals = e4m3_values()
    q8 = np.asarray(q8, dtype=np.int64)
    k8 = np.asarray(k8, dtype=np.int64)
    v8 = np.asarray(v8, dtype=np.int64)
    sq = np.asarray(sq, dtype=np.float32)
    sk = np.asarray(sk, dtype=np.float32)
    sv = np.asarray(sv, dtype=np.float32)
    n, nk = q8.shape[0], k8.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    qv, kv, vv = vals[q8[rows]], vals[k8], vals[v8]
    s_q = sq[rows // block].astype(np.float64)
    sv_max = np.float32(sv.max())
    r = rows.shape[0]
    m = np.full(r, NEG_INF)
    l = np.zeros(r)
    u = np.zeros((r, vv.shape[1]))
    for j in range(-(-nk // block)):
        cols = np.arange(j * block, min((j + 1) * block, nk))
        s = (qv @ kv[cols].T) * (s_q[:, None] * float(sk[j]) * float(scale))
        if causal:
            s = np.where(cols[None, :] > rows[:, None], NEG_INF, s)
        m_new = np.maximum(m, s.max(axis=1))
        base = np.where(np.isneginf(m_new), 0.0, m_new)  # fully-masked guard
        alpha = np.exp(m - base)
        p = np.exp(s - base[:, None])
        l = alpha * l + p.sum(axis=1)
        if quantize_p:
            inv_sp = np.float32(np.float32(256.0) * sv[j]) / sv_max     # 1 / s_p, in fp32
            x = p.astype(np.float32) * inv_sp
            if trace is not None:
                trace.append({"cols": cols, "x": x, "m": m_new.copy()})
            p_t = vals[round_to_e4m3(x).astype(np.int64)]
            s_p = float(sv_max) / (256.0 * float(sv[j]))
            u = alpha[:, None] * u + (p_t @ vv[cols]) * (s_p * float(sv[j]))
        else:
            u = alpha[:, None] * u + p @ (vv[cols] * float(sv[j]))
        m = m_new
    safe_l = np.where(l > 0, l, 1.0)
    o = np.where(l[:, None] > 0, u / safe_l[:, None], 0.0)
    lse = np.where(l > 0, m + np.log(safe_l), NEG_INF)
    return o, lse


def attention_fp8(q8, sq, k8, sk, v8, sv, scale: float, causal: bool = False, rows=None, block: int = 128,
                  quantize_p: bool = True):
    """attention_fp8_head over [B, H, N, d] codes and [B, H, nb] scales; ``rows`` as for ``attention``."""
    b_, h_, n = q8.shape[0], q8.shape[1], q8.shape[2]
    r = n if rows is None else np.asarray(rows).shape[-1]
    out = np.zeros((b_, h_, r, q8.shape[-1]))
    lse = np.zeros((b_, h_, r))
    for b in range(b_):
        for h in range(h_):
            sel = None
            if rows is not None:
                rw = np.asarray(rows, dtype=np.int64)
                sel = rw if rw.ndim == 1 else rw[b, h]
            out[b, h], lse[b, h] = attention_fp8_head(q8[b, h], sq[b, h], k8[b, h], sk[b, h], v8[b, h], sv[b, h],
                                                      scale, causal, sel, block, quantize_p)
    return out, lse
