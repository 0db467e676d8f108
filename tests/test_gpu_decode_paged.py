"""GPU parity of fa_decode_paged (split-KV decode over a paged KV cache) against the
oracle's decode_paged, with the bounds of the contiguous decode (same kernels, same
arithmetic; only the key addresses differ)."""

import math

import numpy as np
import pytest
import torch

import oracle
from _util import assert_parity, ensure_built
from exact_attention_06_gb300 import fattn, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def make_paged(B, H, lens, d, page_size, seed, spare_pages=3, max_pages=None):
    """A pool holding every sequence's pages in a seeded random order, plus spare pages; every
    slot no sequence owns (spare pages, the tail of a last page) holds NaN."""
    n_of = [-(-int(n) // page_size) for n in lens]
    max_pages = max_pages or max(max(n_of), 1)
    P = sum(n_of) + spare_pages
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(P, generator=g)
    kp = torch.full((P, H, page_size, d), float("nan"), dtype=torch.bfloat16)
    vp = torch.full_like(kp, float("nan"))
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    nxt = 0
    for b in range(B):
        kb = inputs.normal_bf16((H, int(lens[b]), d), seed=seed * 100 + 2 * b)
        vb = inputs.normal_bf16((H, int(lens[b]), d), seed=seed * 100 + 2 * b + 1)
        for i in range(n_of[b]):
            pid = int(perm[nxt])
            nxt += 1
            table[b, i] = pid
            rows = slice(i * page_size, min((i + 1) * page_size, int(lens[b])))
            m = rows.stop - rows.start
            kp[pid, :, :m] = kb[:, rows]
            vp[pid, :, :m] = vb[:, rows]
    q = inputs.normal_bf16((B, H, d), seed=seed * 100 + 99)
    return q, kp, vp, table, torch.tensor(lens, dtype=torch.int32)


def run_paged(q, kp, vp, table, lens, scale, max_seq_len, splits=0, o_fp32=False):
    B, H, d = q.shape
    o = torch.full((B, H, d), float("nan"), dtype=torch.float32 if o_fp32 else torch.bfloat16, device=DEV)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
    fattn.fa_decode_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), lens.to(DEV), o, lse, scale,
                          max_seq_len, splits=splits)
    fattn.fa_get_status()
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("page_size", [64, 128, 256])
def test_paged_decode_ragged_lengths(d, page_size):
    lens = [1, 63, 64, 65, 300, 1000, 2113, 0]
    B, H = len(lens), 3
    q, kp, vp, table, lt = make_paged(B, H, lens, d, page_size, seed=page_size + d)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle.decode_paged(q, kp, vp, table.numpy(), lt.numpy(), scale)
    L = max(lens)
    n_chunks = -(-L // 128)
    for splits in sorted({0, 1, 3, n_chunks}):
        o, lse = run_paged(q, kp, vp, table, lt, scale, L, splits, o_fp32=True)
        assert_parity(o.reshape(B * H, d), lse.reshape(B * H), o_ref, lse_ref,
                      f"d={d} page={page_size} splits={splits} fp32")
        ob, lseb = run_paged(q, kp, vp, table, lt, scale, L, splits)
        assert_parity(ob.reshape(B * H, d), lseb.reshape(B * H), o_ref, lse_ref,
                      f"d={d} page={page_size} splits={splits}")
        assert torch.equal(lse, lseb)


def test_paged_decode_foreign_page_ids_read_zeros():
    # ids -1 and >= P inside a sequence's length read as zero rows, as the oracle defines them
    lens = [500, 300]
    q, kp, vp, table, lt = make_paged(2, 2, lens, 128, 64, seed=5, spare_pages=0)
    table[0, 2] = -1
    table[1, 1] = kp.shape[0] + 4
    kp[torch.isnan(kp)] = 0  # the pages these ids displace are simply not referenced
    o_ref, lse_ref = oracle.decode_paged(q, kp, vp, table.numpy(), lt.numpy(), 0.1)
    o, lse = run_paged(q, kp, vp, table, lt, 0.1, 500, o_fp32=True)
    assert_parity(o.reshape(4, 128), lse.reshape(4), o_ref, lse_ref, "foreign ids")


def test_paged_decode_lengths_clamped_to_max_seq_len():
    lens = [700, 200]
    q, kp, vp, table, lt = make_paged(2, 1, lens, 64, 64, seed=9)
    o_ref, lse_ref = oracle.decode_paged(q, kp, vp, table.numpy(), np.array([512, 200]), 0.125)
    o, lse = run_paged(q, kp, vp, table, lt, 0.125, 512, o_fp32=True)  # 700 > max_seq_len = 512: 512 keys
    assert_parity(o.reshape(2, 64), lse.reshape(2), o_ref, lse_ref, "clamped")


def test_paged_decode_full_size_sampled_pairs():
    # B64 H32 L32768 d128 with 128-key pages in a shuffled pool (the bench's paged workload)
    B, H, L, d, ps = 64, 32, 32768, 128, 128
    n = L // ps
    q, k, v = inputs.decode_inputs(B, H, L, d, seed=0, device=DEV)
    perm = torch.randperm(B * n, generator=torch.Generator().manual_seed(3)).to(DEV)
    table = perm.view(B, n).to(torch.int32)
    kp = torch.empty((B * n, H, ps, d), dtype=torch.bfloat16, device=DEV)
    vp = torch.empty_like(kp)
    # pool page table[b, i] <- keys i*ps .. of sequence b (all heads)
    kp[perm] = k.view(B, H, n, ps, d).permute(0, 2, 1, 3, 4).reshape(B * n, H, ps, d)
    vp[perm] = v.view(B, H, n, ps, d).permute(0, 2, 1, 3, 4).reshape(B * n, H, ps, d)
    lens = torch.full((B,), L, dtype=torch.int32, device=DEV)
    outs = []
    for dt in (torch.bfloat16, torch.float32):
        o = torch.empty((B, H, d), dtype=dt, device=DEV)
        lse = torch.empty((B, H), dtype=torch.float32, device=DEV)
        fattn.fa_decode_paged(q, kp, vp, table, lens, o, lse, 1 / math.sqrt(d), L)
        fattn.fa_get_status()
        outs.append((o, lse, str(dt)))
    del kp, vp
    rows = inputs.sample_rows(B * H, 48, seed=11).numpy()
    pairs = [(int(r) // H, int(r) % H) for r in rows]
    kc = torch.stack([k[b, h] for b, h in pairs]).cpu()
    vc = torch.stack([v[b, h] for b, h in pairs]).cpu()
    qc = torch.stack([q[b, h] for b, h in pairs]).cpu()
    o_ref, lse_ref = oracle.decode(qc[:, None], kc[:, None], vc[:, None], 1 / math.sqrt(d))
    for o, lse, tag in outs:
        got_o = torch.stack([o[b, h] for b, h in pairs])
        got_l = torch.stack([lse[b, h] for b, h in pairs])
        # |O| ~ 0.03 over 32768 keys: bf16 O meets the raw bounds as well
        assert_parity(got_o, got_l, o_ref, lse_ref, f"paged full size {tag}", raw=True)
