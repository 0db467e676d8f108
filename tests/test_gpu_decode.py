"""GPU parity of fa_decode_splitkv and fa_combine against the fp64 oracle."""

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


def run_decode(q, k, v, scale, splits=0, o_fp32=False):
    B, H, L, d = k.shape
    o = torch.full((B, H, d), float("nan"), dtype=torch.float32 if o_fp32 else torch.bfloat16, device=DEV)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
    nbytes = fattn.fa_decode_workspace_bytes(B, H, L, d, 128, splits)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    fattn.fa_decode_splitkv(q, k, v, o, lse, scale, ws, 128, splits)
    fattn.fa_get_status()
    return o, lse, ws


def _pairs(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L", [1, 63, 64, 127, 128, 129, 1000, 4103])
def test_decode_small_shapes_all_split_counts(L, d):
    B, H = 2, 3
    q, k, v = inputs.decode_inputs(B, H, L, d, seed=L + d, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), scale)
    n_chunks = -(-L // 128)
    for splits in sorted({0, 1, min(3, n_chunks), n_chunks}):
        o, lse, _ = run_decode(q, k, v, scale, splits, o_fp32=True)
        assert_parity(o.reshape(B * H, d), lse.reshape(B * H), o_ref, lse_ref, f"L={L} d={d} splits={splits} fp32")
        ob, lseb, _ = run_decode(q, k, v, scale, splits)
        # bf16 O: held to the raw bounds once a row averages enough keys that |O| is small
        assert_parity(ob.reshape(B * H, d), lseb.reshape(B * H), o_ref, lse_ref, f"L={L} d={d} splits={splits}",
                      raw=L >= 1000)
        assert torch.equal(lse, lseb)


def test_decode_partials_are_the_oracle_chunk_partials():
    """With one split per 128-key chunk the workspace holds each chunk's (U, m, l)."""
    B, H, L, d = 1, 2, 700, 128
    q, k, v = inputs.decode_inputs(B, H, L, d, seed=4, device=DEV)
    scale = 1.0 / math.sqrt(d)
    n_chunks = -(-L // 128)
    o, lse, ws = run_decode(q, k, v, scale, n_chunks)
    R, S = B * H, n_chunks
    u = ws[: R * S * d * 4].view(torch.float32).reshape(R, S, d).cpu().double().numpy()
    m_off = ((R * S * d * 4 + 255) // 256) * 256
    m = ws[m_off: m_off + R * S * 4].view(torch.float32).reshape(R, S).cpu().double().numpy()
    l_off = m_off + ((R * S * 4 + 255) // 256) * 256
    l = ws[l_off: l_off + R * S * 4].view(torch.float32).reshape(R, S).cpu().double().numpy()
    for r, (b, h) in enumerate(_pairs(B, H)):
        u_ref, m_ref, l_ref = oracle.chunk_partials(q[b, h].cpu(), k[b, h].cpu(), v[b, h].cpu(), scale, 128)
        np.testing.assert_allclose(m[r], m_ref, atol=1e-4)
        np.testing.assert_allclose(l[r], l_ref, rtol=1e-4)
        np.testing.assert_allclose(u[r] / l[r][:, None], u_ref / l_ref[:, None], atol=5e-3)


def test_empty_splits_have_zero_weight():
    """More splits than needed leaves trailing splits empty (m = -inf, l = 0)."""
    B, H, L, d = 2, 2, 300, 64  # 3 chunks; 3 splits of 1 chunk each
    q, k, v = inputs.decode_inputs(B, H, L, d, seed=8, device=DEV)
    scale = 0.125
    o_ref, lse_ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), scale)
    for splits in (1, 2, 3):
        o, lse, _ = run_decode(q, k, v, scale, splits, o_fp32=True)
        assert_parity(o.reshape(-1, d), lse.reshape(-1), o_ref, lse_ref, f"splits={splits}")


@pytest.mark.parametrize("d", [64, 128])
def test_combine_matches_oracle(d):
    R, S = 37, 9
    g = torch.Generator(device=DEV).manual_seed(1)
    # realistic partials: U_s = l_s * o_s with o_s a unit-scale output, so O is a convex combination
    m = torch.randn(R, S, device=DEV, generator=g) * 5
    l = torch.rand(R, S, device=DEV, generator=g) * 100 + 0.5
    u = torch.randn(R, S, d, device=DEV, generator=g) * l[:, :, None]
    m[:, 2] = float("-inf")  # an empty partial in every row
    l[:, 2] = 0
    u[:, 2] = 0
    m[5] = float("-inf")  # a row whose partials are all empty
    l[5] = 0
    u[5] = 0
    o_ref, lse_ref = oracle.combine(u.cpu(), m.cpu(), l.cpu())
    # an empty partial's U and l are not read: garbage there must not matter
    u[:, 2] = float("nan")
    l[:, 2] = float("nan")
    u[5] = float("nan")
    keep = [r for r in range(R) if r != 5]
    lses = []
    for dt in (torch.float32, torch.bfloat16):  # fp32 O: the raw bounds; bf16 O: after its own rounding
        o = torch.full((R, d), float("nan"), dtype=dt, device=DEV)
        lse = torch.empty(R, dtype=torch.float32, device=DEV)
        fattn.fa_combine(u, m, l, o, lse)
        fattn.fa_get_status()
        assert torch.all(o[5] == 0) and torch.isneginf(lse[5])
        assert_parity(o[keep], lse[keep], o_ref[keep], lse_ref[keep], f"combine {dt}")
        lses.append(lse)
    assert torch.equal(lses[0], lses[1])


def test_decode_config_sampled_rows():
    w = inputs.WORKLOADS["decode"]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    o, lse, _ = run_decode(q, k, v, w.scale, 0)
    o32, lse32, _ = run_decode(q, k, v, w.scale, 0, o_fp32=True)
    idx = inputs.sample_rows(w.B * w.H, w.oracle_rows, seed=3)
    pairs = [(int(i) // w.H, int(i) % w.H) for i in idx]
    o_ref = np.zeros((len(pairs), w.d))
    lse_ref = np.zeros(len(pairs))
    for n, (b, h) in enumerate(pairs):
        o_r, l_r = oracle.decode(q[b:b + 1, h:h + 1].cpu(), k[b:b + 1, h:h + 1].cpu(), v[b:b + 1, h:h + 1].cpu(),
                                 w.scale)
        o_ref[n], lse_ref[n] = o_r[0], l_r[0]
    for oo, ll, tag in ((o, lse, "bf16"), (o32, lse32, "fp32")):
        o_s = torch.stack([oo[b, h] for b, h in pairs])
        lse_s = torch.stack([ll[b, h] for b, h in pairs])
        # |O| ~ 0.03 here: bf16 O meets the raw bounds as well
        assert_parity(o_s, lse_s, o_ref, lse_ref, f"decode B64 H32 L32768 d128 {tag}", raw=True)
    # the literal reading: one partial per 128-key chunk, on a slice of the same cache
    qs, ks, vs = q[:2].contiguous(), k[:2].contiguous(), v[:2].contiguous()
    o1, lse1, _ = run_decode(qs, ks, vs, w.scale, 256)
    o2, lse2, _ = run_decode(qs, ks, vs, w.scale, 0)
    assert float((o1.float() - o2.float()).abs().max()) <= 1e-2
    assert float((lse1 - lse2).abs().max()) <= 1e-4
