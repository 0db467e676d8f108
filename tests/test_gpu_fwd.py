"""GPU parity of fa_fwd against the fp64 oracle (bf16 inputs, fp32 accumulation).

Tolerances: max|O - O_ref| <= 1e-2, mean|O - O_ref| <= 1e-3, max|lse - lse_ref| <= 1e-3.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from _util import assert_parity, ensure_built, gather_rows, run_fwd
from exact_attention_06_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _oracle(q, k, v, scale, causal, rows=None):
    return oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, causal, rows=rows)


def test_worked_example_on_the_gpu(golden_dir):
    """cnblogs §二 scores: Q rows e0, e1 (plus two zero rows), keys (s_0j, s_1j), scale 1, N = 4 < 128."""
    with open(os.path.join(golden_dir, "worked_example_cnblogs.json")) as f:
        g = json.load(f)
    s = np.concatenate([np.array(g["S11"]), np.array(g["S12"])], axis=1)
    q = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    q[0, 0, 0, 0] = 1
    q[0, 0, 1, 1] = 1
    k = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    k[0, 0, :, 0] = torch.tensor(s[0])
    k[0, 0, :, 1] = torch.tensor(s[1])
    v = inputs.normal_bf16((1, 1, 4, 64), 77)
    o, lse = run_fwd(q.to(DEV), k.to(DEV), v.to(DEV), 1.0, False, o_fp32=True)
    o_ref, lse_ref = _oracle(q, k, v, 1.0, False)
    assert_parity(o, lse, o_ref, lse_ref, "worked example")
    # closed forms: row 0 lse = 30 + ln(1 + e^-10 + e^-20 + e^-25); zero rows: mean of V, lse = ln 4
    assert abs(float(lse[0, 0, 0]) - (30 + math.log1p(math.exp(-10) + math.exp(-20) + math.exp(-25)))) < 1e-4
    assert abs(float(lse[0, 0, 2]) - math.log(4)) < 1e-5
    np.testing.assert_allclose(o[0, 0, 3].cpu().numpy(), v[0, 0].float().mean(0).numpy(), atol=1e-5)


@pytest.mark.parametrize("o_fp32", [False, True])
def test_tiny_config_all_rows(o_fp32):
    w = inputs.WORKLOADS["tiny"]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    o, lse = run_fwd(q, k, v, w.scale, w.causal, o_fp32=o_fp32)
    o_ref, lse_ref = _oracle(q, k, v, w.scale, w.causal)
    assert_parity(o, lse, o_ref, lse_ref, "tiny")


SMALL_N = [1, 2, 3, 64, 127, 128, 129, 255, 257, 389]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", SMALL_N)
def test_small_and_ragged_shapes(n, causal, d):
    q, k, v = inputs.prefill_inputs(2, 3, n, d, seed=n * 7 + d, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, scale, causal, o_fp32=True)
    o_ref, lse_ref = _oracle(q, k, v, scale, causal)
    assert_parity(o, lse, o_ref, lse_ref, f"N={n} causal={causal} d={d}")
    ob, lseb = run_fwd(q, k, v, scale, causal, o_fp32=False)
    assert_parity(ob, lseb, o_ref, lse_ref, f"bf16 O, N={n} causal={causal} d={d}")
    assert torch.equal(lseb, lse)


@pytest.mark.parametrize("d", [64, 128])
def test_causal_row_zero_is_v0_and_zero_queries_average(d):
    n = 300
    _, k, v = inputs.prefill_inputs(1, 2, n, d, seed=3, device=DEV)
    q = torch.zeros(1, 2, n, d, dtype=torch.bfloat16, device=DEV)
    o, lse = run_fwd(q, k, v, 0.5, True, o_fp32=True)
    np.testing.assert_array_equal(o[:, :, 0].cpu().numpy(), v[:, :, 0].float().cpu().numpy())
    cnt = torch.arange(1, n + 1, dtype=torch.float64)
    np.testing.assert_allclose(lse[0, 0].double().cpu().numpy(), np.log(cnt.numpy()), atol=1e-5)
    mean = torch.cumsum(v.double(), dim=2) / cnt.to(DEV)[None, None, :, None]
    assert float((o.double() - mean).abs().max()) < 1e-4


def test_large_scores_rescale_without_overflow():
    """Scores of magnitude ~100 with growing maxima: alpha far below 1, no inf/NaN."""
    n, d = 600, 64
    q, k, v = inputs.prefill_inputs(1, 2, n, d, seed=9, device=DEV)
    k = (k.float() * torch.linspace(0.5, 4.0, n, device=DEV)[None, None, :, None]).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = run_fwd(q, k, v, 1.0, causal, o_fp32=True)
        o_ref, lse_ref = _oracle(q, k, v, 1.0, causal)
        assert_parity(o, lse, o_ref, lse_ref, f"large scores causal={causal}")


def test_deterministic():
    w = inputs.WORKLOADS["tiny"]
    q, k, v = inputs.prefill_inputs(2, 4, 1000, 128, seed=5, device=DEV)
    o1, l1 = run_fwd(q, k, v, 0.09, True)
    o2, l2 = run_fwd(q, k, v, 0.09, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_prefill_config_all_rows():
    w = inputs.WORKLOADS["prefill"]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    o_ref, lse_ref = _oracle(q, k, v, w.scale, w.causal)
    o, lse = run_fwd(q, k, v, w.scale, w.causal)
    # non-causal N=2048: |O| is small, so bf16 O is held to the raw bounds too
    assert_parity(o, lse, o_ref, lse_ref, "prefill B4 H16 N2048 d64 (bf16 O)", raw=True)
    o32, lse32 = run_fwd(q, k, v, w.scale, w.causal, o_fp32=True)
    assert_parity(o32, lse32, o_ref, lse_ref, "prefill B4 H16 N2048 d64 (fp32 O)")


@pytest.mark.parametrize("name", ["causal", "ragged"])
def test_long_causal_configs_sampled_rows(name):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    rows = inputs.sample_rows_per_head(w.B, w.H, w.N, w.oracle_rows, seed=3)
    # always include the first rows, both sides of the last tile boundary and the last row
    edge = torch.tensor([0, 1, 127, 128, (w.N - 1) // 128 * 128 - 1, (w.N - 1) // 128 * 128, w.N - 1])
    rows = torch.sort(torch.cat([rows, edge.expand(w.B, w.H, -1)], dim=2), dim=2).values
    o_ref = np.zeros((w.B, w.H, rows.shape[2], w.d))
    lse_ref = np.zeros((w.B, w.H, rows.shape[2]))
    for b in range(w.B):
        for h in range(w.H):
            # the sampled rows of a head against that head's full K, V
            o_ref[b, h], lse_ref[b, h] = oracle.attention_head(
                q[b, h].cpu(), k[b, h].cpu(), v[b, h].cpu(), w.scale, w.causal, rows=rows[b, h].numpy())
    for o_fp32 in (True, False):
        o, lse = run_fwd(q, k, v, w.scale, w.causal, o_fp32=o_fp32)
        assert_parity(gather_rows(o, rows), gather_rows(lse, rows), o_ref, lse_ref, f"{name} o_fp32={o_fp32}")


@pytest.mark.parametrize("causal", [True, False])
def test_uneven_head_groups_cover_every_block(causal):
    """37 heads of N = 4096: the block order cuts them into head groups of unequal size (19 + 18
    causal, 13 + 12 + 12 non-causal); every block of every head is computed once and right."""
    B, H, N, d = 1, 37, 4096, 128
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=37, device=DEV)
    scale = 1.0 / math.sqrt(d)
    rows = inputs.sample_rows_per_head(B, H, N, 12, seed=6)
    edge = torch.tensor([0, 255, 256, N - 257, N - 1])
    rows = torch.sort(torch.cat([rows, edge.expand(B, H, -1)], dim=2), dim=2).values
    o_ref, lse_ref = _oracle(q, k, v, scale, causal, rows=rows.numpy())
    o, lse = run_fwd(q, k, v, scale, causal, o_fp32=True)
    assert_parity(gather_rows(o, rows), gather_rows(lse, rows), o_ref, lse_ref, f"37 heads causal={causal}")


@pytest.mark.parametrize("d,causal", [(64, True), (64, False), (128, False)])
def test_long_spiky_sampled_rows(d, causal):
    """Long sequences with x8 key spikes and a ragged last tile (N = 8189) on the schedules the
    bench's workloads do not cover: d = 64 causal (separate P~, fwd_kernel<64, causal>), the
    persistent d = 64 non-causal kernel over 64 key tiles per block, and d = 128 non-causal;
    seeded rows plus tile edges of every head."""
    B, H, N = 1, 6, 8189
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=d + causal, device=DEV, spike=True)
    scale = 1.0 / math.sqrt(d)
    rows = inputs.sample_rows_per_head(B, H, N, 24, seed=8)
    edge = torch.tensor([0, 127, 128, 255, 256, N - 126, N - 125, N - 1])
    rows = torch.sort(torch.cat([rows, edge.expand(B, H, -1)], dim=2), dim=2).values
    o_ref, lse_ref = _oracle(q, k, v, scale, causal, rows=rows.numpy())
    for o_fp32 in (True, False):
        o, lse = run_fwd(q, k, v, scale, causal, o_fp32=o_fp32)
        assert_parity(gather_rows(o, rows), gather_rows(lse, rows), o_ref, lse_ref,
                      f"d={d} N={N} causal={causal} o_fp32={o_fp32}")
