"""GPU parity of the forward's split last round (non-causal d = 64, persistent kernel).

When the last round of 256-row blocks only partly fills the SMs, fa_fwd_ex cuts its blocks:
with a workspace (fa_fwd_workspace_bytes > 0) into key pieces whose partial (U, m, l) rows the
combine kernel merges, else into their two query tiles.  Every shape here is one the planner
splits that way on a 152-SM GB300 (checked through fa_fwd_workspace_bytes), compared with the
oracle and, for key splits, with the same call without a workspace."""

import math

import numpy as np
import pytest
import torch

import oracle
from _util import assert_parity, ensure_built, gather_rows
from exact_attention_06_gb300 import fattn, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def run(q, k, v, scale, o_fp32, workspace=None):
    B, H, N, d = q.shape
    o = torch.full((B, H, N, d), float("nan"), dtype=torch.float32 if o_fp32 else torch.bfloat16, device=DEV)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=DEV)
    fattn.fa_fwd_ex(q, k, v, o, lse, scale, False, workspace=workspace)
    fattn.fa_get_status()
    return o, lse


def key_split_workspace(B, H, N, d, fill=float("nan")):
    """The key split's workspace, filled so that unwritten bytes would show up as NaN."""
    nbytes = fattn.fa_fwd_workspace_bytes(B, H, N, d, False)
    assert nbytes > 0, f"no key split planned for B{B} H{H} N{N} d{d}"
    return torch.full((nbytes // 4,), fill, dtype=torch.float32, device=DEV).view(torch.uint8)


# (B, H, N, d) the planner cuts into key pieces: 8 pieces of 2 key tiles; 4 pieces with a
# ragged query block; 2 pieces of 16 key tiles; 6 pieces with a ragged last key tile; 6 pieces
# with the second query tile of the last block past N (N mod 256 <= 128); 4 pieces, 4 heads
KEY_SPLIT = [(1, 1, 2048, 64), (1, 2, 1000, 64), (1, 4, 4096, 64), (1, 3, 1500, 64), (1, 2, 2100, 64),
             (2, 2, 2048, 64)]
# (B, H, N, d) cut into single query tiles: the prefill workload's shape in miniature (56 of 512
# blocks); ragged blocks; an empty second tile in the last block of every head; one block
QUERY_SPLIT = [(8, 16, 1000, 64), (2, 3, 777, 64), (3, 5, 600, 64), (1, 1, 1100, 64), (1, 1, 256, 64)]


@pytest.mark.parametrize("B,H,N,d", KEY_SPLIT)
@pytest.mark.parametrize("o_fp32", [True, False])
def test_key_split_all_rows(B, H, N, d, o_fp32):
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=N + d, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = run(q, k, v, scale, o_fp32, key_split_workspace(B, H, N, d))
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, False)
    assert_parity(o, lse, o_ref, lse_ref, f"key split B{B} H{H} N{N} d{d} o_fp32={o_fp32}")
    # without a workspace the same call splits by query tiles (or not at all): each piece rounds
    # its own P~ (relative to its own row max) to bf16, so the two differ by about that rounding
    o1, l1 = run(q, k, v, scale, o_fp32)
    assert_parity(o1, l1, o_ref, lse_ref, f"no workspace B{B} H{H} N{N} d{d} o_fp32={o_fp32}")
    assert float((o.float() - o1.float()).abs().max()) <= 2e-3
    assert float((lse - l1).abs().max()) <= 1e-4


@pytest.mark.parametrize("B,H,N,d", QUERY_SPLIT)
@pytest.mark.parametrize("o_fp32", [True, False])
def test_query_split_all_rows(B, H, N, d, o_fp32):
    assert fattn.fa_fwd_workspace_bytes(B, H, N, d, False) == 0  # no key split planned
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=N + d + 1, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = run(q, k, v, scale, o_fp32)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, False)
    assert_parity(o, lse, o_ref, lse_ref, f"query split B{B} H{H} N{N} d{d} o_fp32={o_fp32}")


def test_prefill_workload_fp32_sampled_rows():
    # the bench's launch (B4 H16 N2048 d64: 512 blocks on 152 SMs, the last 56 as 112 single
    # query tiles) with fp32 O; bf16 O on every row is in test_gpu_fwd.py
    w = inputs.WORKLOADS["prefill"]
    assert fattn.fa_fwd_workspace_bytes(w.B, w.H, w.N, w.d, w.causal) == 0
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    rows = inputs.sample_rows_per_head(w.B, w.H, w.N, 96, seed=8)
    edge = torch.tensor([0, 127, 128, 255, 256, w.N - 1])
    rows = torch.sort(torch.cat([rows, edge.expand(w.B, w.H, -1)], dim=2), dim=2).values
    o_ref = np.zeros((w.B, w.H, rows.shape[2], w.d))
    lse_ref = np.zeros((w.B, w.H, rows.shape[2]))
    for b in range(w.B):
        for h in range(w.H):
            o_ref[b, h], lse_ref[b, h] = oracle.attention_head(q[b, h].cpu(), k[b, h].cpu(), v[b, h].cpu(), w.scale,
                                                               False, rows=rows[b, h].numpy())
    o, lse = run(q, k, v, w.scale, True)
    assert_parity(gather_rows(o, rows), gather_rows(lse, rows), o_ref, lse_ref, "prefill, fp32 O")
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


def test_split_launches_are_deterministic():
    q, k, v = inputs.prefill_inputs(1, 2, 1000, 64, seed=3, device=DEV)
    o1, l1 = run(q, k, v, 0.1, False, key_split_workspace(1, 2, 1000, 64))
    o2, l2 = run(q, k, v, 0.1, False, key_split_workspace(1, 2, 1000, 64, fill=0.0))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    q, k, v = inputs.prefill_inputs(8, 16, 1000, 64, seed=4, device=DEV)
    o1, l1 = run(q, k, v, 0.1, False)
    o2, l2 = run(q, k, v, 0.1, False)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_no_key_split_planned_for_causal_d128_or_full_rounds():
    assert fattn.fa_fwd_workspace_bytes(1, 1, 2048, 64, True) == 0
    assert fattn.fa_fwd_workspace_bytes(1, 1, 2048, 128, False) == 0
    assert fattn.fa_fwd_workspace_bytes(1, 1, 256, 64, False) == 0  # two key tiles: nothing to cut
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fattn.fa_fwd_workspace_bytes(sms, 1, 512, 64, False) == 0  # exactly full rounds


def test_key_split_workspace_too_small():
    q, k, v = inputs.prefill_inputs(1, 1, 2048, 64, seed=1, device=DEV)
    need = fattn.fa_fwd_workspace_bytes(1, 1, 2048, 64, False)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 2048), dtype=torch.float32, device=DEV)
    with pytest.raises(fattn.FattnError) as ei:
        fattn.fa_fwd_ex(q, k, v, o, lse, 0.125, False, workspace=ws)
    assert ei.value.status == fattn.FA_ERR_WORKSPACE
