"""GPU parity of the forward's tail split (fa_fwd_ex with a workspace): the blocks of a partly
filled last wave are cut into key pieces whose partial (U, m, l) rows the combine kernel merges.

Every case here is one the planner splits on a 152-SM GB300 (checked through
fa_fwd_workspace_bytes), and is compared with the oracle and with the unsplit launch."""

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


def run_tail(q, k, v, scale, o_fp32, ws_fill=float("nan")):
    """The split launch, with a workspace whose unwritten bytes would show up as NaN."""
    B, H, N, d = q.shape
    nbytes = fattn.fa_fwd_workspace_bytes(B, H, N, d, False)
    assert nbytes > 0, f"no tail split planned for B{B} H{H} N{N} d{d}"
    ws = torch.full((nbytes // 4,), ws_fill, dtype=torch.float32, device=DEV).view(torch.uint8)
    o = torch.full((B, H, N, d), float("nan"), dtype=torch.float32 if o_fp32 else torch.bfloat16, device=DEV)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=DEV)
    fattn.fa_fwd_ex(q, k, v, o, lse, scale, False, workspace=ws)
    fattn.fa_get_status()
    return o, lse


def run_plain(q, k, v, scale, o_fp32):
    B, H, N, d = q.shape
    o = torch.empty((B, H, N, d), dtype=torch.float32 if o_fp32 else torch.bfloat16, device=DEV)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    fattn.fa_fwd_ex(q, k, v, o, lse, scale, False)
    fattn.fa_get_status()
    return o, lse


# (B, H, N, d): 8 pieces of 2 key tiles; 4 pieces with a ragged query block; 2 pieces, the
# second of 1 key tile + 1 key; several heads with a ragged last block per head; pieces of 16
# key tiles; a second query tile past N in every head's last block (N mod 256 <= 128)
SMALL = [(1, 1, 2048, 64), (1, 2, 1000, 64), (1, 1, 513, 64), (2, 3, 777, 64), (1, 4, 4096, 64), (3, 5, 600, 64)]


@pytest.mark.parametrize("B,H,N,d", SMALL)
@pytest.mark.parametrize("o_fp32", [True, False])
def test_tail_split_small_all_rows(B, H, N, d, o_fp32):
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=N + d, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_tail(q, k, v, scale, o_fp32)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, False)
    assert_parity(o, lse, o_ref, lse_ref, f"tail B{B} H{H} N{N} d{d} o_fp32={o_fp32}")
    # and the unsplit launch agrees: each piece rounds its own P~ (relative to its own row max)
    # to bf16, so the two differ by about that rounding, far inside the oracle bounds
    o1, l1 = run_plain(q, k, v, scale, o_fp32)
    assert float((o.float() - o1.float()).abs().max()) <= 2e-3
    assert float((lse - l1).abs().max()) <= 1e-4


def test_tail_split_prefill_workload_all_rows():
    # the bench's launch: B4 H16 N2048 d64 with bf16 O, 512 blocks on 152 SMs, the last 56 cut
    # into two key halves; every row against the oracle
    w = inputs.WORKLOADS["prefill"]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    o, lse = run_tail(q, k, v, w.scale, False)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, False)
    assert_parity(o, lse, o_ref, lse_ref, "prefill tail, all rows (bf16 O)")


def test_tail_split_prefill_workload():
    # the same launch with fp32 O and bf16 O on sampled rows (and tile edges)
    w = inputs.WORKLOADS["prefill"]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    rows = inputs.sample_rows_per_head(w.B, w.H, w.N, 96, seed=8)
    edge = torch.tensor([0, 255, 256, w.N - 1])
    rows = torch.sort(torch.cat([rows, edge.expand(w.B, w.H, -1)], dim=2), dim=2).values
    o_ref = np.zeros((w.B, w.H, rows.shape[2], w.d))
    lse_ref = np.zeros((w.B, w.H, rows.shape[2]))
    for b in range(w.B):
        for h in range(w.H):
            o_ref[b, h], lse_ref[b, h] = oracle.attention_head(q[b, h].cpu(), k[b, h].cpu(), v[b, h].cpu(), w.scale,
                                                               False, rows=rows[b, h].numpy())
    for o_fp32 in (True, False):
        o, lse = run_tail(q, k, v, w.scale, o_fp32)
        assert_parity(gather_rows(o, rows), gather_rows(lse, rows), o_ref, lse_ref, f"prefill tail o_fp32={o_fp32}")
        assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


def test_tail_split_is_deterministic():
    q, k, v = inputs.prefill_inputs(1, 2, 1000, 64, seed=3, device=DEV)
    o1, l1 = run_tail(q, k, v, 0.1, False)
    o2, l2 = run_tail(q, k, v, 0.1, False, ws_fill=0.0)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_no_split_planned_for_causal_d128_or_full_waves():
    assert fattn.fa_fwd_workspace_bytes(4, 16, 2048, 64, True) == 0
    assert fattn.fa_fwd_workspace_bytes(1, 1, 2048, 128, False) == 0
    assert fattn.fa_fwd_workspace_bytes(1, 1, 256, 64, False) == 0  # two key tiles: nothing to cut
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # exactly full waves of 256-row blocks
    assert fattn.fa_fwd_workspace_bytes(sms, 1, 512, 64, False) == 0


def test_tail_split_workspace_too_small():
    q, k, v = inputs.prefill_inputs(1, 1, 2048, 64, seed=1, device=DEV)
    need = fattn.fa_fwd_workspace_bytes(1, 1, 2048, 64, False)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 2048), dtype=torch.float32, device=DEV)
    with pytest.raises(fattn.FattnError) as ei:
        fattn.fa_fwd_ex(q, k, v, o, lse, 0.125, False, workspace=ws)
    assert ei.value.status == fattn.FA_ERR_WORKSPACE
