"""Failure detection on the GPU, without a fault: every wait in the kernels is
bounded, and a wait that runs out ends the kernel with a status the host reads.

fa_fwd_ex (and fa_decode_splitkv_ex / fa_decode_paged_ex) with a one-cycle wait
budget makes the first waits of every CTA run out (the data they wait for
cannot arrive within one cycle).  The kernel must report FA_ERR_TIMEOUT through
fa_get_status, drain its in-flight copies (and MMAs), free its TMEM, and leave
the context usable: the next normal call on the same inputs must be correct.
"""

import math

import pytest
import torch

import oracle
from _util import assert_parity, ensure_built, run_fwd
from exact_attention_06_gb300 import fattn, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


# (d, causal, O dtype, key split): the persistent d = 64 kernel with fp32 O (stored by each
# thread, the last round as single query tiles) and with bf16 O (the staged TMA store) plus the
# key split's pieces and combine;
# the one-block-per-CTA kernel at d = 128 causal
@pytest.mark.parametrize("d,causal,o_fp32,tail", [(64, False, True, False), (64, False, False, True),
                                                  (128, True, True, False)])
def test_wait_budget_expiry_is_reported_and_the_context_survives(d, causal, o_fp32, tail):
    ensure_built()
    B, H, N = 1, 4, 2000
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=21, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o = torch.zeros(B, H, N, d, dtype=torch.float32 if o_fp32 else torch.bfloat16, device=DEV)
    lse = torch.zeros(B, H, N, dtype=torch.float32, device=DEV)
    ws = None
    if tail:
        nbytes = fattn.fa_fwd_workspace_bytes(B, H, N, d, causal)
        assert nbytes > 0
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    fattn.fa_fwd_ex(q, k, v, o, lse, scale, causal, wait_budget_cycles=1, workspace=ws)
    with pytest.raises(fattn.FattnError) as err:
        fattn.fa_get_status()
    assert err.value.status == fattn.FA_ERR_TIMEOUT
    assert fattn.fa_get_status() == fattn.FA_OK  # the status word was cleared by the read
    # the same context still computes correct results
    o2, lse2 = run_fwd(q, k, v, scale, causal, o_fp32=o_fp32)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, causal,
                                      rows=inputs.sample_rows(N, 256, seed=1).numpy())
    rows = inputs.sample_rows(N, 256, seed=1)
    assert_parity(o2[:, :, rows], lse2[:, :, rows], o_ref, lse_ref, "after a timeout")


@pytest.mark.parametrize("paged", [False, True])
def test_decode_wait_budget_expiry_is_reported_and_the_context_survives(paged):
    ensure_built()
    B, H, L, d, ps = 2, 4, 4992, 128, 128  # 39 pages of 128 keys per sequence
    q, k, v = inputs.decode_inputs(B, H, L, d, seed=31, device=DEV)
    scale = 1.0 / math.sqrt(d)
    n = L // ps
    if paged:
        kp = k.view(B, H, n, ps, d).permute(0, 2, 1, 3, 4).reshape(B * n, H, ps, d).contiguous()
        vp = v.view(B, H, n, ps, d).permute(0, 2, 1, 3, 4).reshape(B * n, H, ps, d).contiguous()
        table = torch.arange(B * n, dtype=torch.int32, device=DEV).view(B, n)
        lens = torch.full((B,), L, dtype=torch.int32, device=DEV)

    def call(o, lse, budget):
        if paged:
            fattn.fa_decode_paged(q, kp, vp, table, lens, o, lse, scale, L, wait_budget_cycles=budget)
        else:
            ws = torch.empty(fattn.fa_decode_workspace_bytes(B, H, L, d, 128, 0), dtype=torch.uint8, device=DEV)
            fattn.fa_decode_splitkv(q, k, v, o, lse, scale, ws, 128, 0, wait_budget_cycles=budget)

    o = torch.zeros(B, H, d, dtype=torch.float32, device=DEV)
    lse = torch.zeros(B, H, dtype=torch.float32, device=DEV)
    call(o, lse, 1)
    with pytest.raises(fattn.FattnError) as err:
        fattn.fa_get_status()
    assert err.value.status == fattn.FA_ERR_TIMEOUT
    assert fattn.fa_get_status() == fattn.FA_OK  # the status word was cleared by the read
    o2 = torch.full((B, H, d), float("nan"), dtype=torch.float32, device=DEV)
    lse2 = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
    call(o2, lse2, 0)
    assert fattn.fa_get_status() == fattn.FA_OK
    o_ref, lse_ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), scale)
    assert_parity(o2.reshape(B * H, d), lse2.reshape(B * H), o_ref, lse_ref, f"decode after a timeout paged={paged}")



def test_backward_wait_budget_expiry_is_reported_and_the_context_survives():
    """fa_bwd_ex with a one-cycle budget: the dK/dV and dQ kernels give up at their first waits,
    drain their copies and MMAs, report FA_ERR_TIMEOUT, and the next backward on the same
    context matches the oracle."""
    ensure_built()
    B, H, N, d = 1, 3, 700, 128
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=41, device=DEV)
    do = inputs.normal_bf16((B, H, N, d), seed=42, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, scale, True)
    grads = [torch.zeros(B, H, N, d, dtype=torch.float32, device=DEV) for _ in range(3)]
    fattn.fa_bwd(q, k, v, o, do, lse, *grads, scale, True, wait_budget_cycles=1)
    with pytest.raises(fattn.FattnError) as err:
        fattn.fa_get_status()
    assert err.value.status == fattn.FA_ERR_TIMEOUT
    assert fattn.fa_get_status() == fattn.FA_OK
    grads = [torch.full((B, H, N, d), float("nan"), dtype=torch.float32, device=DEV) for _ in range(3)]
    fattn.fa_bwd(q, k, v, o, do, lse, *grads, scale, True)
    assert fattn.fa_get_status() == fattn.FA_OK
    ref = oracle.attention_backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), scale, True)
    for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
        e = g.double().cpu().numpy() - r
        assert abs(e).max() <= 2e-2 * abs(r).max(), f"{name} after a timeout"
        assert abs(e).mean() <= 1e-2 * abs(r).mean(), f"{name} after a timeout"
