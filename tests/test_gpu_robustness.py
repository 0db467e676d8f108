"""GPU properties beyond the parity cases: bitwise determinism (no kernel uses atomics or a
run-dependent order), extreme score magnitudes, a very long decode and a wide grid."""

import math

import numpy as np
import pytest
import torch

import oracle
from _util import assert_parity, ensure_built, run_fwd
from exact_attention_06_gb300 import fattn, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_forward_is_bitwise_deterministic(d, causal):
    q, k, v = inputs.prefill_inputs(2, 4, 1000, d, seed=d, device=DEV)
    o1, l1 = run_fwd(q, k, v, 1 / math.sqrt(d), causal)
    o2, l2 = run_fwd(q, k, v, 1 / math.sqrt(d), causal)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_backward_is_bitwise_deterministic():
    B, H, N, d = 1, 4, 777, 128
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=5, device=DEV)
    do = inputs.normal_bf16(q.shape, seed=6, device=DEV)
    o, lse = run_fwd(q, k, v, 1 / math.sqrt(d), True)
    grads = []
    for _ in range(2):
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        fattn.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, 1 / math.sqrt(d), True)
        fattn.fa_get_status()
        grads.append((dq, dk, dv))
    for a, b in zip(*grads):
        assert torch.equal(a, b)


@pytest.mark.parametrize("causal", [False, True])
def test_extreme_scores_do_not_overflow(causal):
    # q and k scaled by 8: scaled scores reach several hundred (exp overflows fp32 past 88), so
    # without the running max every row would overflow; rows are then nearly one-hot
    B, H, N, d = 1, 2, 640, 128
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=12, device=DEV)
    q, k = q * 8, k * 8  # exact in bf16 (a power of two)
    o, lse = run_fwd(q, k, v, 1 / math.sqrt(d), causal, o_fp32=True)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(d), causal)
    assert np.abs(lse_ref).max() > 200
    assert_parity(o, lse, o_ref, lse_ref, "x8 scores")


def test_decode_very_long_sequence():
    # B1 H2 L = 262144 (2048 chunks): automatic splits, every split merged by the combine
    B, H, L, d = 1, 2, 262144, 128
    q, k, v = inputs.decode_inputs(B, H, L, d, seed=21, device=DEV)
    o = torch.empty((B, H, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((B, H), dtype=torch.float32, device=DEV)
    ws = torch.empty(fattn.fa_decode_workspace_bytes(B, H, L, d, 128, 0), dtype=torch.uint8, device=DEV)
    fattn.fa_decode_splitkv(q, k, v, o, lse, 1 / math.sqrt(d), ws, 128, 0)
    fattn.fa_get_status()
    o_ref, lse_ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), 1 / math.sqrt(d))
    assert_parity(o.reshape(B * H, d), lse.reshape(B * H), o_ref, lse_ref, "L=262144")


def test_forward_wide_grid():
    # B*H = 4096 heads of N = 200 (a ragged second tile): grid.x = 4096
    B, H, N, d = 64, 64, 200, 64
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=33, device=DEV)
    o, lse = run_fwd(q, k, v, 0.125, False, o_fp32=True)
    rows = inputs.sample_rows_per_head(B, H, N, 3, seed=4)
    picks = [(0, 0), (17, 41), (63, 63)]
    for b, h in picks:
        sel = rows[b, h].numpy()
        o_ref, lse_ref = oracle.attention_head(q[b, h].cpu(), k[b, h].cpu(), v[b, h].cpu(), 0.125, False, rows=sel)
        got_o = o[b, h].index_select(0, rows[b, h].to(DEV))
        got_l = lse[b, h].index_select(0, rows[b, h].to(DEV))
        assert_parity(got_o, got_l, o_ref, lse_ref, f"b{b} h{h}")
    # and no row anywhere is left unwritten
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_back_to_back_dependent_launches(d, causal):
    # The forward is launched with programmatic stream serialization: its set-up may overlap the
    # previous kernel, and its global accesses must wait for it.  Chain three forwards on one
    # stream without a synchronisation, each reading the previous one's output as its q (and
    # writing over the buffer the previous one read), then check every link against the oracle.
    B, H, N = 1, 4, 700
    scale = 1.0 / math.sqrt(d)
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=40 + d, device=DEV)
    bufs = [q.clone(), torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)]
    lses = [torch.empty((B, H, N), dtype=torch.float32, device=DEV) for _ in range(3)]
    for i in range(3):
        fattn.fa_fwd_ex(bufs[i], k, v, bufs[i + 1], lses[i], scale, causal)
    fattn.fa_get_status()
    for i in range(3):
        o_ref, lse_ref = oracle.attention(bufs[i].cpu(), k.cpu(), v.cpu(), scale, causal)
        assert_parity(bufs[i + 1], lses[i], o_ref, lse_ref, f"link {i}")


def test_back_to_back_ping_pong_overwrites_inputs():
    # Two buffers A, B: A -> B, B -> A, A -> B.  The second launch overwrites A while the first
    # one reads it unless its writes wait for the first launch to complete.  The oracle chains
    # the same three steps, rounding each output to bf16 as the next input.
    B, H, N, d = 1, 4, 700, 64
    scale = 0.125
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=50, device=DEV)
    a, b = q.clone(), torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    fattn.fa_fwd_ex(a, k, v, b, lse, scale, False)
    fattn.fa_fwd_ex(b, k, v, a, lse, scale, False)
    fattn.fa_fwd_ex(a, k, v, b, lse, scale, False)
    fattn.fa_get_status()
    x = q.cpu()
    for _ in range(3):
        o_ref, lse_ref = oracle.attention(x, k.cpu(), v.cpu(), scale, False)
        x = torch.from_numpy(o_ref).reshape(B, H, N, d).to(torch.bfloat16)
    assert_parity(b, lse, o_ref, lse_ref, "ping-pong")


# The persistent forward (non-causal d = 64): many CTAs walk many items with three MMA-issuing
# threads and barrier phases counted across items.  Repeated launches over item mixes (whole
# blocks, single query tiles of a split last round, key pieces with a workspace, a second tile
# past N) must keep the status clear and give bit-identical results.
@pytest.mark.parametrize("B,H,N", [(4, 16, 2048), (8, 16, 1000), (1, 2, 2100), (2, 3, 777), (16, 16, 4096)])
def test_persistent_forward_repeated_launches(B, H, N):
    q, k, v = inputs.prefill_inputs(B, H, N, 64, seed=N, device=DEV)
    nb = fattn.fa_fwd_workspace_bytes(B, H, N, 64, False)
    modes = [None] + ([torch.empty(nb, dtype=torch.uint8, device=DEV)] if nb else [])
    for ws in modes:
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
        fattn.fa_fwd_ex(q, k, v, o, lse, 0.125, False, workspace=ws)
        fattn.fa_get_status()
        o_first, l_first = o.clone(), lse.clone()
        for _ in range(40):
            fattn.fa_fwd_ex(q, k, v, o, lse, 0.125, False, workspace=ws)
        fattn.fa_get_status()
        assert torch.equal(o, o_first) and torch.equal(lse, l_first)
