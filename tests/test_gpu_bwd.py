"""GPU parity of fa_bwd (gradients with recomputation) against the fp64 oracle.

Tolerance (no page states one for the backward): P~ and dS enter the gradient
MMAs rounded to bf16 (2^-9 relative) and D is computed from the bf16 O, with
fp32 accumulation everywhere, so each gradient element carries a few 2^-9 of
relative error.  The bound: max|g - g_ref| <= 2e-2 * max|g_ref| and
mean|g - g_ref| <= 1e-2 * mean|g_ref|, per gradient, for fp32 and bf16 outputs.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from _util import ensure_built
from exact_attention_06_gb300 import fattn, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
REL_MAX, REL_MEAN = 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def run_bwd(q, k, v, do, scale, causal, grad_fp32=True):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    fattn.fa_fwd(q, k, v, o, lse, scale, causal)
    dt = torch.float32 if grad_fp32 else torch.bfloat16
    dq, dk, dv = (torch.full((B, H, N, d), float("nan"), dtype=dt, device=DEV) for _ in range(3))
    fattn.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, causal)
    assert fattn.fa_get_status() == fattn.FA_OK
    return dq, dk, dv


def assert_grads(got, ref, what):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = g.double().cpu().numpy()
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        e = np.abs(g - r)
        scale_max, scale_mean = np.abs(r).max(), np.abs(r).mean()
        if scale_max == 0:
            assert e.max() <= 1e-5, f"{what} {name}: {e.max():.2e} where the gradient is 0"
            continue
        assert e.max() <= REL_MAX * scale_max, f"{what} {name}: max err {e.max():.3e} > {REL_MAX} * {scale_max:.3e}"
        assert e.mean() <= REL_MEAN * scale_mean, f"{what} {name}: mean err {e.mean():.3e} > {REL_MEAN} * {scale_mean:.3e}"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 3, 64, 127, 128, 129, 300, 1000])
def test_backward_small_and_ragged(n, causal, d):
    q, k, v = inputs.prefill_inputs(1, 2, n, d, seed=n + 3 * d, device=DEV)
    do = inputs.normal_bf16((1, 2, n, d), seed=500 + n, device=DEV)
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), scale, causal)
    assert_grads(run_bwd(q, k, v, do, scale, causal, True), ref, f"N={n} causal={causal} d={d} fp32")
    assert_grads(run_bwd(q, k, v, do, scale, causal, False), ref, f"N={n} causal={causal} d={d} bf16")


def test_backward_spiky_scores():
    """x8 key spikes (peaked softmax, large alpha jumps in the forward) at N=2048, d=128, causal."""
    q, k, v = inputs.prefill_inputs(1, 2, 2048, 128, seed=4, device=DEV, spike=True)
    do = inputs.normal_bf16((1, 2, 2048, 128), seed=41, device=DEV)
    scale = 1.0 / math.sqrt(128)
    ref = oracle.attention_backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), scale, True)
    assert_grads(run_bwd(q, k, v, do, scale, True), ref, "spikes")


def test_backward_deterministic_and_identities_at_full_causal_size():
    """B2 H16 N8192 d128 causal: bitwise repeatable, and sum_keys dV = sum_rows dO, sum_keys dK = 0."""
    w = inputs.WORKLOADS["causal"]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    do = inputs.normal_bf16(q.shape, seed=9, device=DEV)
    g1 = run_bwd(q, k, v, do, w.scale, True)
    g2 = run_bwd(q, k, v, do, w.scale, True)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)
    dq, dk, dv = (g.double() for g in g1)
    sum_dv = dv.sum(dim=2)
    sum_do = do.double().sum(dim=2)
    assert float((sum_dv - sum_do).abs().max()) <= 2e-2 * float(sum_do.abs().max())
    assert float(dk.sum(dim=2).abs().max()) <= 2e-2 * float(dk.abs().sum(dim=2).max())


def test_backward_full_causal_size_sampled_rows_against_the_oracle():
    """B2 H16 N8192 d128 causal with x8 key spikes (the bench's backward workload), as the bench runs
    it (bf16 gradients) and with fp32 gradients: on two seeded heads, dQ at 64 seeded query rows and
    dK, dV at 64 seeded key rows (plus tile-edge rows) against the fp64 oracle restricted to those
    rows, which forms every query row's softmax statistics and the keys' full score columns."""
    w = inputs.WORKLOADS["causal"]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    do = inputs.normal_bf16(q.shape, seed=9, device=DEV)
    grads = {dt: run_bwd(q, k, v, do, w.scale, True, grad_fp32=dt) for dt in (True, False)}
    heads = [(int(i) // w.H, int(i) % w.H) for i in inputs.sample_rows(w.B * w.H, 2, seed=21)]
    edge = [0, 1, 127, 128, 4095, 4096, w.N - 129, w.N - 128, w.N - 1]
    for n, (b, h) in enumerate(heads):
        qr = np.unique(np.concatenate([inputs.sample_rows(w.N, 64, seed=30 + n).numpy(), edge]))
        kr = np.unique(np.concatenate([inputs.sample_rows(w.N, 64, seed=40 + n).numpy(), edge]))
        dq_ref, dk_ref, dv_ref = oracle.attention_backward_rows(q[b, h].cpu(), k[b, h].cpu(), v[b, h].cpu(),
                                                                do[b, h].cpu(), w.scale, True, q_rows=qr, k_rows=kr)
        qi, ki = torch.from_numpy(qr).to(DEV), torch.from_numpy(kr).to(DEV)
        for fp32, (dq, dk, dv) in grads.items():
            got = (dq[b, h].index_select(0, qi), dk[b, h].index_select(0, ki), dv[b, h].index_select(0, ki))
            assert_grads(got, (dq_ref, dk_ref, dv_ref), f"full causal b={b} h={h} grad_fp32={fp32}")


def test_backward_uneven_head_groups():
    """37 heads of N = 2048, causal: the key (query) tiles are dispatched in head groups of unequal
    size; dQ, dK, dV of heads in different groups against the row-restricted oracle."""
    B, H, N, d = 1, 37, 2048, 128
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=73, device=DEV)
    do = inputs.normal_bf16((B, H, N, d), seed=74, device=DEV)
    scale = 1.0 / math.sqrt(d)
    got = run_bwd(q, k, v, do, scale, True)
    edge = [0, 127, 128, N - 1]
    for h in (0, 18, 19, 36):
        qr = np.unique(np.concatenate([inputs.sample_rows(N, 24, seed=h).numpy(), edge]))
        kr = np.unique(np.concatenate([inputs.sample_rows(N, 24, seed=100 + h).numpy(), edge]))
        ref = oracle.attention_backward_rows(q[0, h].cpu(), k[0, h].cpu(), v[0, h].cpu(), do[0, h].cpu(), scale,
                                             True, q_rows=qr, k_rows=kr)
        qi, ki = torch.from_numpy(qr).to(DEV), torch.from_numpy(kr).to(DEV)
        g = (got[0][0, h].index_select(0, qi), got[1][0, h].index_select(0, ki), got[2][0, h].index_select(0, ki))
        assert_grads(g, ref, f"37 heads h={h}")


@pytest.mark.parametrize("causal", [True, False])
def test_backward_d64_long_sampled_rows(causal):
    """d = 64 (the dK/dV kernel in two 64-query halves per query tile) over N = 4093 with x8 key
    spikes and a ragged last tile: dQ at seeded query rows and dK, dV at seeded key rows (plus
    tile edges) of every head against the row-restricted fp64 oracle, fp32 and bf16 gradients."""
    B, H, N, d = 1, 3, 4093, 64
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=90 + causal, device=DEV, spike=True)
    do = inputs.normal_bf16((B, H, N, d), seed=91, device=DEV)
    scale = 1.0 / math.sqrt(d)
    grads = {fp32: run_bwd(q, k, v, do, scale, causal, grad_fp32=fp32) for fp32 in (True, False)}
    edge = [0, 63, 64, 127, 128, N - 62, N - 61, N - 1]
    for h in range(H):
        qr = np.unique(np.concatenate([inputs.sample_rows(N, 32, seed=200 + h).numpy(), edge]))
        kr = np.unique(np.concatenate([inputs.sample_rows(N, 32, seed=300 + h).numpy(), edge]))
        ref = oracle.attention_backward_rows(q[0, h].cpu(), k[0, h].cpu(), v[0, h].cpu(), do[0, h].cpu(), scale,
                                             causal, q_rows=qr, k_rows=kr)
        qi, ki = torch.from_numpy(qr).to(DEV), torch.from_numpy(kr).to(DEV)
        for fp32, (dq, dk, dv) in grads.items():
            got = (dq[0, h].index_select(0, qi), dk[0, h].index_select(0, ki), dv[0, h].index_select(0, ki))
            assert_grads(got, ref, f"d=64 N={N} causal={causal} h={h} grad_fp32={fp32}")
