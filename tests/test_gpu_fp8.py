"""GPU parity of the FP8 path: the E4M3 block quantizer (byte-exact) and the FP8
forward (fa_fwd_fp8) against the oracle's FP8 forward.

Tolerance of the FP8 forward.  The oracle models every quantization the kernel
makes (Q, K, V codes; P~ codes), so what remains is fp32 arithmetic plus the
rare P~ code that lands on the other side of a rounding midpoint: the kernel's
p (fp32 scores from the tensor core, ex2.approx) differs from the oracle's by a
relative 2^-10 at most (S accumulated in fp32 over 128 products: |dS| <=
128 * 2^-24 * sum|q k|, under 1e-3 in log2 units for these inputs; ex2.approx
adds about 2^-22), so a code may differ from the oracle's only when the
oracle's fp32 value x has round(x (1 - 2^-10)) != round(x (1 + 2^-10)), and then
by at most that spacing.  Per row the bound is therefore

    |O - O_ref| <= 2e-5 (1 + max|O_ref|) + sum_k spacing_k * max|V8_k| * e^(m_k - m) * max(s_v) / 256 / l

over the ambiguous keys k (m_k: running max when key k was quantized), plus
half a bf16 ulp for bf16 O.  lse has the bf16 path's bound (it uses the
unquantized p).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from _util import LSE_MAX, bf16_half_ulp, ensure_built

pytestmark = pytest.mark.gpu

DELTA = 2.0 ** -10     # relative difference of the kernel's p from the oracle's fp32 p
ATOL_FP32 = 2e-5       # fp32 accumulation of S, l and U (no code flips)


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _quant_gpu(x):
    from exact_attention_06_gb300 import fattn
    B, H, N, d = x.shape
    codes = torch.full(x.shape, 0x7F, dtype=torch.uint8, device=x.device)
    sc = torch.full((B, H, (N + 127) // 128), float("nan"), dtype=torch.float32, device=x.device)
    fattn.fa_quantize_e4m3(x, codes, sc)
    fattn.fa_get_status()
    return codes, sc


@pytest.mark.parametrize("shape", [(1, 2, 300, 128), (2, 3, 1000, 64), (1, 1, 128, 128), (1, 1, 1, 64),
                                   (1, 2, 129, 128)])
def test_quantizer_is_byte_exact(shape):
    from exact_attention_06_gb300 import inputs
    x = inputs.normal_bf16(shape, seed=sum(shape), device="cuda")
    x[..., ::37, :] *= 100.0              # large blocks next to ordinary ones
    x[..., 5::41, 3] = -0.0               # negative zeros keep their sign bit
    x[..., 7::53, :] *= 1e-6              # values that round into the subnormal range
    if shape[2] > 200:
        x[0, 0, 128:256] = 0.0            # an all-zero block: scale 1
    codes, sc = _quant_gpu(x)
    rc, rs = oracle.quantize_e4m3_blocks(x.cpu().float())
    np.testing.assert_array_equal(sc.cpu().numpy(), rs)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)


def test_quantizer_full_size_sampled_heads():
    # the causal workload's K (B2 H16 N8192 d128, x8 spikes); quantization is per head, so
    # the oracle checks a few whole heads and every block scale
    from exact_attention_06_gb300 import inputs
    w = inputs.WORKLOADS["causal"]
    _, k, _ = inputs.workload_inputs(w, seed=0, device="cuda")
    codes, sc = _quant_gpu(k)
    kc = k.cpu().float()
    amax = kc.abs().reshape(w.B, w.H, w.N // 128, -1).amax(dim=-1).numpy()
    np.testing.assert_array_equal(sc.cpu().numpy(), np.where(amax > 0, (amax / np.float32(448.0)), 1.0)
                                  .astype(np.float32))
    for b, h in ((0, 0), (1, 15), (0, 7)):
        rc, rs = oracle.quantize_e4m3_blocks(kc[b:b + 1, h:h + 1])
        np.testing.assert_array_equal(codes[b, h].cpu().numpy(), rc[0, 0])
        np.testing.assert_array_equal(sc[b, h].cpu().numpy(), rs[0, 0])


def _flip_budget(trace, lse_ref, v8_head, sv_max):
    """Per-row bound on |O - O_ref| from P~ codes that may round the other way (module docstring)."""
    vals = oracle.e4m3_values()
    vmax = np.abs(vals[v8_head.astype(np.int64)]).max(axis=1)
    m_fin = trace[-1]["m"]
    acc = np.zeros_like(m_fin)
    for tr in trace:
        x = tr["x"].astype(np.float64)
        lo = oracle.round_to_e4m3(x * (1 - DELTA)).astype(np.int64)
        hi = oracle.round_to_e4m3(x * (1 + DELTA)).astype(np.int64)
        gap = np.where(lo != hi, np.abs(vals[hi] - vals[lo]), 0.0)
        w = np.where(np.isneginf(tr["m"]), 0.0, np.exp(tr["m"] - np.where(np.isneginf(m_fin), 0.0, m_fin)))
        acc += (gap @ vmax[tr["cols"]]) * w
    l_fin = np.exp(lse_ref - m_fin)
    return np.where(np.isfinite(lse_ref), acc * float(sv_max) / 256.0 / np.where(l_fin > 0, l_fin, 1.0), 0.0)


def _run_and_check(q, k, v, scale, causal, rows_per_head=None, seed=0):
    from exact_attention_06_gb300 import fattn, inputs
    B, H, N, d = q.shape
    (q8, sq), (k8, sk), (v8, sv) = _quant_gpu(q), _quant_gpu(k), _quant_gpu(v)
    o32 = torch.full((B, H, N, d), float("nan"), dtype=torch.float32, device=q.device)
    o16 = torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16, device=q.device)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    lse16 = torch.full_like(lse, float("nan"))
    fattn.fa_fwd_fp8(q8, k8, v8, sq, sk, sv, o32, lse, scale, causal)
    fattn.fa_fwd_fp8(q8, k8, v8, sq, sk, sv, o16, lse16, scale, causal)
    fattn.fa_get_status()
    assert torch.equal(lse, lse16)
    # the oracle quantizes the bf16 inputs itself (the GPU codes are checked byte-exact above)
    cpu = [t.cpu() for t in (q8, sq, k8, sk, v8, sv)]
    rows = None if rows_per_head is None else inputs.sample_rows_per_head(B, H, N, rows_per_head, seed).numpy()
    worst = []
    for b in range(B):
        for h in range(H):
            sel = np.arange(N) if rows is None else rows[b, h]
            a = [cpu[i][b, h].numpy() for i in range(6)]
            trace = []
            ro, rl = oracle.attention_fp8_head(*a, scale, causal, rows=sel, trace=trace)
            budget = _flip_budget(trace, rl, a[4], a[5].max())
            g32 = o32[b, h].index_select(0, torch.from_numpy(sel).to(q.device)).double().cpu().numpy()
            g16 = o16[b, h].index_select(0, torch.from_numpy(sel).to(q.device)).double().cpu().numpy()
            gl = lse[b, h].index_select(0, torch.from_numpy(sel).to(q.device)).double().cpu().numpy()
            assert np.all(np.isfinite(g32)) and np.all(np.isfinite(g16))
            tol = ATOL_FP32 * (1 + np.abs(ro).max(axis=1)) + budget
            e32 = np.abs(g32 - ro).max(axis=1)
            assert np.all(e32 <= tol), f"b{b} h{h}: fp32 O row error {e32.max():.3e} above its bound"
            e16 = np.maximum(np.abs(g16 - ro) - bf16_half_ulp(np.maximum(np.abs(g16), np.abs(ro))), 0).max(axis=1)
            assert np.all(e16 <= tol), f"b{b} h{h}: bf16 O row error {e16.max():.3e} above its bound"
            fin = np.isfinite(rl)
            assert np.all(np.isneginf(gl[~fin]))
            if fin.any():
                assert np.abs(gl[fin] - rl[fin]).max() <= LSE_MAX
            worst.append(np.median(e32))
    # most rows see no flip at all: their error is fp32 rounding only
    assert float(np.median(worst)) <= 1e-5


@pytest.mark.parametrize("N,causal", [(300, False), (300, True), (129, True), (1, False), (1000, True),
                                      (2048, False)])
def test_fp8_forward_small(N, causal):
    from exact_attention_06_gb300 import inputs
    B, H, d = (1, 2, 128) if N != 1000 else (2, 3, 128)
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=N + 17, device="cuda")
    _run_and_check(q, k, v, 1 / math.sqrt(d), causal)


def test_fp8_forward_causal_workload_sampled_rows():
    # B2 H16 N8192 d128 causal with x8 key spikes: the launch configuration the bench times
    from exact_attention_06_gb300 import inputs
    w = inputs.WORKLOADS["causal"]
    q, k, v = inputs.workload_inputs(w, seed=0, device="cuda")
    _run_and_check(q, k, v, w.scale, True, rows_per_head=24, seed=5)


def test_fp8_forward_ragged_sampled_rows():
    # N = 16381 (a ragged last tile of 125 rows), causal, all 32 heads
    from exact_attention_06_gb300 import inputs
    w = inputs.WORKLOADS["ragged"]
    q, k, v = inputs.workload_inputs(w, seed=0, device="cuda")
    _run_and_check(q, k, v, w.scale, True, rows_per_head=8, seed=6)


def test_fp8_forward_long_noncausal_sampled_rows():
    # N = 8189 non-causal with x8 key spikes: every block scans all 64 key tiles, the last ragged
    from exact_attention_06_gb300 import inputs
    q, k, v = inputs.prefill_inputs(1, 3, 8189, 128, seed=81, device="cuda", spike=True)
    _run_and_check(q, k, v, 1 / math.sqrt(128), False, rows_per_head=16, seed=7)


def test_fp8_rejects_d64_on_device():
    from exact_attention_06_gb300 import fattn
    x = torch.zeros(1, 1, 128, 64, dtype=torch.uint8, device="cuda")
    s = torch.ones(1, 1, 1, device="cuda")
    o = torch.empty(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 1, 128, device="cuda")
    with pytest.raises(fattn.FattnError) as ei:
        fattn.fa_fwd_fp8(x, x, x, s, s, s, o, lse, 0.125)
    assert ei.value.status == fattn.FA_ERR_UNSUPPORTED
