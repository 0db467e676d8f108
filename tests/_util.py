"""Shared helpers of the GPU parity tests: run the library, compare with the oracle."""

from __future__ import annotations

import numpy as np
import torch

# Tolerances for bf16 inputs with fp32 accumulation, against the fp64 oracle.
O_MAX = 1e-2
O_MEAN = 1e-3
LSE_MAX = 1e-3


def ensure_built():
    from exact_attention_06_gb300 import build
    return build.build()


def run_fwd(q, k, v, scale, causal, o_fp32=False):
    from exact_attention_06_gb300 import fattn
    B, H, N, d = q.shape
    o = torch.full((B, H, N, d), float("nan"), dtype=torch.float32 if o_fp32 else torch.bfloat16, device=q.device)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=q.device)
    fattn.fa_fwd_ex(q, k, v, o, lse, scale, causal, o_fp32=o_fp32)
    fattn.fa_get_status()
    return o, lse


def gather_rows(t, rows):
    """t [B, H, N, ...] on any device, rows [B, H, R] (CPU long) -> CPU tensor [B, H, R, ...]."""
    B, H = t.shape[0], t.shape[1]
    out = []
    for b in range(B):
        out.append(torch.stack([t[b, h].index_select(0, rows[b, h].to(t.device)).cpu() for h in range(H)]))
    return torch.stack(out)


def errors(o, lse, o_ref, lse_ref):
    o = o.detach().cpu().double().numpy() if hasattr(o, "detach") else np.asarray(o, dtype=np.float64)
    lse = lse.detach().cpu().double().numpy() if hasattr(lse, "detach") else np.asarray(lse, dtype=np.float64)
    e = np.abs(o - o_ref)
    le = np.abs(lse - lse_ref)
    return float(e.max()), float(e.mean()), float(le.max())


def bf16_half_ulp(x):
    """Half the bf16 spacing at |x| (8 significant bits): the rounding a bf16 output cannot avoid."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 8), 0.0)


def assert_parity(o, lse, o_ref, lse_ref, what="", raw=False):
    """The bounds max|O - O_ref| <= 1e-2, mean <= 1e-3, max|lse - lse_ref| <= 1e-3.

    fp32 O: applied to |O - O_ref| as it is.  bf16 O with ``raw``: applied as
    it is too (used where |O| is small enough that bf16's own rounding stays
    well inside the bounds, e.g. decode over long caches, |O| ~ 0.03).  bf16 O
    without ``raw``: applied to what remains after the output's own
    round-to-nearest (half a bf16 ulp), i.e. O must be the bf16 rounding of a
    value that meets the bounds; every such check has an fp32-O twin that is
    held to the raw bounds."""
    is_bf16 = getattr(o, "dtype", None) == torch.bfloat16 and not raw
    o_np = o.detach().cpu().double().numpy()
    lse_np = lse.detach().cpu().double().numpy()
    assert np.all(np.isfinite(o_np)), f"{what}: non-finite O"
    assert np.all(np.isfinite(lse_np) | np.isneginf(lse_ref)), f"{what}: non-finite lse"
    e = np.abs(o_np - o_ref)
    if is_bf16:
        e = np.maximum(e - bf16_half_ulp(np.maximum(np.abs(o_np), np.abs(o_ref))), 0.0)
    emax, emean = float(e.max()), float(e.mean())
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(lse_np[~fin])), f"{what}: lse of an empty row must be -inf"
    lmax = float(np.abs(lse_np[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    tag = " (after bf16 output rounding)" if is_bf16 else ""
    assert emax <= O_MAX, f"{what}: max|O-O_ref|{tag} = {emax:.3e} > {O_MAX}"
    assert emean <= O_MEAN, f"{what}: mean|O-O_ref|{tag} = {emean:.3e} > {O_MEAN}"
    assert lmax <= LSE_MAX, f"{what}: max|lse-lse_ref| = {lmax:.3e} > {LSE_MAX}"
    return emax, emean, lmax
