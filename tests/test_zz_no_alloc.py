"""fa_decode_splitkv_noalloc: the decode entry point for callers that cannot allocate.

Plugins inside inference runtimes are often given only their input and output
buffers, and request paths may not call cudaMalloc/cudaFree (both can stall the
device and may fail mid-request).  This entry point keeps the split partials in
a fixed device array inside the library instead of a caller workspace.  Here it
is called through the C ABI, on two calls in a row, and compared with
fa_decode_splitkv given a torch-allocated workspace and with the fp64 oracle.
The file name makes pytest collect it last.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from _util import O_MAX, O_MEAN, LSE_MAX, assert_parity, ensure_built
from exact_attention_06_gb300 import fattn, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _noalloc(lib, q, k, v, o, lse, scale, splits):
    B, H, L, d = k.shape
    vp = ctypes.c_void_p
    return lib.fa_decode_splitkv_noalloc(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()),
                                         vp(lse.data_ptr()), B, H, L, d, ctypes.c_float(scale), 128, splits,
                                         vp(torch.cuda.current_stream().cuda_stream))


def _with_workspace(q, k, v, scale, splits):
    B, H, L, d = k.shape
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, H, dtype=torch.float32, device=DEV)
    ws = torch.empty(fattn.fa_decode_workspace_bytes(B, H, L, d, 128, splits), dtype=torch.uint8, device=DEV)
    fattn.fa_decode_splitkv(q, k, v, o, lse, scale, ws, 128, splits)
    return o, lse


def _oracle_pairs(q, k, v, scale, pairs):
    d = q.shape[-1]
    o_ref = np.zeros((len(pairs), d))
    lse_ref = np.zeros(len(pairs))
    for n, (b, h) in enumerate(pairs):
        o_r, l_r = oracle.decode(q[b:b + 1, h:h + 1].cpu(), k[b:b + 1, h:h + 1].cpu(), v[b:b + 1, h:h + 1].cpu(),
                                 scale)
        o_ref[n], lse_ref[n] = o_r[0], l_r[0]
    return o_ref, lse_ref


def _check(o, lse, q, k, v, scale, splits, what, pairs=None):
    B, H = q.shape[0], q.shape[1]
    pairs = pairs or [(b, h) for b in range(B) for h in range(H)]
    o_ref, lse_ref = _oracle_pairs(q, k, v, scale, pairs)
    got_o = torch.stack([o[b, h] for b, h in pairs])
    got_l = torch.stack([lse[b, h] for b, h in pairs])
    assert_parity(got_o, got_l, o_ref, lse_ref, f"{what} against the oracle", raw=True)
    o_ws, lse_ws = _with_workspace(q, k, v, scale, splits)
    assert fattn.fa_get_status() == fattn.FA_OK
    err = (o.double() - o_ws.double()).abs()
    assert float(err.max()) <= O_MAX and float(err.mean()) <= O_MEAN, what
    assert float((lse.double() - lse_ws.double()).abs().max()) <= LSE_MAX, what


def test_noalloc_decode_matches_the_oracle_and_the_workspace_entry_point_twice():
    ensure_built()
    lib = fattn.lib()
    cases = [(4, 8, 3000, 128, 0, 11), (2, 16, 1000, 64, 3, 12)]  # two different calls in a row
    for B, H, L, d, splits, seed in cases:
        q, k, v = inputs.decode_inputs(B, H, L, d, seed=seed, device=DEV)
        scale = 1.0 / math.sqrt(d)
        o = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
        st = _noalloc(lib, q, k, v, o, lse, scale, splits)
        assert st == fattn.FA_OK, fattn.fa_last_error()
        assert fattn.fa_get_status() == fattn.FA_OK
        _check(o, lse, q, k, v, scale, splits, f"B{B} H{H} L{L} d{d} splits={splits}")


def test_noalloc_automatic_splits_shrink_to_fit_the_scratch():
    """splits = 0 where the automatic plan's partials exceed the fixed scratch: the entry point takes
    the largest smaller split count that fits instead of refusing."""
    ensure_built()
    lib = fattn.lib()
    L, d, H = 256, 128, 8
    cap = fattn.FA_NOALLOC_SCRATCH_BYTES
    found = None
    for B in range(1000, 2000):
        if (fattn.fa_decode_workspace_bytes(B, H, L, d, 128, 0) > cap >=
                fattn.fa_decode_workspace_bytes(B, H, L, d, 128, 1)):
            found = B
            break
    assert found is not None, "no batch size in range whose automatic plan exceeds the scratch"
    B = found
    q, k, v = inputs.decode_inputs(B, H, L, d, seed=5, device=DEV)
    scale = 1.0 / math.sqrt(d)
    o = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
    st = _noalloc(lib, q, k, v, o, lse, scale, 0)
    assert st == fattn.FA_OK, fattn.fa_last_error()
    assert fattn.fa_get_status() == fattn.FA_OK
    pairs = [(int(i) // H, int(i) % H) for i in inputs.sample_rows(B * H, 64, seed=6)]
    _check(o, lse, q, k, v, scale, 1, f"B{B} H{H} L{L} automatic splits", pairs=pairs)
    # an explicit split count that does not fit is still refused
    assert _noalloc(lib, q, k, v, o, lse, scale, 2) == fattn.FA_ERR_WORKSPACE
    assert "fixed scratch" in fattn.fa_last_error()


def test_noalloc_rejects_requests_beyond_its_scratch():
    ensure_built()
    lib = fattn.lib()
    B, H, L, d = 64, 32, 4096, 128  # 2048 rows x 8 splits need a little over 8 MiB
    q = torch.zeros(B, H, d, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(B, H, L, d, dtype=torch.bfloat16, device=DEV)
    o = torch.zeros(B, H, d, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(B, H, dtype=torch.float32, device=DEV)
    assert fattn.fa_decode_workspace_bytes(B, H, L, d, 128, 8) > fattn.FA_NOALLOC_SCRATCH_BYTES
    st = _noalloc(lib, q, k, k, o, lse, 0.1, 8)
    assert st == fattn.FA_ERR_WORKSPACE
    assert "fixed scratch" in fattn.fa_last_error()
    assert fattn.fa_decode_workspace_bytes(B, H, L, d, 128, 7) <= fattn.FA_NOALLOC_SCRATCH_BYTES
    assert _noalloc(lib, q, k, k, o, lse, 0.1, 7) == fattn.FA_OK
    assert fattn.fa_get_status() == fattn.FA_OK
