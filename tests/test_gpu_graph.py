"""The library's calls can be captured in a CUDA graph and replayed.

Serving code captures its per-token decode (and often the prefill) in CUDA graphs so that the
host does not launch each kernel again.  Every entry point here only enqueues work on the given
stream (no synchronisation, no allocation), so a capture of a causal forward, a split-KV decode
and a paged decode replays as the same launches: the graph is replayed on new input values
written into the captured buffers and checked against the fp64 oracle each time.
"""

import math

import pytest
import torch

import oracle
from _util import assert_parity, ensure_built
from exact_attention_06_gb300 import fattn, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


def test_forward_and_decodes_replay_from_a_cuda_graph():
    ensure_built()
    B, H, N, d, L, ps = 1, 4, 700, 128, 1500, 64
    scale = 1.0 / math.sqrt(d)
    q = torch.empty(B, H, N, d, dtype=torch.bfloat16, device=DEV)
    k, v = torch.empty_like(q), torch.empty_like(q)
    o = torch.empty(B, H, N, d, dtype=torch.float32, device=DEV)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    dq = torch.empty(2, H, d, dtype=torch.bfloat16, device=DEV)
    dk = torch.empty(2, H, L, d, dtype=torch.bfloat16, device=DEV)
    dv = torch.empty_like(dk)
    do = torch.empty(2, H, d, dtype=torch.float32, device=DEV)
    dl = torch.empty(2, H, dtype=torch.float32, device=DEV)
    ws = torch.empty(fattn.fa_decode_workspace_bytes(2, H, L, d, 128, 0), dtype=torch.uint8, device=DEV)
    n_pages = -(-L // ps)
    kp = torch.empty(2 * n_pages, H, ps, d, dtype=torch.bfloat16, device=DEV)
    vp = torch.empty_like(kp)
    table = torch.arange(2 * n_pages, dtype=torch.int32, device=DEV).view(2, n_pages).flip(1).contiguous()
    lens = torch.tensor([L, L - 333], dtype=torch.int32, device=DEV)
    po = torch.empty(2, H, d, dtype=torch.float32, device=DEV)
    pl = torch.empty(2, H, dtype=torch.float32, device=DEV)
    pws = torch.empty(fattn.fa_decode_paged_workspace_bytes(2, H, L, d, ps, n_pages, 0), dtype=torch.uint8,
                      device=DEV)

    def fill(seed):
        a, b, c = inputs.prefill_inputs(B, H, N, d, seed=seed, device=DEV, spike=True)
        q.copy_(a), k.copy_(b), v.copy_(c)
        x, y, z = inputs.decode_inputs(2, H, L, d, seed=seed + 7, device=DEV)
        dq.copy_(x), dk.copy_(y), dv.copy_(z)
        # page table[b, i] holds keys i*ps .. of sequence b for every head (pages laid out in reverse)
        pad = n_pages * ps - L
        for src, pool in ((dk, kp), (dv, vp)):
            full = torch.nn.functional.pad(src, (0, 0, 0, pad))
            pages = full.view(2, H, n_pages, ps, d).permute(0, 2, 1, 3, 4)
            pool[table.view(-1).long()] = pages.reshape(2 * n_pages, H, ps, d)

    def step(stream):
        fattn.fa_fwd_ex(q, k, v, o, lse, scale, True, stream=stream)
        fattn.fa_decode_splitkv(dq, dk, dv, do, dl, scale, ws, 128, 0, stream=stream)
        fattn.fa_decode_paged(dq, kp, vp, table, lens, po, pl, scale, L, workspace=pws, stream=stream)

    fill(1)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # one call outside the capture (warm-up, as torch recommends)
        step(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    for seed in (11, 12):
        fill(seed)
        o.fill_(float("nan")), do.fill_(float("nan")), po.fill_(float("nan"))
        g.replay()
        assert fattn.fa_get_status() == fattn.FA_OK
        rows = inputs.sample_rows(N, 96, seed=seed).numpy()
        o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, True, rows=rows)
        r = torch.from_numpy(rows).to(DEV)
        assert_parity(o[:, :, r], lse[:, :, r], o_ref, lse_ref, f"graph forward seed={seed}")
        d_ref, dl_ref = oracle.decode(dq.cpu(), dk.cpu(), dv.cpu(), scale)
        assert_parity(do.reshape(-1, d), dl.reshape(-1), d_ref, dl_ref, f"graph decode seed={seed}")
        p_ref, pl_ref = oracle.decode_paged(dq.cpu(), kp.cpu(), vp.cpu(), table.cpu().numpy(), lens.cpu().numpy(),
                                            scale)
        assert_parity(po.reshape(-1, d), pl.reshape(-1), p_ref, pl_ref, f"graph paged decode seed={seed}")
