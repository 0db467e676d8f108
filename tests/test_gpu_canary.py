"""Guard canaries: no kernel writes outside the buffers it is given.

Every output and workspace below is a view into a larger device buffer whose
leading and trailing 4 KiB hold a sentinel byte; after each call the sentinel
bytes must be unchanged.  The sizes are the ragged ones where an overrun would
come from: query counts that are not a multiple of the 128-row tile
(N = 16381, 129, 1), KV lengths that end inside a 64-key stage or a 128-key
chunk (L = 1, 129, 4103), one partial per chunk (splits = ceil(L / 128)), and
the key split of the forward's last round.  Each output is also checked
against the fp64 oracle (on sampled rows for the long workload), so the
buffers are known to be fully written, not merely untouched outside.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from _util import assert_parity, ensure_built, gather_rows
from exact_attention_06_gb300 import fattn, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
SENTINEL = 0xA5
PAD = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


class Guarded:
    """A tensor of `shape` and `dtype` in the middle of a byte buffer padded by PAD sentinel bytes on
    each side; the tensor's own bytes start as the sentinel too."""

    def __init__(self, shape, dtype):
        self.nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((2 * PAD + self.nbytes,), SENTINEL, dtype=torch.uint8, device=DEV)
        self.t = self.buf[PAD:PAD + self.nbytes].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        head = self.buf[:PAD]
        tail = self.buf[PAD + self.nbytes:]
        assert bool((head == SENTINEL).all()), f"{what}: bytes before the buffer were written"
        assert bool((tail == SENTINEL).all()), f"{what}: bytes after the buffer were written"


def guarded_ws(nbytes):
    return Guarded((max(int(nbytes), 256),), torch.uint8)


@pytest.mark.parametrize("d,causal", [(64, False), (64, True), (128, False), (128, True)])
@pytest.mark.parametrize("N", [1, 129])
@pytest.mark.parametrize("o_fp32", [False, True])
def test_forward_small_ragged(N, d, causal, o_fp32):
    B, H = 2, 3
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=N + d, device=DEV)
    scale = 1 / math.sqrt(d)
    o = Guarded((B, H, N, d), torch.float32 if o_fp32 else torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    fattn.fa_fwd_ex(q, k, v, o.t, lse.t, scale, causal)
    fattn.fa_get_status()
    o.check("O")
    lse.check("lse")
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, causal)
    assert_parity(o.t, lse.t, o_ref, lse_ref, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("o_fp32", [False, True])
def test_forward_ragged_workload_16381(o_fp32):
    w = inputs.WORKLOADS["ragged"]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    o = Guarded((w.B, w.H, w.N, w.d), torch.float32 if o_fp32 else torch.bfloat16)
    lse = Guarded((w.B, w.H, w.N), torch.float32)
    fattn.fa_fwd_ex(q, k, v, o.t, lse.t, w.scale, True)
    fattn.fa_get_status()
    o.check("O")
    lse.check("lse")
    # the last tile's rows (16256 .. 16380) and a few others, on 4 heads
    rows = torch.tensor([0, 127, 128, 16255, 16256, 16300, 16379, 16380]).expand(w.B, 4, -1)
    o_ref, lse_ref = oracle.attention(q[:, :4].cpu(), k[:, :4].cpu(), v[:, :4].cpu(), w.scale, True,
                                      rows=rows.numpy())
    assert_parity(gather_rows(o.t[:, :4], rows), gather_rows(lse.t[:, :4], rows), o_ref, lse_ref, "ragged 16381")


@pytest.mark.parametrize("B,H,N", [(1, 1, 1024), (1, 4, 2048), (1, 1, 1000)])
def test_forward_key_split_workspace(B, H, N):
    d = 64
    nbytes = fattn.fa_fwd_workspace_bytes(B, H, N, d, False)
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=B * H + N, device=DEV)
    ws = guarded_ws(nbytes)
    o = Guarded((B, H, N, d), torch.bfloat16)
    lse = Guarded((B, H, N), torch.float32)
    fattn.fa_fwd_ex(q, k, v, o.t, lse.t, 0.125, False, workspace=ws.t if nbytes else None)
    fattn.fa_get_status()
    for g, name in ((ws, "key-split workspace"), (o, "O"), (lse, "lse")):
        g.check(name)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), 0.125, False)
    assert_parity(o.t, lse.t, o_ref, lse_ref, f"key split B{B} H{H} N{N}", raw=True)


@pytest.mark.parametrize("L", [1, 129, 4103])
@pytest.mark.parametrize("d", [64, 128])
def test_decode(L, d):
    B, H = 2, 3
    q, k, v = inputs.decode_inputs(B, H, L, d, seed=L + d, device=DEV)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.decode(q.cpu(), k.cpu(), v.cpu(), scale)
    for splits in sorted({0, -(-L // 128)}):
        ws = guarded_ws(fattn.fa_decode_workspace_bytes(B, H, L, d, 128, splits))
        for dt in (torch.bfloat16, torch.float32):
            o = Guarded((B, H, d), dt)
            lse = Guarded((B, H), torch.float32)
            fattn.fa_decode_splitkv(q, k, v, o.t, lse.t, scale, ws.t, 128, splits)
            fattn.fa_get_status()
            for g, name in ((ws, "decode workspace"), (o, "O"), (lse, "lse")):
                g.check(f"{name} L={L} splits={splits}")
            assert_parity(o.t.reshape(B * H, d), lse.t.reshape(B * H), o_ref, lse_ref, f"L={L} splits={splits}")


@pytest.mark.parametrize("L", [1, 129, 4103])
def test_paged_decode(L):
    B, H, d, ps = 2, 2, 128, 64
    n = -(-L // ps)
    q, k, v = inputs.decode_inputs(B, H, n * ps, d, seed=L, device=DEV)
    kp = k.view(B, H, n, ps, d).permute(0, 2, 1, 3, 4).reshape(B * n, H, ps, d).contiguous()
    vp = v.view(B, H, n, ps, d).permute(0, 2, 1, 3, 4).reshape(B * n, H, ps, d).contiguous()
    table = torch.arange(B * n, dtype=torch.int32, device=DEV).view(B, n)
    lens = torch.full((B,), L, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle.decode(q.cpu(), k[:, :, :L].cpu(), v[:, :, :L].cpu(), scale)
    for splits in sorted({0, -(-L // 128)}):
        ws = guarded_ws(fattn.fa_decode_paged_workspace_bytes(B, H, L, d, ps, n, splits))
        o = Guarded((B, H, d), torch.float32)
        lse = Guarded((B, H), torch.float32)
        fattn.fa_decode_paged(q, kp, vp, table, lens, o.t, lse.t, scale, L, workspace=ws.t, splits=splits)
        fattn.fa_get_status()
        for g, name in ((ws, "paged workspace"), (o, "O"), (lse, "lse")):
            g.check(f"{name} L={L} splits={splits}")
        assert_parity(o.t.reshape(B * H, d), lse.t.reshape(B * H), o_ref, lse_ref, f"paged L={L} splits={splits}")


@pytest.mark.parametrize("N,cuts", [(129, [0, 1, 129]), (1, [0, 1])])
@pytest.mark.parametrize("d", [64, 128])
def test_sharded_partials_and_combine(N, cuts, d):
    B, H, causal = 1, 2, True
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=7 * N + d, device=DEV)
    scale = 1 / math.sqrt(d)
    S, R = len(cuts) - 1, B * H * N
    u = Guarded((R, S, d), torch.float32)
    m = Guarded((R, S), torch.float32)
    l = Guarded((R, S), torch.float32)
    for s in range(S):
        ks = k[:, :, cuts[s]:cuts[s + 1]].contiguous()
        vs = v[:, :, cuts[s]:cuts[s + 1]].contiguous()
        fattn.fa_fwd_partial(q, ks, vs, u.t, m.t, l.t, scale, cuts[s], s, causal)
    fattn.fa_get_status()
    for g, name in ((u, "u_part"), (m, "m_part"), (l, "l_part")):
        g.check(name)
    o = Guarded((R, d), torch.float32)
    lse = Guarded((R,), torch.float32)
    fattn.fa_combine(u.t, m.t, l.t, o.t, lse.t)
    fattn.fa_get_status()
    o.check("combined O")
    lse.check("combined lse")
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, causal)
    assert_parity(o.t.view(B, H, N, d), lse.t.view(B, H, N), o_ref, lse_ref, f"sharded N={N}")


@pytest.mark.parametrize("N", [1, 129])
@pytest.mark.parametrize("d", [64, 128])
def test_backward(N, d):
    B, H, causal = 1, 2, True
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=3 * N + d, device=DEV)
    do = inputs.normal_bf16((B, H, N, d), seed=N + 5, device=DEV)
    scale = 1 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    fattn.fa_fwd(q, k, v, o, lse, scale, causal)
    ws = guarded_ws(fattn.fa_bwd_workspace_bytes(B, H, N))
    for dt in (torch.bfloat16, torch.float32):
        grads = [Guarded((B, H, N, d), dt) for _ in range(3)]
        fattn.fa_bwd(q, k, v, o, do, lse, *(g.t for g in grads), scale, causal, workspace=ws.t)
        fattn.fa_get_status()
        ws.check("backward workspace")
        for g, name in zip(grads, ("dq", "dk", "dv")):
            g.check(f"{name} {dt}")
        ref = oracle.attention_backward(q.cpu(), k.cpu(), v.cpu(), do.cpu(), scale, causal)
        for g, r, name in zip(grads, ref, ("dq", "dk", "dv")):
            e = np.abs(g.t.double().cpu().numpy() - r)
            assert e.max() <= 2e-2 * max(np.abs(r).max(), 1e-6) + 1e-6, f"{name} N={N} {dt}"


@pytest.mark.parametrize("N", [1, 129])
def test_fp8_quantize_and_forward(N):
    B, H, d = 1, 2, 128
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=N + 11, device=DEV)
    nb = -(-N // 128)
    packed = []
    for x in (q, k, v):
        codes = Guarded((B, H, N, d), torch.uint8)
        scales = Guarded((B, H, nb), torch.float32)
        fattn.fa_quantize_e4m3(x, codes.t, scales.t)
        fattn.fa_get_status()
        codes.check("E4M3 codes")
        scales.check("block scales")
        c_ref, s_ref = oracle.quantize_e4m3_blocks(x.cpu())
        assert np.array_equal(codes.t.cpu().numpy(), c_ref)
        packed += [codes.t, scales.t]
    q8, sq, k8, sk, v8, sv = packed
    o = Guarded((B, H, N, d), torch.float32)
    lse = Guarded((B, H, N), torch.float32)
    fattn.fa_fwd_fp8(q8, k8, v8, sq, sk, sv, o.t, lse.t, 1 / math.sqrt(d), True)
    fattn.fa_get_status()
    o.check("FP8 O")
    lse.check("FP8 lse")
    o_ref, lse_ref = oracle.attention_fp8(q8.cpu(), sq.cpu(), k8.cpu(), sk.cpu(), v8.cpu(), sv.cpu(),
                                          1 / math.sqrt(d), True)
    err = np.abs(o.t.double().cpu().numpy() - o_ref)
    assert err.max() <= 0.35 and np.abs(lse.t.double().cpu().numpy() - lse_ref).max() <= 1e-3
