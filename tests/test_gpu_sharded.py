"""GPU parity of the sequence-sharded prefill: fa_fwd_partial over each key shard, merged by
fa_combine, against the oracle (per-shard partials and the merged forward)."""

import math

import numpy as np
import pytest
import torch

import oracle
from _util import LSE_MAX, O_MAX, assert_parity, ensure_built
from exact_attention_06_gb300 import fattn, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def run_sharded(q, k, v, cuts, scale, causal, streams=False, o_fp32=False, views=False):
    """One fa_fwd_partial per shard [cuts[s], cuts[s+1]) (each shard its own K/V buffers, or with
    ``views`` the whole K/V tensors and the shard's key range), then fa_combine (fp32 or bf16 O);
    with ``streams`` every shard runs on its own stream.  Returns (o [B,H,N,d], lse, u, m, l)."""
    B, H, N, d = q.shape
    S = len(cuts) - 1
    R = B * H * N
    u = torch.full((R, S, d), float("nan"), dtype=torch.float32, device=DEV)
    m = torch.full((R, S), float("nan"), dtype=torch.float32, device=DEV)
    l = torch.full((R, S), float("nan"), dtype=torch.float32, device=DEV)
    ks = [k[:, :, cuts[s]:cuts[s + 1]].contiguous() for s in range(S)]
    vs = [v[:, :, cuts[s]:cuts[s + 1]].contiguous() for s in range(S)]
    main = torch.cuda.current_stream()
    side = [torch.cuda.Stream() for _ in range(S)] if streams else [main] * S
    for s in range(S):
        side[s].wait_stream(main)
        if views:
            fattn.fa_fwd_partial(q, k, v, u, m, l, scale, key_offset=cuts[s], shard=s, causal=causal, stream=side[s],
                                 nk=cuts[s + 1] - cuts[s])
        else:
            fattn.fa_fwd_partial(q, ks[s], vs[s], u, m, l, scale, key_offset=cuts[s], shard=s, causal=causal,
                                 stream=side[s])
        main.wait_stream(side[s])
    o = torch.empty((R, d), dtype=torch.float32 if o_fp32 else torch.bfloat16, device=DEV)
    lse = torch.empty(R, dtype=torch.float32, device=DEV)
    fattn.fa_combine(u, m, l, o, lse)
    fattn.fa_get_status()
    return o.view(B, H, N, d), lse.view(B, H, N), u, m, l


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,cuts", [(1000, [0, 300, 700, 1000]), (256, [0, 256]), (517, [0, 1, 129, 500, 517]),
                                    (2048, [0, 512, 1024, 1536, 2048])])
def test_sharded_prefill_matches_oracle(N, cuts, causal, d):
    B, H = 1, 2
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=N + d, device=DEV)
    scale = 1 / math.sqrt(d)
    o, lse, u, m, l = run_sharded(q, k, v, cuts, scale, causal, o_fp32=True)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, causal)
    assert_parity(o, lse, o_ref, lse_ref, f"merged N={N} cuts={cuts} fp32")
    ob, lseb = run_sharded(q, k, v, cuts, scale, causal)[:2]
    assert_parity(ob, lseb, o_ref, lse_ref, f"merged N={N} cuts={cuts} bf16")
    assert torch.equal(lse, lseb)
    # each shard's partial: m and l against the oracle's, and U / l (the shard-local O)
    S = len(cuts) - 1
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    for b in range(B):
        for h in range(H):
            r0 = (b * H + h) * N
            for s in range(S):
                ru, rm, rl = oracle.shard_partials_head(qc[b, h], kc[b, h, cuts[s]:cuts[s + 1]],
                                                        vc[b, h, cuts[s]:cuts[s + 1]], scale, causal, cuts[s])
                gm = m[r0:r0 + N, s].double().cpu().numpy()
                gl = l[r0:r0 + N, s].double().cpu().numpy()
                gu = u[r0:r0 + N, s].double().cpu().numpy()
                empty = np.isneginf(rm)
                assert np.all(np.isneginf(gm[empty])) and np.all(gl[empty] == 0)  # U slot left unwritten
                ok = ~empty
                if ok.any():
                    assert np.abs(gm[ok] - rm[ok]).max() <= LSE_MAX
                    assert np.abs(gl[ok] / rl[ok] - 1).max() <= 2e-3
                    e = np.abs(gu[ok] / gl[ok, None] - ru[ok] / rl[ok, None]).max()
                    assert e <= O_MAX, f"shard {s}: |U/l - U_ref/l_ref| = {e:.3e}"


def test_sharded_equals_unsharded_kernel_bitwise_lse_close():
    # one shard over all keys is the ordinary forward up to the final division
    B, H, N, d = 2, 4, 1536, 128
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=3, device=DEV)
    o, lse, *_ = run_sharded(q, k, v, [0, N], 1 / math.sqrt(d), True)
    o2 = torch.empty_like(q)
    lse2 = torch.empty(B, H, N, device=DEV)
    fattn.fa_fwd(q, k, v, o2, lse2, 1 / math.sqrt(d), True)
    fattn.fa_get_status()
    # at most one bf16 rounding step apart (U / l is formed in a different order)
    assert bool(((o.float() - o2.float()).abs() <= o2.float().abs() * 2 ** -7 + 1e-6).all())
    assert (lse - lse2).abs().max().item() <= 1e-5


def test_sharded_causal_workload_sampled_rows():
    # B2 H16 N8192 d128 causal with x8 key spikes, four 2048-key shards
    w = inputs.WORKLOADS["causal"]
    q, k, v = inputs.workload_inputs(w, seed=0, device=DEV)
    rows = inputs.sample_rows_per_head(w.B, w.H, w.N, 32, seed=7)
    from _util import gather_rows
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, True, rows=rows.numpy())
    for o_fp32 in (True, False):  # fp32 O: the raw bounds; bf16 O: after its own rounding
        o, lse, *_ = run_sharded(q, k, v, [0, 2048, 4096, 6144, 8192], w.scale, True, streams=True, o_fp32=o_fp32)
        assert_parity(gather_rows(o, rows), gather_rows(lse, rows), o_ref, lse_ref,
                      f"sharded causal workload o_fp32={o_fp32}")


def test_sharded_noncausal_d64_many_items_per_cta():
    # non-causal d = 64 shards run on the persistent kernel: B4 H16 N2048 is 512 blocks per shard
    # on at most 152 CTAs, so every CTA writes partials for several blocks in turn
    B, H, N, d = 4, 16, 2048, 64
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=11, device=DEV)
    o, lse, *_ = run_sharded(q, k, v, [0, 1000, 2048], 0.125, False, streams=True)
    rows = inputs.sample_rows_per_head(B, H, N, 24, seed=12)
    from _util import gather_rows
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), 0.125, False, rows=rows.numpy())
    # non-causal N=2048: every row averages 2048 keys, |O| is small and bf16 O meets the raw bounds
    assert_parity(gather_rows(o, rows), gather_rows(lse, rows), o_ref, lse_ref, "sharded d64 non-causal",
                  raw=True)


@pytest.mark.parametrize("d,causal", [(64, False), (64, True), (128, False), (128, True)])
def test_shards_read_from_the_whole_key_tensors(d, causal):
    """fa_fwd_partial_ex on the whole K/V tensors (each shard a key range, no copy) gives the
    partials of the per-shard buffers bit for bit, also where a shard's last key tile runs into
    the next shard's keys (cuts off the 128-key grid), and the merged forward matches the oracle."""
    B, H, N = 1, 3, 1000
    cuts = [0, 300, 701, 1000]
    q, k, v = inputs.prefill_inputs(B, H, N, d, seed=d + 5, device=DEV)
    scale = 1 / math.sqrt(d)
    o1, lse1, u1, m1, l1 = run_sharded(q, k, v, cuts, scale, causal, o_fp32=True)
    o2, lse2, u2, m2, l2 = run_sharded(q, k, v, cuts, scale, causal, o_fp32=True, views=True)
    assert torch.equal(m1, m2) and torch.equal(l1, l2)
    ne = ~torch.isneginf(m1)
    assert torch.equal(u1[ne], u2[ne])  # an empty partial's U is never written
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)
    o_ref, lse_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, causal)
    assert_parity(o2, lse2, o_ref, lse_ref, f"whole-tensor shards d={d} causal={causal}")
