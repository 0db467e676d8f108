"""Host-side checks of the seeded input generators (no attention arithmetic here)."""

import torch

from exact_attention_06_gb300 import inputs


def test_seeded_and_bf16():
    a = inputs.normal_bf16((3, 5, 7), 11)
    b = inputs.normal_bf16((3, 5, 7), 11)
    c = inputs.normal_bf16((3, 5, 7), 12)
    assert a.dtype == torch.bfloat16
    assert torch.equal(a, b) and not torch.equal(a, c)


def test_slabbed_draw_is_deterministic(monkeypatch):
    monkeypatch.setattr(inputs, "SLAB_ELEMS", 333)
    a = inputs.normal_bf16((4, 1000), 3)
    b = inputs.normal_bf16((4, 1000), 3)
    assert torch.equal(a, b) and a.float().std() > 0.9


def test_spike_rows_are_exact_times_eight():
    q, k, v = inputs.prefill_inputs(1, 2, 300, 8, seed=0, spike=False)
    _, k2, _ = inputs.prefill_inputs(1, 2, 300, 8, seed=0, spike=True)
    rows = torch.arange(300)
    hit = (rows % 64) == 63
    assert hit.sum() == 4
    assert torch.equal(k2[:, :, hit].float(), k[:, :, hit].float() * 8)
    assert torch.equal(k2[:, :, ~hit], k[:, :, ~hit])


def test_sample_rows():
    r = inputs.sample_rows(16381, 512, 3)
    assert r.numel() == 512 and torch.all(r[1:] > r[:-1]) and int(r.max()) < 16381
    assert torch.equal(inputs.sample_rows(10, 512, 3), torch.arange(10))
    per = inputs.sample_rows_per_head(1, 3, 1000, 16, 0)
    assert per.shape == (1, 3, 16) and not torch.equal(per[0, 0], per[0, 1])


def test_workload_sizes_match_the_configs():
    w = inputs.WORKLOADS
    assert (w["causal"].B, w["causal"].H, w["causal"].N, w["causal"].d) == (2, 16, 8192, 128)
    assert w["ragged"].N % 128 == 125
    assert w["decode"].kv_bytes() == 34359738368
    assert abs(w["causal"].flops() - 5.497558e11) / 5.497558e11 < 1e-6
