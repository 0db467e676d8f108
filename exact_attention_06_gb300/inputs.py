"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws tensors and names
shapes.  It is the one piece of Python shared by the tests, the bench and the
oracle checks, so that both sides see the same values.

Recipe (the pages measure no dataset; every workload is synthetic):
* Q, K, V are iid N(0, 1) drawn in fp32 by a seeded ``torch.Generator`` on the
  target device and rounded to bf16 (round-to-nearest-even), in slabs along
  the batch dimension so that the 17 GB decode tensors need no fp32 copy.
* Seeds: q = seed, k = seed + 1, v = seed + 2, sampled rows = seed + 3.
* The causal "spike" workload multiplies every 64th key row (0-based index
  j = 63 mod 64) by 8 after rounding; x8 is exact in bf16.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

SLAB_ELEMS = 1 << 27  # fp32 elements drawn at once (512 MB)


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "prefill" or "decode"
    B: int
    H: int
    N: int  # query rows (prefill) or KV length L (decode)
    d: int
    causal: bool
    spike: bool = False
    oracle_rows: int = 0  # 0 = every row; else seeded rows per head (prefill) or (b, h) rows (decode)

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)

    def flops(self) -> float:
        """Algorithmic FLOPs: 4 * B * H * N^2 * d, halved when causal (decode: 4 * B * H * L * d)."""
        if self.kind == "decode":
            return 4.0 * self.B * self.H * self.N * self.d
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def kv_bytes(self) -> int:
        """K and V bytes a decode step must read (bf16)."""
        return 2 * self.B * self.H * self.N * self.d * 2


WORKLOADS = {
    "tiny": Workload("tiny", "prefill", 1, 1, 256, 64, False),
    "prefill": Workload("prefill", "prefill", 4, 16, 2048, 64, False),
    "causal": Workload("causal", "prefill", 2, 16, 8192, 128, True, spike=True, oracle_rows=512),
    "ragged": Workload("ragged", "prefill", 1, 32, 16381, 128, True, oracle_rows=512),
    "decode": Workload("decode", "decode", 64, 32, 32768, 128, False, oracle_rows=256),
    # a 2.1 GB slice of the decode workload for profiler captures (still larger than L2)
    "decode_small": Workload("decode_small", "decode", 4, 32, 32768, 128, False, oracle_rows=16),
}


def normal_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """iid N(0,1) drawn in fp32 with a seeded generator, rounded to bf16."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    if out.numel() == 0:
        return out
    flat = out.view(-1)
    step = SLAB_ELEMS
    for start in range(0, flat.numel(), step):
        n = min(step, flat.numel() - start)
        flat[start:start + n] = torch.randn(n, generator=gen, dtype=torch.float32, device=device).to(torch.bfloat16)
    return out


def spike_every_64th_key(k: torch.Tensor) -> torch.Tensor:
    """Multiply key rows j = 63, 127, 191, ... (every 64th, 1-based) by 8, in place."""
    k[..., 63::64, :] *= 8
    return k


def prefill_inputs(B, H, N, d, seed=0, device="cpu", spike=False):
    q = normal_bf16((B, H, N, d), seed, device)
    k = normal_bf16((B, H, N, d), seed + 1, device)
    v = normal_bf16((B, H, N, d), seed + 2, device)
    if spike:
        spike_every_64th_key(k)
    return q, k, v


def decode_inputs(B, H, L, d, seed=0, device="cpu"):
    q = normal_bf16((B, H, d), seed, device)
    k = normal_bf16((B, H, L, d), seed + 1, device)
    v = normal_bf16((B, H, L, d), seed + 2, device)
    return q, k, v


def workload_inputs(w: Workload, seed=0, device="cpu"):
    if w.kind == "decode":
        return decode_inputs(w.B, w.H, w.N, w.d, seed, device)
    return prefill_inputs(w.B, w.H, w.N, w.d, seed, device, spike=w.spike)


def sample_rows(n: int, count: int, seed: int) -> torch.Tensor:
    """``count`` distinct sorted indices in [0, n) (all of them when count >= n)."""
    if count <= 0 or count >= n:
        return torch.arange(n)
    gen = torch.Generator().manual_seed(int(seed))
    return torch.randperm(n, generator=gen)[:count].sort().values


def sample_rows_per_head(B, H, n, count, seed) -> torch.Tensor:
    """[B, H, count] row indices, an independent seeded draw per head."""
    out = torch.empty(B, H, min(count, n) if count > 0 else n, dtype=torch.long)
    for b in range(B):
        for h in range(H):
            out[b, h] = sample_rows(n, count, seed * 100003 + b * H + h)
    return out
