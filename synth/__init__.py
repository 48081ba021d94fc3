"""Seeded synthetic inputs and the workload table for fused exact attention.

This module holds none of the attention arithmetic.  It only draws random
inputs (CPU ``torch.Generator`` -> fp32 normal -> bf16 round-to-nearest-even)
and names the workloads, so that the tests, the benchmark and the oracle
checks all see the same tensors.  Layout is [B, H, S, D] row-major.

Workloads (shapes and value distributions):

* ``tiny``      B=1, Hq=Hkv=2, S=256, D=64, N(0,1), seed 42, non-causal, scale 1/8.
* ``train``     B=4, Hq=Hkv=16, S=2048, D=128, N(0,1), seed 1, causal and
                non-causal, scale 1/sqrt(128).
* ``sweep``     B=max(1, 16384/S), H=16, S in 1k..32k, D in {64, 128}, seed 2.
* ``gqa_spike`` B=2, Hq=32, Hkv=8, S=8192, D=128, causal.  Q, K = 3*N(0,1);
                per (b, kv head) floor(0.01*Sk) key rows, chosen uniformly
                without replacement, are scaled x8 before rounding; V ~ N(0,1);
                seed 3.
* ``bwd``       B=2, Hq=Hkv=16, S=8192, D=128, causal; Q, K, V, dO ~ N(0,1); seed 4.

Draw order is Q, K, V, then dO (when wanted), then the spike positions.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    seed: int
    qk_std: float = 1.0
    spike_frac: float = 0.0
    spike_mult: float = 1.0
    scale: float | None = None
    with_do: bool = False
    tags: tuple = field(default_factory=tuple)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    def flops(self, backward: bool = False) -> float:
        return flop_count(self.B, self.Hq, self.Sq, self.Sk, self.D, self.causal, backward)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def flop_count(B, Hq, Sq, Sk, D, causal: bool, backward: bool = False) -> float:
    """Measurement convention: 4*B*Hq*Sq*Sk*D for the forward pass, halved when
    causal; the backward pass counts 2.5x the forward."""
    f = 4.0 * B * Hq * Sq * Sk * D
    if causal:
        f *= 0.5
    return f * 2.5 if backward else f


TINY = Workload("tiny", 1, 2, 2, 256, 256, 64, False, 42, scale=1.0 / 8.0)
TRAIN = Workload("train", 4, 16, 16, 2048, 2048, 128, True, 1)
TRAIN_NONCAUSAL = TRAIN.with_(name="train_noncausal", causal=False)
GQA_SPIKE = Workload("gqa_spike", 2, 32, 8, 8192, 8192, 128, True, 3, qk_std=3.0,
                     spike_frac=0.01, spike_mult=8.0)
BWD = Workload("bwd", 2, 16, 16, 8192, 8192, 128, True, 4, with_do=True)
SWEEP_S = (1024, 2048, 4096, 8192, 16384, 32768)


def sweep(S: int, D: int, causal: bool) -> Workload:
    B = max(1, 16384 // S)
    return Workload(f"sweep_s{S}_d{D}_{'causal' if causal else 'noncausal'}", B, 16, 16, S, S,
                    D, causal, 2)


def _randn(shape, gen, std=1.0):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x


def make_inputs(w: Workload, device="cpu", with_do: bool | None = None):
    """Draw (q, k, v[, do]) as bf16 tensors for workload ``w``.

    Spiked key rows (``spike_frac`` > 0) are scaled in fp32 before the single
    rounding to bf16.
    """
    gen = torch.Generator().manual_seed(w.seed)
    q = _randn((w.B, w.Hq, w.Sq, w.D), gen, w.qk_std)
    k = _randn((w.B, w.Hkv, w.Sk, w.D), gen, w.qk_std)
    v = _randn((w.B, w.Hkv, w.Sk, w.D), gen)
    want_do = w.with_do if with_do is None else with_do
    do = _randn((w.B, w.Hq, w.Sq, w.D), gen) if want_do else None
    if w.spike_frac > 0:
        n_spike = int(math.floor(w.spike_frac * w.Sk))
        for b in range(w.B):
            for hk in range(w.Hkv):
                rows = torch.randperm(w.Sk, generator=gen)[:n_spike]
                k[b, hk, rows, :] *= w.spike_mult
    out = [t.to(torch.bfloat16).to(device) for t in (q, k, v)]
    if do is not None:
        out.append(do.to(torch.bfloat16).to(device))
    return tuple(out)


def sample_rows(w: Workload, n_per_head: int = 256, full_heads: int = 2, seed: int = 7):
    """Seeded flat row indices (b*Hq + h)*Sq + i for sampled checks.

    ``full_heads`` whole (b, h) heads plus ``n_per_head`` rows of every other
    head; every head's sample includes rows 0, Sq-1 and the tile edges 127/128
    when they exist.
    """
    g = torch.Generator().manual_seed(seed)
    BH = w.B * w.Hq
    full = set(torch.randperm(BH, generator=g)[:full_heads].tolist())
    fixed = [i for i in (0, 127, 128, w.Sq - 1) if 0 <= i < w.Sq]
    rows = []
    for bh in range(BH):
        if bh in full:
            idx = list(range(w.Sq))
        else:
            pick = torch.randperm(w.Sq, generator=g)[:n_per_head].tolist()
            idx = sorted(set(pick) | set(fixed))
        rows.extend(bh * w.Sq + i for i in idx)
    return rows


def shard_units(n_units: int, rank: int, world: int):
    """Contiguous, balanced slice [lo, hi) of ``n_units`` independent units for
    ``rank`` of ``world`` (used to split batches across ranks)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, rem = divmod(n_units, world)
    lo = rank * base + min(rank, rem)
    hi = lo + base + (1 if rank < rem else 0)
    return lo, hi
