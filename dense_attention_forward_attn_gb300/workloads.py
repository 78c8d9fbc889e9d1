"""Seeded synthetic inputs for the attention forward.

This module holds no attention arithmetic: it only draws Q, K and V, rounds
them to BF16 and names the workload shapes.  Both the CUDA path and the CPU
oracle are fed from here (the one thing they share).

Shapes and distributions follow the benchmark shapes of "B200 Attention Kernel
from Scratch to Near-SOTA in 60 Diagrams" (Chapter 14, the FA4-paper shapes: S
in {4K, 8K, 16K}, 16 heads, head_dim 128, dense, non-causal, BF16) at half the
batch, plus a tiny case, a softmax-stress case and a 12K / 24-head case whose
tile count is not a power of two.

Draws use numpy's PCG64 generator (``standard_normal`` in float32), so a seed
gives the same bits on every machine; rounding to BF16 is round-to-nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    D: int = 128
    qk_std: float = 1.0          # standard deviation of Q and K entries
    v_std: float = 1.0
    spike_every: int = 0         # if > 0, key rows j with j % spike_every == spike_every-1 ...
    spike_factor: float = 1.0    # ... are multiplied by this (after BF16 rounding)
    seeds: tuple = field(default=(0,))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """4*B*H*Sq*Sk*D: two matmuls of 2*Sq*Sk*D each, per head."""
        return 4.0 * self.B * self.H * self.Sq * self.Sk * self.D

    def describe(self) -> dict:
        d = {"workload": self.name, "B": self.B, "H": self.H, "Sq": self.Sq, "Sk": self.Sk,
             "D": self.D, "causal": False, "layout": "BHSD contiguous", "dtype": "bf16",
             "qk_std": self.qk_std, "v_std": self.v_std}
        if self.spike_every:
            d["key_spike"] = f"rows j % {self.spike_every} == {self.spike_every - 1} x{self.spike_factor:g}"
        return d


TINY = Workload("tiny", 1, 2, 256, 256, seeds=(0, 1, 2))
STRESS = Workload("softmax-stress", 1, 4, 1024, 1024, qk_std=3.0, spike_every=64, spike_factor=8.0)
S4K = Workload("S=4K", 4, 16, 4096, 4096)
S8K = Workload("S=8K", 2, 16, 8192, 8192)
S16K = Workload("S=16K", 1, 16, 16384, 16384)
S12K = Workload("S=12K,H=24", 1, 24, 12288, 12288)

ALL = {w.name: w for w in (TINY, STRESS, S4K, S8K, S16K, S12K)}
HEADLINE = (S4K, S8K, S16K)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns (uint16), round to nearest even; NaN stays NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((u + rounding) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_inputs_bits(B: int, H: int, Sq: int, Sk: int, D: int = 128, seed: int = 0,
                     qk_std: float = 1.0, v_std: float = 1.0, spike_every: int = 0,
                     spike_factor: float = 1.0):
    """(q, k, v) as BF16 bit patterns, shapes [B,H,Sq,D], [B,H,Sk,D], [B,H,Sk,D]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((B, H, Sq, D), dtype=np.float32)
    k = rng.standard_normal((B, H, Sk, D), dtype=np.float32)
    v = rng.standard_normal((B, H, Sk, D), dtype=np.float32)
    if qk_std != 1.0:
        q *= np.float32(qk_std)
        k *= np.float32(qk_std)
    if v_std != 1.0:
        v *= np.float32(v_std)
    qb, kb, vb = to_bf16_bits(q), to_bf16_bits(k), to_bf16_bits(v)
    if spike_every:
        kf = bf16_bits_to_f32(kb)
        kf[:, :, spike_every - 1::spike_every, :] *= np.float32(spike_factor)
        kb = to_bf16_bits(kf)   # exact when the factor is a power of two
    return qb, kb, vb


def workload_inputs_bits(w: Workload, seed: int | None = None):
    return make_inputs_bits(w.B, w.H, w.Sq, w.Sk, w.D, w.seeds[0] if seed is None else seed,
                            w.qk_std, w.v_std, w.spike_every, w.spike_factor)


def bits_to_torch(bits: np.ndarray):
    """uint16 BF16 bit patterns -> torch.bfloat16 CPU tensor (no copy of values)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
