"""The pages' tiled online-softmax recurrence, in fp64 -- TEST INFRASTRUCTURE ONLY.

Sources (all from "B200 Attention Kernel from Scratch to Near-SOTA in 60 Diagrams"):
  * Chapter 1, section B, "Online Softmax": per K/V tile, the tile row max, the
    new basis, the rescale of the running row sum and of O, P = exp(S - max),
    the row-sum update, and O += P V; the division by the row sum after the loop.
  * Chapter 8, "Hardware Approximations": exponents in base 2, with the softmax
    scale folded into log2(e); the row max is taken on the raw scores and the
    scalar is then multiplied by that folded factor.  P, the row sum and O are
    not in log2 space.
  * Chapter 11, "Skip O rescale": the kept row max is replaced only when the new
    candidate exceeds it by at least the threshold (8 base-2 units); otherwise P
    is taken relative to the stale kept max.
LSE in natural-log units: "Attention for sm90, Line by Line", the exp2 question.

This is the method's own recurrence, written from the pages' description in
their order: tile max -> candidate -> gap -> (rebase: rescale, new kept max)
-> P -> row sum -> O.  It reaches the plain definition in attn_oracle.c up to
rounding; tests/test_oracle.py pins it to that definition and to the worked
numbers the chapter prints (a gap of 7.78 keeps the old max and yields a P of
about 219; exp2(8) = 256; a gap of 20 yields 1,048,576).

Precision: fp64 throughout, no flush-to-zero, no BF16 rounding of P.
"""
from __future__ import annotations

import math

import numpy as np

LOG2E = 1.0 / math.log(2.0)
REBASE_THRESHOLD_LOG2 = 8.0  # Chapter 11, "Actual thresh value"


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns (uint16) to fp64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def online_attention_head(q, k, v, scale: float, block_n: int = 128,
                          threshold_log2: float = REBASE_THRESHOLD_LOG2):
    """One head: q [Sq,D], k/v [Sk,D] (fp64 values).  Returns (O, LSE, rebases, m_kept, rowsum).

    ``rebases`` counts, per row, the tiles at which the kept max was replaced
    (the first tile always counts: the kept max starts at minus infinity).
    ``m_kept`` and ``rowsum`` are the final carrier state in the pages' units.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if scale < 0:
        raise ValueError("the row max is taken on raw scores and then scaled: needs scale >= 0")
    Sq, D = q.shape
    Sk = k.shape[0]
    softmax_scale_log2 = scale * LOG2E
    kept_rowmax = np.full(Sq, -np.inf)
    rowsum = np.zeros(Sq)
    o_acc = np.zeros((Sq, v.shape[1]))
    rebases = np.zeros(Sq, dtype=np.int64)
    for j0 in range(0, Sk, block_n):
        s = q @ k[j0:j0 + block_n].T                      # raw scores of this tile
        tile_rowmax = s.max(axis=1) * softmax_scale_log2   # scalar per row, base-2 units
        candidate = np.maximum(kept_rowmax, tile_rowmax)
        gap = candidate - kept_rowmax                      # +inf on the first tile
        rebase = gap >= threshold_log2
        rescale = np.where(rebase, np.exp2(np.where(rebase, kept_rowmax - candidate, 0.0)), 1.0)
        rowsum = rowsum * rescale
        o_acc = o_acc * rescale[:, None]
        kept_rowmax = np.where(rebase, candidate, kept_rowmax)
        rebases += rebase
        p = np.exp2(s * softmax_scale_log2 - kept_rowmax[:, None])
        rowsum = rowsum + p.sum(axis=1)
        o_acc = o_acc + p @ v[j0:j0 + block_n]
    o = o_acc / rowsum[:, None]
    lse = (kept_rowmax + np.log2(rowsum)) / LOG2E
    return o, lse, rebases, kept_rowmax, rowsum


def online_attention(q_bits, k_bits, v_bits, scale: float, block_n: int = 128,
                     threshold_log2: float = REBASE_THRESHOLD_LOG2):
    """All heads of BF16 bit-pattern inputs [B,H,S,D]: returns (O, LSE, rebases)."""
    q = bf16_bits_to_f64(q_bits)
    k = bf16_bits_to_f64(k_bits)
    v = bf16_bits_to_f64(v_bits)
    B, H, Sq, D = q.shape
    o = np.empty((B, H, Sq, v.shape[3]))
    lse = np.empty((B, H, Sq))
    reb = np.empty((B, H, Sq), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h], reb[b, h], _, _ = online_attention_head(
                q[b, h], k[b, h], v[b, h], scale, block_n, threshold_log2)
    return o, lse, reb
