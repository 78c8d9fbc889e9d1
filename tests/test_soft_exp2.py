"""The optional software exp2 of the forward kernel (ATTN_FLAG_SOFT_EXP2), pinned on the CPU.

"B200 Attention Kernel from Scratch to Near-SOTA in 60 Diagrams", Chapter 9 and the appendix on the
approximation: 2^x = 2^floor(x) * p(x - floor(x)) with a cubic p on [0, 1).  These tests check the
kernel's constants against the minimax fit in soft_exp2_fit.py and the whole approximation, evaluated
the way the kernel does it in fp32 (single-rounding FMAs, exponent-field add), against fp64 exp2.
"""
import os
import re

import numpy as np

from dense_attention_forward_attn_gb300 import soft_exp2_fit

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KERNEL = os.path.join(ROOT, "dense_attention_forward_attn_gb300", "csrc", "attn_fwd_kernel.cuh")


def kernel_coefficients():
    src = open(KERNEL).read()
    vals = {}
    for name in ("kExp2C1", "kExp2C2", "kExp2C3"):
        m = re.search(name + r"\s*=\s*([0-9.eE+-]+)f", src)
        assert m, name
        vals[name] = np.float32(float(m.group(1)))
    return vals["kExp2C1"], vals["kExp2C2"], vals["kExp2C3"]


def fma32(a, b, c):
    """fp32 fused multiply-add: exact in fp64 for fp32 operands of these magnitudes, one rounding."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def soft_exp2_fp32(x):
    """The kernel's algorithm in fp32: clamp at -127, n = floor(x), f = x - n (exact), Horner in
    single-rounding FMAs, n added to the exponent field; 0 below -126."""
    c1, c2, c3 = kernel_coefficients()
    x = x.astype(np.float32)
    low = x < np.float32(-126.0)
    x = np.maximum(x, np.float32(-127.0))
    n = np.floor(x)
    f = (x - n).astype(np.float32)
    y = fma32(np.full_like(f, c3), f, np.full_like(f, c2))
    y = fma32(y, f, np.full_like(f, c1))
    y = fma32(y, f, np.ones_like(f))
    bits = y.view(np.int32) + (n.astype(np.int32) << 23)
    return np.where(low, np.float32(0.0), bits.view(np.float32))


def test_kernel_coefficients_are_the_minimax_fit():
    (c1, c2, c3), err = soft_exp2_fit.fit()
    assert kernel_coefficients() == (np.float32(c1), np.float32(c2), np.float32(c3))
    assert 5e-5 < err < 1e-4   # a cubic cannot do better; a wrong fit does worse


def test_fit_equioscillates():
    # the minimax property: the relative error reaches +-E at 4 points of (0, 1] with alternating signs
    (c1, c2, c3), err = soft_exp2_fit.fit()
    g = np.linspace(0.0, 1.0, 100001)
    e = soft_exp2_fit.relative_error((c1, c2, c3), g)
    peaks = [i for i in range(1, len(g) - 1) if abs(e[i]) >= abs(e[i - 1]) and abs(e[i]) >= abs(e[i + 1])
             and abs(e[i]) > 0.99 * err] + ([len(g) - 1] if abs(e[-1]) > 0.99 * err else [])
    signs = [np.sign(e[i]) for i in peaks]
    assert len(peaks) >= 4
    assert all(signs[i] != signs[i + 1] for i in range(len(signs) - 1))


def test_software_exp2_against_fp64():
    # every fp32 spacing region of the range P values take (x <= 8 by the rebase threshold)
    rng = np.random.default_rng(0)
    x = np.concatenate([np.linspace(-126.0, 8.0, 400001), rng.uniform(-126.0, 8.0, 200000),
                        np.arange(-126, 9, dtype=np.float64)]).astype(np.float32)
    got = soft_exp2_fp32(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 1.0e-4
    # exact at integers (p(0) = 1)
    xi = np.arange(-126, 9, dtype=np.float32)
    assert np.array_equal(soft_exp2_fp32(xi), np.exp2(xi.astype(np.float64)).astype(np.float32))


def test_software_exp2_is_zero_below_the_normal_range():
    # as the flushing hardware exp2: masked scores (-inf) and anything below -126 give exactly 0
    v = soft_exp2_fp32(np.array([-126.5, -127.0, -150.0, -1e30, -np.inf], dtype=np.float32))
    assert np.all(v == 0.0)
    assert soft_exp2_fp32(np.array([-126.0], dtype=np.float32))[0] == np.float32(2.0 ** -126)
