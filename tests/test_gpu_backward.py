"""GPU parity of the backward (through the C ABI) against the fp64 oracle's gradients.

The GPU forward's own O and LSE feed the GPU backward (the way the two are used together); the
oracle differentiates the plain definition from the same BF16 inputs.  Tolerance, derived from
the arithmetic: P and dS enter the tensor-core products as BF16 (relative rounding 2^-9), the
products accumulate in fp32, and the gradients are rounded to BF16 once; errors therefore scale
with the gradient's own magnitude.  delta = rowsum(dO o O) is taken from the forward's BF16 O, so
on rows where P is nearly one-hot (the softmax-stress logits) dP - delta cancels and its rounding
error grows relative to the result.  Per tensor: max-abs error <= 2e-2 * max|ref| and mean-abs
error <= 2e-2 * mean|ref|.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from dense_attention_forward_attn_gb300 import attn, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _status_clean():
    torch.cuda.set_device(0)
    attn.device_status(clear=True)
    yield
    torch.cuda.synchronize()
    assert attn.device_status() == 0, "a bounded wait expired inside a kernel"


def _grads(B, H, Sq, Sk, seed, causal=False, scale=None, **kw):
    qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, 128, seed=seed, **kw)
    dob = wl.make_inputs_bits(B, H, Sq, Sq, 128, seed=seed + 1000)[0]
    scale = 1.0 / math.sqrt(128) if scale is None else scale
    q, k, v, do = (wl.bits_to_torch(x).cuda() for x in (qb, kb, vb, dob))
    o, lse = attn.fwd(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = attn.bwd(q, k, v, o, do, lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    got = [t.float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]
    ref = oracle.attn_bwd(qb, kb, vb, dob, scale, causal=causal)
    return got, ref


def _check(got, ref):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        assert np.isfinite(g).all(), name
        err = np.abs(g - r)
        scale_max, scale_mean = np.abs(r).max(), np.abs(r).mean()
        assert err.max() <= 2e-2 * scale_max + 1e-6, f"{name} max-abs {err.max():.3g} vs {scale_max:.3g}"
        assert err.mean() <= 2e-2 * scale_mean + 1e-7, f"{name} mean-abs {err.mean():.3g} vs {scale_mean:.3g}"


@pytest.mark.parametrize("shape", [(1, 2, 256, 256), (1, 3, 384, 640), (2, 2, 640, 256),
                                   (1, 1, 128, 128), (1, 2, 200, 300), (1, 1, 1, 1)])
def test_backward(shape):
    _check(*_grads(*shape, seed=sum(shape)))


@pytest.mark.parametrize("shape", [(1, 2, 256, 256), (1, 2, 640, 640), (1, 2, 300, 300),
                                   (1, 2, 640, 300), (1, 2, 300, 900)])
def test_backward_causal(shape):
    _check(*_grads(*shape, seed=sum(shape) + 3, causal=True))


def test_backward_stress_logits():
    w = wl.STRESS
    _check(*_grads(w.B, w.H, w.Sq, w.Sk, seed=5, qk_std=w.qk_std, spike_every=w.spike_every,
                   spike_factor=w.spike_factor))


def test_backward_deterministic():
    qb, kb, vb = wl.make_inputs_bits(1, 4, 1024, 1024, 128, seed=9)
    q, k, v, do = (wl.bits_to_torch(x).cuda() for x in (qb, kb, vb, qb))
    o, lse = attn.fwd(q, k, v)
    a = attn.bwd(q, k, v, o, do, lse)
    b = attn.bwd(q, k, v, o, do, lse)
    assert all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("name,heads", [("S=4K", (1,)), ("S=8K", (1,)), ("S=16K", (0, 5, 10, 15))])
def test_backward_full_size_whole_heads(name, heads):
    # the workload on the GPU (all heads, the benchmark's launch); the oracle checks every
    # gradient element of the listed heads (of batch 1, or 0 when B == 1).  The oracle runs one
    # thread per head, so the four S=16K heads take about as long as one (~2-3 min).
    w = wl.ALL[name]
    qb, kb, vb = wl.workload_inputs_bits(w)
    dob = wl.make_inputs_bits(w.B, w.H, w.Sq, w.Sq, 128, seed=77)[0]
    q, k, v, do = (wl.bits_to_torch(x).cuda() for x in (qb, kb, vb, dob))
    o, lse = attn.fwd(q, k, v, scale=w.scale)
    dq, dk, dv = attn.bwd(q, k, v, o, do, lse, scale=w.scale)
    torch.cuda.synchronize()
    b = min(1, w.B - 1)
    hs = list(heads)
    pick = lambda x: np.ascontiguousarray(x[b:b + 1][:, hs])
    ref = oracle.attn_bwd(pick(qb), pick(kb), pick(vb), pick(dob), w.scale)
    got = [t[b:b + 1][:, hs].float().cpu().numpy().astype(np.float64) for t in (dq, dk, dv)]
    _check(got, ref)


@pytest.mark.parametrize("shape,causal", [((2, 3, 256, 384), False), ((3, 2, 300, 300), True),
                                          ((1, 4, 640, 200), False)])
def test_backward_bshd_layout(shape, causal):
    """[B,S,H,D] tensors read and written in place: bitwise equal to the [B,H,S,D] path on the
    same values, and within tolerance of the oracle."""
    B, H, Sq, Sk = shape
    qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, 128, seed=sum(shape) + 11)
    dob = wl.make_inputs_bits(B, H, Sq, Sq, 128, seed=sum(shape) + 12)[0]
    scale = 1.0 / math.sqrt(128)
    bhsd = [wl.bits_to_torch(x).cuda() for x in (qb, kb, vb, dob)]
    o, lse = attn.fwd(*bhsd[:3], scale=scale, causal=causal)
    ref_t = attn.bwd(*bhsd[:3], o, bhsd[3], lse, scale=scale, causal=causal)
    t = lambda x: x.transpose(1, 2).contiguous()
    q2, k2, v2, do2 = (t(x) for x in bhsd)
    o2, lse2 = attn.fwd(q2, k2, v2, scale=scale, causal=causal, layout="bshd")
    got_t = attn.bwd(q2, k2, v2, o2, do2, lse2, scale=scale, causal=causal, layout="bshd")
    torch.cuda.synchronize()
    for a, b in zip(ref_t, got_t):
        assert torch.equal(a, b.transpose(1, 2))
    got = [x.transpose(1, 2).float().cpu().numpy().astype(np.float64) for x in got_t]
    _check(got, oracle.attn_bwd(qb, kb, vb, dob, scale, causal=causal))
