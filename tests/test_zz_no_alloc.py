"""The allocation-free backward entry point, attn_bwd_noalloc, through the C ABI.

Some callers of this library cannot allocate device memory around it: code running under a
fixed memory budget or its own allocator, embedders that own every device allocation, or paths
where a cudaMalloc would synchronise the device.  attn_bwd needs a scratch buffer (delta, one
float per query row) from its caller; attn_bwd_noalloc uses a fixed 4 MiB array compiled into
the library instead.  These tests check that its gradients agree with attn_bwd's on the same
inputs, on two calls in a row with different inputs (the array keeps the previous call's
contents, which must not leak into the next result), that calls after the first one on a device
leave the device's free memory unchanged (also a larger problem after a smaller one), and that
a problem beyond the array's size is rejected.  The file runs last (its name) and also passes
alone in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from dense_attention_forward_attn_gb300 import attn, build, workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build.build()
    torch.cuda.set_device(0)
    return attn.library()


def _noalloc(lib, q, k, v, o, do, lse, scale, causal, out=None):
    dq, dk, dv = out if out is not None else (torch.empty_like(q), torch.empty_like(k),
                                              torch.empty_like(v))
    B, H, Sq, D = q.shape
    rc = lib.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                              lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Sq,
                              k.shape[2], D, scale, attn.ATTN_FLAG_CAUSAL if causal else 0,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == attn.ATTN_OK, attn.status_string(rc)
    return dq, dk, dv


def _close(got, ref):
    # the backward tests' tolerance: per tensor, max-abs <= 2e-2 * max|ref|, mean-abs <= 2e-2 * mean|ref|
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = g.float().cpu().numpy().astype(np.float64)
        r = r.float().cpu().numpy().astype(np.float64)
        err = np.abs(g - r)
        assert np.isfinite(g).all(), name
        assert err.max() <= 2e-2 * np.abs(r).max() + 1e-6, name
        assert err.mean() <= 2e-2 * np.abs(r).mean() + 1e-7, name


def test_noalloc_backward_matches_attn_bwd_on_two_calls(lib):
    attn.device_status(clear=True)
    cases = [((1, 4, 512, 640), False, 0), ((2, 3, 300, 300), True, 1)]
    for (B, H, Sq, Sk), causal, seed in cases:
        qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, 128, seed=60 + seed)
        dob = wl.make_inputs_bits(B, H, Sq, Sq, 128, seed=70 + seed)[0]
        q, k, v, do = (wl.bits_to_torch(x).cuda() for x in (qb, kb, vb, dob))
        scale = 1.0 / math.sqrt(128)
        o, lse = attn.fwd(q, k, v, scale=scale, causal=causal)
        ref = attn.bwd(q, k, v, o, do, lse, scale=scale, causal=causal)
        got = _noalloc(lib, q, k, v, o, do, lse, scale, causal)
        torch.cuda.synchronize()
        _close(got, ref)
    assert attn.device_status() == 0


def _problem(B, H, Sq, Sk, seed, causal=False):
    qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, 128, seed=seed)
    dob = wl.make_inputs_bits(B, H, Sq, Sq, 128, seed=seed + 1)[0]
    q, k, v, do = (wl.bits_to_torch(x).cuda() for x in (qb, kb, vb, dob))
    scale = 1.0 / math.sqrt(128)
    o, lse = attn.fwd(q, k, v, scale=scale, causal=causal)
    ref = attn.bwd(q, k, v, o, do, lse, scale=scale, causal=causal)
    out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    return (q, k, v, o, do, lse, scale, causal), ref, out


def test_noalloc_call_allocates_no_device_memory(lib):
    """After the first call on the device (its one-time set-up), calls change the device's free
    memory by nothing, also when a larger problem follows a smaller one; the larger one's
    gradients still agree with attn_bwd's.  Every buffer, including attn_bwd's reference results,
    is allocated before the measured calls."""
    attn.device_status(clear=True)
    small, ref_small, out_small = _problem(1, 2, 256, 384, seed=81)
    large, ref_large, out_large = _problem(4, 16, 1024, 1024, seed=83, causal=True)   # 64K rows
    _noalloc(lib, *small, out=out_small)   # the first call on this device may set things up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    _noalloc(lib, *small, out=out_small)
    _noalloc(lib, *large, out=out_large)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    _close(out_small, ref_small)
    _close(out_large, ref_large)
    assert attn.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # B*H*Sq = 2**20 + 128 rows of delta do not fit the fixed 4 MiB array; nothing is launched
    vp = ctypes.c_void_p
    big = 1 << 40
    rc = lib.attn_bwd_noalloc(*(vp(big * (i + 1)) for i in range(9)), 1, 8193, 128, 128, 128, 0.1, 0,
                              None)
    assert rc == attn.ATTN_ERR_TOO_LARGE
    assert "scratch" in attn.status_string(rc)
