"""The kernel's failure path on the GPU, without a fault: a wait that runs out.

With ATTN_FLAG_TEST_WITHHOLD the TMA warp of CTA 0 never loads its first K tile, so the MMA warp's
bounded wait on that tile expires (after 2 s).  The CTA must then record the expiry in the device
status word, stop every role, wait for its own copies in flight, free its tensor memory and exit;
the context stays usable and the next call is exact again.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from dense_attention_forward_attn_gb300 import attn, workloads as wl

pytestmark = pytest.mark.gpu

STATUS_TIMEOUT_MMA = 1 << 1


def test_expired_wait_is_reported_and_the_context_survives():
    torch.cuda.set_device(0)
    B, H, S = 1, 2, 512
    qb, kb, vb = wl.make_inputs_bits(B, H, S, S, 128, seed=3)
    q, k, v = (wl.bits_to_torch(x).cuda() for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, device="cuda")
    scale = 1.0 / math.sqrt(128)
    attn.device_status(clear=True)
    rc = attn.library().attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), B, H, S, S, 128, scale,
                                    attn.ATTN_FLAG_TEST_WITHHOLD,
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == attn.ATTN_OK
    torch.cuda.synchronize()   # returns: the waits are bounded
    status = attn.device_status(clear=True)
    assert status & STATUS_TIMEOUT_MMA, f"status {status:#x}"
    # the same context computes the next call exactly
    o2, lse2 = attn.fwd(q, k, v, scale=scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(qb, kb, vb, scale)
    err = np.abs(o2.float().cpu().numpy().astype(np.float64) - o_ref)
    assert err.max() <= 2e-2 and np.abs(lse2.cpu().numpy() - lse_ref).max() <= 1e-3
