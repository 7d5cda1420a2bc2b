"""Failure detection on the GPU without faulting or hanging it.

Every in-kernel wait of the library is bounded.  attn_selftest_wait_timeout
launches a kernel whose wait can never be satisfied (a barrier phase nothing
completes) with a short limit: the wait must give up, record ATTN_ERR_TIMEOUT
in the device status word and let the kernel return, leaving the context
usable -- a normal call afterwards succeeds with a clean status.
"""
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_reports_timeout():
    import causal_gqa_attention_fwd_gb300 as g
    lib = g.lib()
    assert g.get_device_status() in (0, 9)            # clear anything earlier
    t0 = time.perf_counter()
    st = lib.attn_selftest_wait_timeout(50, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    code = g.get_device_status(clear=True)
    elapsed = time.perf_counter() - t0
    assert code == 9, g.status_string(code)            # ATTN_ERR_TIMEOUT
    assert 0.04 < elapsed < 5.0
    assert g.get_device_status() == 0                  # cleared
    # the context is still healthy: a real call works and reports no error
    q = torch.randn(1, 2, 130, 64, device="cuda").to(torch.bfloat16)
    k = torch.randn(1, 1, 130, 64, device="cuda").to(torch.bfloat16)
    o, lse = g.attn_fwd(q, k, k)
    torch.cuda.synchronize()
    assert g.get_device_status() == 0
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_selftest_rejects_bad_limits():
    import causal_gqa_attention_fwd_gb300 as g
    lib = g.lib()
    assert lib.attn_selftest_wait_timeout(0, None) == 2
    assert lib.attn_selftest_wait_timeout(6000, None) == 2
