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


@pytest.mark.parametrize("kernel,name", [(1, "forward"), (2, "backward dK/dV"), (3, "backward dQ")])
def test_production_kernel_wait_expires_and_next_call_is_clean(kernel, name):
    """attn_test_inject_timeout makes one wait of a production kernel run out
    (its first CTA's producer stops before its second step, waits limited to
    50 ms): the launch must record ATTN_ERR_TIMEOUT and return -- drained and
    with its TMEM freed, or the next launch on that SM could not allocate --
    and the next normal call must reproduce a clean run bit for bit."""
    import causal_gqa_attention_fwd_gb300 as g
    from causal_gqa_attention_fwd_gb300 import workloads as W
    lib = g.lib()
    x = W.dense_inputs(1, 4, 2, 1024, 128, seed=kernel)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1.0 / np.sqrt(128)

    def run():
        o, lse = g.attn_fwd(q, k, v, scale=scale)
        dq, dk, dv = g.attn_bwd(q, k, v, o, lse, do, scale=scale)
        return [t.clone() for t in (o, lse, dq, dk, dv)]

    assert g.get_device_status() in (0, 9)             # clear anything earlier
    ref = run()
    assert g.get_device_status() == 0
    assert lib.attn_test_inject_timeout(kernel, 50) == 0
    run()
    code = g.get_device_status(clear=True)
    assert code == 9, f"{name}: {g.status_string(code)}"   # ATTN_ERR_TIMEOUT
    again = run()
    assert g.get_device_status() == 0
    for a, b in zip(again, ref):
        assert torch.equal(a, b), name
