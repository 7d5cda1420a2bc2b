"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory or pass the library a workspace (a framework whose pool already owns
the device, a plugin that only receives its tensors, a stream being captured
into a CUDA graph, where cudaMalloc is not allowed).  It uses a scratch array
built into the library instead, so its results must match attn_bwd's, which
gets a caller-provided workspace -- on consecutive calls that share that
scratch.

Kept in a file of its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

from causal_gqa_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _noalloc(g, q, k, v, o, lse, do, scale):
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = g.lib().attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, T, D, 1,
                                  scale, torch.cuda.current_stream().cuda_stream)
    assert st == 0, g.status_string(st)
    return dq, dk, dv


@pytest.mark.parametrize("shapes", [[(2, 8, 2, 777, 128, 11), (1, 6, 6, 300, 64, 12)]])
def test_noalloc_matches_workspace_backward_on_consecutive_calls(shapes):
    import causal_gqa_attention_fwd_gb300 as g
    g.lib()
    for B, Hq, Hkv, T, D, seed in shapes:          # two calls in a row, different problems
        x = W.dense_inputs(B, Hq, Hkv, T, D, seed=seed)
        scale = 1.0 / np.sqrt(D)
        q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
        o, lse = g.attn_fwd(q, k, v, scale=scale)
        ref = g.attn_bwd(q, k, v, o, lse, do, scale=scale)          # caller-provided workspace
        got = _noalloc(g, q, k, v, o, lse, do, scale)
        assert g.get_device_status() == 0
        # every gradient is summed in a fixed order: bit for bit
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(a, b), name


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import causal_gqa_attention_fwd_gb300 as g
    lib = g.lib()
    cap = lib.attn_bwd_noalloc_scratch_bytes()
    assert cap == 16 << 20
    B, Hq, Hkv, T, D = 2, 1024, 8, 2048, 64
    assert lib.attn_bwd_workspace_size(B, Hq, Hkv, T, D) > cap
    p = 256      # aligned placeholder address: the call must return before touching it
    st = lib.attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, Hq, Hkv, T, D, 1, 0.088, None)
    assert st == 10, g.status_string(st)
