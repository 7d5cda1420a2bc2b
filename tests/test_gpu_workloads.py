"""The benchmark's workloads on the GPU against the fp64 oracle.

GPT-2-small MHA and the packed variable-length batch are compared in full.
The long-context GQA layer (B=2, Hq=32, Hkv=8, T=4096, D=128) runs in full on
the GPU exactly as the benchmark launches it; the oracle recomputes four sampled
(batch, kv-head) groups -- every output row of those groups, forward and
backward (a group's dK/dV need all of its query heads).
"""
import numpy as np
import pytest

import oracle
from parity_util import TOL_REL_GRAD, TOL_REL_O, check, check_lse, to64
from causal_gqa_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    import causal_gqa_attention_fwd_gb300 as g
    g.lib()
    oracle.set_threads(0)
    return g


def gpu_dense(gq, w, x):
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = gq.attn_fwd(q, k, v, scale=w.softmax_scale)
    dq, dk, dv = gq.attn_bwd(q, k, v, o, lse, do, scale=w.softmax_scale)
    assert gq.get_device_status() == 0
    return {n: t.cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}


def test_gpt2_small_mha_full(gq):
    w = W.WORKLOADS["gpt2_small_mha"]
    x = W.make_inputs(w)
    g = gpu_dense(gq, w, x)
    ref = oracle.bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), scale=w.softmax_scale,
                     err_terms=True)
    check("o", g["o"], ref["o"], TOL_REL_O)
    check_lse(g["lse"], ref["lse"])
    for n in ("dq", "dk", "dv"):
        check(n, g[n], ref[n], TOL_REL_GRAD, ref["e" + n])


def test_varlen16_full(gq):
    w = W.WORKLOADS["varlen16"]
    x = W.make_inputs(w)
    cu = x["cu_seqlens"]
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    cud = cu.cuda()
    o, lse = gq.attn_varlen_fwd(q, k, v, cud, x["max_seqlen"], scale=w.softmax_scale)
    dq, dk, dv = gq.attn_varlen_bwd(q, k, v, o, lse, do, cud, x["max_seqlen"], scale=w.softmax_scale)
    assert gq.get_device_status() == 0
    ref = oracle.varlen_bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), cu.numpy(),
                            scale=w.softmax_scale, err_terms=True)
    check("o", o, ref["o"], TOL_REL_O)
    check_lse(lse, ref["lse"])
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        check(n, t, ref[n], TOL_REL_GRAD, ref["e" + n])


@pytest.fixture(scope="module")
def long_gqa(gq):
    """The long-context layer run once on the GPU as the benchmark launches it."""
    w = W.WORKLOADS["long_gqa_t4096"]
    x = W.make_inputs(w)
    return w, x, gpu_dense(gq, w, x)


# both batch rows, the first and last K/V heads, and one from the middle
@pytest.mark.parametrize("b,g", [(0, 0), (0, 7), (1, 0), (1, 5)])
def test_long_gqa_t4096_sampled_group(long_gqa, b, g):
    w, x, out = long_gqa
    G = w.Hq // w.Hkv
    hs = slice(g * G, (g + 1) * G)
    ref = oracle.bwd(to64(x["q"][b:b + 1, hs]), to64(x["k"][b:b + 1, g:g + 1]), to64(x["v"][b:b + 1, g:g + 1]),
                     to64(x["do"][b:b + 1, hs]), scale=w.softmax_scale, err_terms=True)
    check("o", out["o"][b:b + 1, hs], ref["o"], TOL_REL_O)
    check_lse(out["lse"][b:b + 1, hs], ref["lse"])
    check("dq", out["dq"][b:b + 1, hs], ref["dq"], TOL_REL_GRAD, ref["edq"])
    check("dk", out["dk"][b:b + 1, g:g + 1], ref["dk"], TOL_REL_GRAD, ref["edk"])
    check("dv", out["dv"][b:b + 1, g:g + 1], ref["dv"], TOL_REL_GRAD, ref["edv"])
