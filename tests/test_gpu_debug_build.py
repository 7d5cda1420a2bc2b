"""The debug build (libgqa_attn_debug.so, -DGQA_DEBUG) on tiny and odd shapes.

In that build every kernel checks each computed tensor-map coordinate,
global row offset, workspace row and rotary-table row against its bounds
before the access; a failed check skips the access and records
ATTN_ERR_CHECK and its source line instead of trapping.  These cases (T = 1,
one row past a tile, ragged lengths, G = 3 and 8, non-causal, a packed batch
with an empty sequence, the rotary forward and backward) must raise no check
and still match the oracle.
"""
import numpy as np
import pytest

import oracle
from parity_util import TOL_REL_GRAD, TOL_REL_O, check, check_lse, to64
from causal_gqa_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    from causal_gqa_attention_fwd_gb300 import _binding, build
    path = build.build(debug=True)
    saved = (_binding._lib, _binding.LIB_PATH)
    _binding._lib, _binding.LIB_PATH = None, path
    assert _binding.lib().attn_is_debug_build() == 1
    import causal_gqa_attention_fwd_gb300 as g
    yield g
    _binding._lib, _binding.LIB_PATH = saved


def no_check_fired(g):
    assert g.get_device_status() == 0
    assert g.get_check_line() == 0


@pytest.mark.parametrize("B,Hq,Hkv,T,D,causal", [
    (1, 2, 1, 1, 64, True),
    (1, 4, 2, 65, 64, True),
    (1, 8, 1, 129, 128, True),
    (1, 6, 2, 333, 128, True),
    (2, 3, 3, 200, 64, False),
])
def test_debug_dense(dbg, B, Hq, Hkv, T, D, causal):
    g = dbg
    x = W.dense_inputs(B, Hq, Hkv, T, D, seed=77 + T)
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = g.attn_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = g.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    no_check_fired(g)
    ref = oracle.bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), causal=causal, scale=scale,
                     err_terms=True)
    check("o", o, ref["o"], TOL_REL_O)
    check_lse(lse, ref["lse"])
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        check(n, t, ref[n], TOL_REL_GRAD, ref["e" + n])


@pytest.mark.parametrize("lens,Hq,Hkv,D", [([1, 130, 64, 257], 4, 2, 128), ([128, 0, 7], 2, 1, 64)])
def test_debug_varlen(dbg, lens, Hq, Hkv, D):
    g = dbg
    x = W.varlen_inputs(lens, Hq, Hkv, D, seed=5 + sum(lens))
    scale = 1.0 / np.sqrt(D)
    cu = x["cu_seqlens"]
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    cud = cu.cuda()
    o, lse = g.attn_varlen_fwd(q, k, v, cud, x["max_seqlen"], scale=scale)
    dq, dk, dv = g.attn_varlen_bwd(q, k, v, o, lse, do, cud, x["max_seqlen"], scale=scale)
    no_check_fired(g)
    ref = oracle.varlen_bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), cu.numpy(), scale=scale,
                            err_terms=True)
    check("o", o, ref["o"], TOL_REL_O)
    check_lse(lse, ref["lse"])
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        check(n, t, ref[n], TOL_REL_GRAD, ref["e" + n])


def test_debug_rope(dbg):
    g = dbg
    B, Hq, Hkv, T, D = 1, 4, 2, 200, 128
    x = W.dense_inputs(B, Hq, Hkv, T, D, seed=91)
    tab = W.rope_cos_sin_table(T, D).cuda()
    scale = 1.0 / np.sqrt(D)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = g.attn_fwd_rope(q, k, v, tab, scale=scale)
    dq, dk, dv = g.attn_bwd_rope(q, k, v, o, lse, do, tab, scale=scale)
    no_check_fired(g)
    ref = oracle.rope_bwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), to64(x["do"]), tab.cpu().double().numpy(),
                          scale=scale, err_terms=True)
    check("o", o, ref["o"], TOL_REL_O)
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        check(n, t, ref[n], TOL_REL_GRAD, ref["e" + n])
