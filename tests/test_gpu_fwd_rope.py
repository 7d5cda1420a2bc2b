"""Forward with rotary queries and keys on the GPU against the fp64 oracle
(``oracle.rope_fwd``: q and k rotated at positions 0..T-1, then attention).

The kernel rotates into f16 copies (11 significant bits) and runs the score
MMA on them; the tolerances are the forward's.  Cases: D 64 and 128, G 1, 2,
3 and 8, causal and not, ragged lengths across several 128-row tiles, the
T = 4096 length with many positions, and a table whose every row is position
0 (no rotation: the result then matches attn_fwd's on the same inputs, whose
bf16 values the f16 copies hold exactly).
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_REL_O, check, check_lse, to64
from causal_gqa_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gq():
    import causal_gqa_attention_fwd_gb300 as g
    g.lib()
    oracle.set_threads(0)
    return g


CASES = [
    # B, Hq, Hkv, T, D, causal
    (1, 4, 2, 128, 64, True),
    (2, 2, 1, 333, 128, True),
    (1, 6, 2, 200, 128, True),     # G = 3
    (1, 8, 1, 1000, 128, True),    # G = 8
    (2, 3, 3, 300, 64, True),      # MHA
    (1, 4, 2, 200, 128, False),
    (1, 2, 1, 4096, 128, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,T,D,causal", CASES)
def test_fwd_rope_matches_oracle(gq, B, Hq, Hkv, T, D, causal):
    x = W.dense_inputs(B, Hq, Hkv, T, D, seed=T + D + 7)
    tab = W.rope_cos_sin_table(T + 5, D)
    scale = 1.0 / np.sqrt(D)
    o, lse = gq.attn_fwd_rope(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), tab.cuda(), causal=causal, scale=scale)
    assert gq.get_device_status() == 0
    ro, rl = oracle.rope_fwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), tab.double().numpy(), causal=causal,
                             scale=scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rl)
    plain, _ = gq.attn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), causal=causal, scale=scale)
    assert not torch.equal(plain, o)


def test_fwd_rope_at_position_zero_is_the_plain_forward(gq):
    B, Hq, Hkv, T, D = 1, 4, 2, 300, 128
    x = W.dense_inputs(B, Hq, Hkv, T, D, seed=3)
    tab = W.rope_cos_sin_table(1, D).expand(T, D).contiguous()   # every row: cos 1, sin 0
    q, k, v = x["q"].cuda(), x["k"].cuda(), x["v"].cuda()
    o, lse = gq.attn_fwd_rope(q, k, v, tab.cuda(), scale=0.1)
    o2, lse2 = gq.attn_fwd(q, k, v, scale=0.1)
    assert gq.get_device_status() == 0
    # same operand values (the f16 copies of these bf16 values are exact);
    # only the MMA's operand format differs
    assert float((o.float() - o2.float()).abs().max()) <= 2.0 ** -7 * float(o2.float().abs().max())
    assert float((lse - lse2).abs().max()) <= 1e-5


VARLEN_CASES = [
    # lengths, Hq, Hkv, D
    ([1, 300, 129, 64], 4, 2, 128),
    ([700, 5, 256], 8, 1, 64),
    ([2048, 17], 6, 2, 128),
]


@pytest.mark.parametrize("lens,Hq,Hkv,D", VARLEN_CASES)
def test_varlen_fwd_rope_matches_oracle(gq, lens, Hq, Hkv, D):
    """Packed batch: each sequence's tokens at positions 0..len-1."""
    x = W.varlen_inputs(lens, Hq, Hkv, D, seed=sum(lens) + 3)
    cu = x["cu_seqlens"]
    tab = W.rope_cos_sin_table(max(lens), D)
    scale = 1.0 / np.sqrt(D)
    o, lse = gq.attn_varlen_fwd_rope(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), cu.cuda(), x["max_seqlen"],
                                     tab.cuda(), scale=scale)
    assert gq.get_device_status() == 0
    ro, rl = oracle.rope_varlen_fwd(to64(x["q"]), to64(x["k"]), to64(x["v"]), cu.numpy(), tab.double().numpy(),
                                    scale=scale)
    check("o", o, ro, TOL_REL_O)
    check_lse(lse, rl)


def test_varlen_fwd_rope_reports_positions_past_the_table(gq):
    """A sequence longer than max_seqlen (malformed cu_seqlens) would need
    table rows past rope_positions: reported, nothing read out of bounds."""
    x = W.varlen_inputs([10, 40], 4, 2, 64, seed=9)
    cu = x["cu_seqlens"]
    tab = W.rope_cos_sin_table(16, 64)       # rows for positions 0..15 only
    gq.attn_varlen_fwd_rope(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), cu.cuda(), 16, tab.cuda(), scale=0.1)
    assert gq.get_device_status() == 5
    assert gq.get_device_status() == 0


def test_fwd_rope_reports_rotated_values_beyond_f16(gq):
    """The rotated copies are f16: a rotated value that does not fit (here a
    q element of 70144 at position 0, where the rotation leaves it as is) is
    recorded as ATTN_ERR_RANGE (13); one that fits (59904) is not; the next
    call on ordinary inputs reports nothing."""
    B, Hq, Hkv, T, D = 1, 2, 1, 128, 128
    x = W.dense_inputs(B, Hq, Hkv, T, D, seed=21)
    tab = W.rope_cos_sin_table(T, D).cuda()
    k, v = x["k"].cuda(), x["v"].cuda()
    q = x["q"].clone()
    q[0, 1, 0, 0] = 60000.0                     # bf16 59904: fits f16
    gq.attn_fwd_rope(q.cuda(), k, v, tab, scale=0.1)
    assert gq.get_device_status() == 0
    q[0, 1, 0, 0] = 70000.0                     # bf16 70144: beyond f16
    gq.attn_fwd_rope(q.cuda(), k, v, tab, scale=0.1)
    assert gq.get_device_status() == 13
    o, lse = gq.attn_fwd_rope(x["q"].cuda(), k, v, tab, scale=0.1)
    assert gq.get_device_status() == 0
    assert torch.isfinite(o.float()).all()
