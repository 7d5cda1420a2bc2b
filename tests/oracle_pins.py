"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each pin takes the loaded oracle library and raises AssertionError when the
oracle disagrees with a closed form, an invariant, a hand-worked case, a
library routine on a special case, or finite differences.  The same list is
run against variants of the oracle with a planted mistake, each of which must
fail at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _ev(x):
    if isinstance(x, list):
        return [_ev(y) for y in x]
    return float(eval(x, {"__builtins__": {}}, {"log": math.log}))


def pin_hand_worked(lib):
    """Two-token case worked by hand (tests/golden/hand_t2.json)."""
    g = json.load(open(os.path.join(GOLDEN, "hand_t2.json")))
    inp = {k: np.array(_ev(v)) for k, v in g["inputs"].items() if k != "scale"}
    scale = _ev(g["inputs"]["scale"])
    q, k, v, do = (inp[n][None, None] for n in ("q", "k", "v", "do"))
    r = oracle.bwd(q, k, v, do, causal=True, scale=scale, lib=lib)
    exp = {n: np.array(_ev(x)) for n, x in g["causal"].items()}
    for n in ("o", "dq", "dk", "dv"):
        np.testing.assert_allclose(r[n][0, 0], exp[n], atol=1e-14, err_msg=n)
    np.testing.assert_allclose(r["lse"][0, 0], exp["lse"], atol=1e-14)
    np.testing.assert_allclose(r["delta"][0, 0], exp["delta"], atol=1e-14)
    o, lse = oracle.fwd(q, k, v, causal=False, scale=scale, lib=lib)
    nc = g["noncausal_row0"]
    np.testing.assert_allclose(o[0, 0, 0], _ev(nc["o"]), atol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], _ev(nc["lse"]), atol=1e-14)


def pin_rows_sum_to_one(lib):
    """V = identity (D = T) makes O equal P: rows sum to 1, entries are
    non-negative and the causal upper triangle is exactly zero; V = ones
    gives O = 1."""
    r = _rng(1)
    T = 9
    q = r.standard_normal((1, 2, T, T))
    k = r.standard_normal((1, 1, T, T))
    eye = np.broadcast_to(np.eye(T), (1, 1, T, T)).copy()
    for causal in (True, False):
        P, _ = oracle.fwd(q, k, eye, causal=causal, scale=0.7, lib=lib)
        np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-13)
        assert (P >= 0).all()
        if causal:
            assert np.all(np.triu(P[0, 0], 1) == 0) and np.all(np.triu(P[0, 1], 1) == 0)
            assert np.all(np.diag(P[0, 0]) > 0)
        else:
            assert np.all(P > 0)
    o, _ = oracle.fwd(q, k, np.ones((1, 1, T, T)), causal=True, scale=0.7, lib=lib)
    np.testing.assert_allclose(o, 1.0, atol=1e-13)


def pin_single_token(lib):
    """T = 1: the only visible key is the query's own: O = V, LSE = scale q.k."""
    r = _rng(2)
    q = r.standard_normal((2, 4, 1, 8))
    k = r.standard_normal((2, 2, 1, 8))
    v = r.standard_normal((2, 2, 1, 8))
    o, lse = oracle.fwd(q, k, v, causal=True, scale=0.3, lib=lib)
    vrep = np.repeat(v, 2, axis=1)
    krep = np.repeat(k, 2, axis=1)
    np.testing.assert_allclose(o, vrep, atol=1e-14)
    np.testing.assert_allclose(lse, 0.3 * (q * krep).sum(-1), atol=1e-13)


def pin_constant_keys(lib):
    """All key rows equal: scores are constant along a row, so P is uniform
    over the visible keys: O_i = mean_{j<=i} V_j and LSE_i = s_i + ln(i+1).
    Every dS row then sums to zero against the same key, so dQ = 0."""
    r = _rng(3)
    T, D = 13, 6
    q = r.standard_normal((1, 2, T, D))
    k = np.broadcast_to(r.standard_normal((1, 1, 1, D)), (1, 1, T, D)).copy()
    v = r.standard_normal((1, 1, T, D))
    do = r.standard_normal((1, 2, T, D))
    res = oracle.bwd(q, k, v, do, causal=True, scale=0.5, lib=lib)
    prefix_mean = np.cumsum(v[0, 0], 0) / np.arange(1, T + 1)[:, None]
    for h in range(2):
        np.testing.assert_allclose(res["o"][0, h], prefix_mean, atol=1e-13)
        s = 0.5 * q[0, h] @ k[0, 0, 0]
        np.testing.assert_allclose(res["lse"][0, h], s + np.log(np.arange(1, T + 1)), atol=1e-12)
    np.testing.assert_allclose(res["dq"], 0.0, atol=1e-13)


def pin_shift_invariance(lib):
    """Adding u to every key shifts row i's scores by scale q_i.u, which the
    row softmax cancels: O is unchanged and LSE_i shifts by exactly that."""
    r = _rng(4)
    T, D = 11, 5
    q = r.standard_normal((1, 2, T, D))
    k = r.standard_normal((1, 1, T, D))
    v = r.standard_normal((1, 1, T, D))
    u = r.standard_normal(D)
    o1, l1 = oracle.fwd(q, k, v, causal=True, scale=0.8, lib=lib)
    o2, l2 = oracle.fwd(q, k + u, v, causal=True, scale=0.8, lib=lib)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 0.8 * (q @ u), atol=1e-12)


def pin_gqa_equals_repeated_mha(lib):
    """GQA equals MHA with each K/V head repeated G times (query head h uses
    key/value head h // G); dK, dV of GQA are the group sums of the MHA ones."""
    r = _rng(5)
    B, Hq, Hkv, T, D = 2, 6, 2, 10, 4
    G = Hq // Hkv
    q = r.standard_normal((B, Hq, T, D))
    k = r.standard_normal((B, Hkv, T, D))
    v = r.standard_normal((B, Hkv, T, D))
    do = r.standard_normal((B, Hq, T, D))
    g = oracle.bwd(q, k, v, do, causal=True, scale=0.4, lib=lib)
    m = oracle.bwd(q, np.repeat(k, G, 1), np.repeat(v, G, 1), do, causal=True, scale=0.4, lib=lib)
    for n in ("o", "lse", "dq"):
        np.testing.assert_allclose(g[n], m[n], atol=1e-12, err_msg=n)
    np.testing.assert_allclose(g["dk"], m["dk"].reshape(B, Hkv, G, T, D).sum(2), atol=1e-12)
    np.testing.assert_allclose(g["dv"], m["dv"].reshape(B, Hkv, G, T, D).sum(2), atol=1e-12)
    # MHA per head equals an independent single-head problem
    for h in range(Hq):
        o1, l1 = oracle.fwd(q[:, h:h + 1], k[:, h // G:h // G + 1], v[:, h // G:h // G + 1],
                            causal=True, scale=0.4, lib=lib)
        np.testing.assert_allclose(g["o"][:, h:h + 1], o1, atol=1e-12)


def pin_torch_sdpa(lib):
    """Special case that reduces to a library routine: PyTorch's
    scaled_dot_product_attention (math path, float64, CPU) and its autograd,
    with K/V repeated to full heads."""
    r = _rng(6)
    B, Hq, Hkv, T, D = 2, 4, 2, 17, 8
    G = Hq // Hkv
    q = r.standard_normal((B, Hq, T, D))
    k = r.standard_normal((B, Hkv, T, D))
    v = r.standard_normal((B, Hkv, T, D))
    do = r.standard_normal((B, Hq, T, D))
    for causal in (True, False):
        res = oracle.bwd(q, k, v, do, causal=causal, scale=0.35, lib=lib)
        tq = torch.tensor(q, requires_grad=True)
        tk = torch.tensor(k, requires_grad=True)
        tv = torch.tensor(v, requires_grad=True)
        with torch.nn.attention.sdpa_kernel(torch.nn.attention.SDPBackend.MATH):
            to = torch.nn.functional.scaled_dot_product_attention(
                tq, tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1), is_causal=causal, scale=0.35)
        to.backward(torch.tensor(do))
        np.testing.assert_allclose(res["o"], to.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(res["dq"], tq.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(res["dk"], tk.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(res["dv"], tv.grad.numpy(), atol=1e-12)


def pin_finite_differences(lib):
    """Central differences of L = sum(dO * O(Q,K,V)) in every element of Q, K
    and V match the backward (h = 1e-6, relative error < 1e-6)."""
    r = _rng(7)
    B, Hq, Hkv, T, D = 1, 2, 1, 5, 3
    q = r.standard_normal((B, Hq, T, D))
    k = r.standard_normal((B, Hkv, T, D))
    v = r.standard_normal((B, Hkv, T, D))
    do = r.standard_normal((B, Hq, T, D))
    scale = 0.6
    res = oracle.bwd(q, k, v, do, causal=True, scale=scale, lib=lib)

    def loss(q_, k_, v_):
        o, _ = oracle.fwd(q_, k_, v_, causal=True, scale=scale, lib=lib)
        return float((o * do).sum())

    h = 1e-6
    for name, x, grad in (("q", q, res["dq"]), ("k", k, res["dk"]), ("v", v, res["dv"])):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            lm = loss(args["q"], args["k"], args["v"])
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - grad).max() / max(np.abs(grad).max(), 1e-12)
        assert err < 1e-6, (name, err)


def pin_delta_identity(lib):
    """The backward's row term Delta_i = sum_j P_ij dP_ij equals sum_d dO_id O_id."""
    r = _rng(8)
    q = r.standard_normal((1, 2, 12, 6))
    k = r.standard_normal((1, 1, 12, 6))
    v = r.standard_normal((1, 1, 12, 6))
    do = r.standard_normal((1, 2, 12, 6))
    res = oracle.bwd(q, k, v, do, causal=True, scale=0.5, lib=lib)
    np.testing.assert_allclose(res["delta"], (res["o"] * do).sum(-1), atol=1e-12)


def pin_varlen_equals_slices(lib):
    """Packed variable length equals independent dense runs on each slice,
    including a length-1 and a zero-length sequence."""
    r = _rng(9)
    lens = [5, 1, 0, 9, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total, Hq, Hkv, D = int(cu[-1]), 4, 2, 5
    q = r.standard_normal((total, Hq, D))
    k = r.standard_normal((total, Hkv, D))
    v = r.standard_normal((total, Hkv, D))
    do = r.standard_normal((total, Hq, D))
    res = oracle.varlen_bwd(q, k, v, do, cu, causal=True, scale=0.45, lib=lib)
    o2, lse2 = oracle.varlen_fwd(q, k, v, cu, causal=True, scale=0.45, lib=lib)
    np.testing.assert_allclose(o2, res["o"], atol=1e-14)
    np.testing.assert_allclose(lse2, res["lse"], atol=1e-14)
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        if a == b:
            continue
        sl = lambda x: np.ascontiguousarray(x[a:b].transpose(1, 0, 2)[None])
        d = oracle.bwd(sl(q), sl(k), sl(v), sl(do), causal=True, scale=0.45, lib=lib)
        for n in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(res[n][a:b], d[n][0].transpose(1, 0, 2), atol=1e-12, err_msg=n)
        np.testing.assert_allclose(res["lse"][:, a:b], d["lse"][0], atol=1e-12)


def _bf16(x):
    return torch.tensor(x).to(torch.bfloat16).double().numpy()


def pin_rounding_error_terms(lib):
    """The backward's root-sum-square rounding-error scales (edq, edk, edv):
    lambda * u * e (lambda = 3, u = 2^-8) bounds, element by element, how far
    a computation moves that rounds P (for PV and P^T dO), the stored O (hence
    Delta) and dS to bf16 while accumulating exactly -- checked on a
    large-logit GQA case (observed worst ratio about 1.6)."""
    r = _rng(10)
    B, Hq, Hkv, T, D, scale = 1, 4, 2, 40, 16, 0.25
    G = Hq // Hkv
    q = _bf16(4.0 * r.standard_normal((B, Hq, T, D)))
    k = _bf16(r.standard_normal((B, Hkv, T, D)))
    v = _bf16(r.standard_normal((B, Hkv, T, D)))
    do = _bf16(r.standard_normal((B, Hq, T, D)))
    res = oracle.bwd(q, k, v, do, causal=True, scale=scale, lib=lib, err_terms=True)
    mask = np.tril(np.ones((T, T))) > 0
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in range(Hq):
        Q, K, V, dO = q[0, h], k[0, h // G], v[0, h // G], do[0, h]
        S = np.where(mask, scale * Q @ K.T, -np.inf)
        P = np.exp(S - S.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        O = _bf16(_bf16(P) @ V)                       # forward with bf16 P, stored in bf16
        delta = (dO * O).sum(1)
        dS = _bf16(P * (dO @ V.T - delta[:, None]))
        dq[0, h] = scale * dS @ K
        dk[0, h // G] += scale * dS.T @ Q
        dv[0, h // G] += _bf16(P).T @ dO
    u = 2.0 ** -8
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        err = np.abs(x - res[name])
        bound = 3.0 * u * res["e" + name] + 1e-12
        assert (err <= bound).all(), (name, float((err - bound).max()))
    assert float(np.abs(dk - res["dk"]).max()) > 1e-4    # the case does exercise rounding


def pin_decode_is_dense_suffix(lib):
    """Cached attention of the newest Tq positions equals the last Tq rows of
    dense causal attention over the row's first cache_lens[b] positions
    (reduction to the dense oracle), for every row and query head; a cache of
    one key gives O = V."""
    r = _rng(11)
    B, Hq, Hkv, Tq, S, D, scale = 3, 6, 2, 3, 21, 8, 0.3
    lens = [3, 21, 10]
    q_full = r.standard_normal((B, Hq, S, D))
    k = r.standard_normal((B, Hkv, S, D))
    v = r.standard_normal((B, Hkv, S, D))
    q = np.stack([q_full[b, :, lens[b] - Tq:lens[b]] for b in range(B)])
    o, lse = oracle.decode_fwd(q, k, v, lens, scale=scale, lib=lib)
    for b in range(B):
        L = lens[b]
        od, ld = oracle.fwd(q_full[b:b + 1, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L], causal=True, scale=scale,
                            lib=lib)
        np.testing.assert_allclose(o[b], od[0, :, L - Tq:L], atol=1e-12)
        np.testing.assert_allclose(lse[b], ld[0, :, L - Tq:L], atol=1e-12)
    o1, _ = oracle.decode_fwd(q[:, :, :1], k, v, [1, 1, 1], scale=scale, lib=lib)
    np.testing.assert_allclose(o1[:, :, 0], np.repeat(v[:, :, 0], Hq // Hkv, axis=1), atol=1e-14)


def pin_paged_decode_is_contiguous_decode(lib):
    """A cache scattered into shuffled pages (page sizes 1, 4 and the whole
    capacity; unused block-table entries pointing anywhere) gives the same
    result as the contiguous cache it came from."""
    r = _rng(12)
    B, Hq, Hkv, Tq, D, scale = 3, 4, 2, 2, 8, 0.4
    for psz in (1, 4, 24):
        maxp = 24 // psz
        S = maxp * psz
        lens = [S, 5, 2]
        q = r.standard_normal((B, Hq, Tq, D))
        k = r.standard_normal((B, Hkv, S, D))
        v = r.standard_normal((B, Hkv, S, D))
        order = r.permutation(B * maxp)               # page of (row b, slot i): order[b * maxp + i]
        kp = np.zeros((B * maxp, Hkv, psz, D))
        vp = np.zeros((B * maxp, Hkv, psz, D))
        bt = np.zeros((B, maxp), dtype=np.int64)
        for b in range(B):
            for i in range(maxp):
                pg = order[b * maxp + i]
                bt[b, i] = pg
                for h in range(Hkv):
                    for t in range(psz):
                        kp[pg, h, t] = k[b, h, i * psz + t]
                        vp[pg, h, t] = v[b, h, i * psz + t]
        for b in range(B):                           # entries past a row's pages may hold anything
            bt[b, (lens[b] + psz - 1) // psz:] = -7
        o, lse = oracle.paged_decode_fwd(q, kp, vp, bt, lens, scale=scale, lib=lib)
        oc, lc = oracle.decode_fwd(q, k, v, lens, scale=scale, lib=lib)
        np.testing.assert_array_equal(o, oc)
        np.testing.assert_array_equal(lse, lc)


def _rope_table(P, D, base=10000.0):
    i = np.arange(D // 2)
    ang = np.arange(P)[:, None] * base ** (-2.0 * i / D)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)


def pin_rope_decode(lib):
    """Rotary decode: position 0 leaves a query as it is and rotation keeps
    its norm; the scores depend only on relative position, so with keys
    rotated (here, in test code, by explicit 2x2 rotations) at their
    positions, shifting every position of a row by the same amount leaves
    O and LSE unchanged; a non-rotary query differs."""
    r = _rng(13)
    D = 8
    tab = _rope_table(400, D)
    x = r.standard_normal((5, D))
    np.testing.assert_allclose(oracle.rope_rotate(x, np.zeros(5, dtype=int), tab), x, atol=0)
    y = oracle.rope_rotate(x, np.array([1, 7, 50, 300, 399]), tab)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)

    def rotate_keys(k, start):          # [Hkv, L, D]: pair (i, i + D/2) turned by (start + j) * theta_i
        out = k.copy()
        for j in range(k.shape[1]):
            for i in range(D // 2):
                a = (start + j) * 10000.0 ** (-2.0 * i / D)
                c, s = np.cos(a), np.sin(a)
                lo, hi = k[:, j, i].copy(), k[:, j, i + D // 2].copy()
                out[:, j, i] = lo * c - hi * s
                out[:, j, i + D // 2] = hi * c + lo * s
        return out

    B, Hq, Hkv, Tq, L = 1, 4, 2, 2, 11
    q = r.standard_normal((B, Hq, Tq, D))
    k0 = r.standard_normal((B, Hkv, L, D))
    v = r.standard_normal((B, Hkv, L, D))
    outs = []
    for shift in (0, 37, 200):
        # the same keys, positions shifted: cache rows are positions shift .. shift + L - 1;
        # the table is indexed from position `shift` on by passing a table that starts there
        kr = rotate_keys(k0[0], shift)[None]
        tab_s = _rope_table(400, D)[shift:]
        outs.append(oracle.decode_fwd(q, kr, v, [L], scale=0.5, lib=lib, rope_cos_sin=tab_s))
        # positions in the table are relative to the cache start; rotate_keys used absolute shift + j,
        # tab_s[p] = table[shift + p]: both sides rotate by shift + position
    for o, l in outs[1:]:
        np.testing.assert_allclose(o, outs[0][0], atol=1e-12)
        np.testing.assert_allclose(l, outs[0][1], atol=1e-12)
    o_plain, _ = oracle.decode_fwd(q, rotate_keys(k0[0], 0)[None], v, [L], scale=0.5, lib=lib)
    assert np.abs(o_plain - outs[0][0]).max() > 1e-3


def pin_fp8_decode(lib):
    """E4M3 decoding matches PyTorch's float8_e4m3fn for all 256 codes (NaN
    codes included) and the worked values of the format (1.0, 448, 2^-9);
    FP8-cache decode equals decode over the decoded, scaled caches."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(mine[ok], ref[ok])
    assert mine[0x38] == 1.0 and mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0xB8] == -1.0
    r = _rng(14)
    B, Hq, Hkv, Tq, S, D = 2, 4, 2, 1, 9, 8
    q = r.standard_normal((B, Hq, Tq, D))
    k8 = r.integers(0, 0x7E, (B, Hkv, S, D)).astype(np.uint8) | (r.integers(0, 2, (B, Hkv, S, D)) << 7).astype(np.uint8)
    v8 = r.integers(0, 0x7E, (B, Hkv, S, D)).astype(np.uint8)
    lens = [9, 4]
    o, l = oracle.fp8_decode_fwd(q, k8, v8, 0.01, 0.02, lens, scale=0.3, lib=lib)
    o2, l2 = oracle.decode_fwd(q, mine[k8] * 0.01, mine[v8] * 0.02, lens, scale=0.3, lib=lib)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(l, l2)


def pin_rope_prefill(lib):
    """Rotary prefill (q and k rotated at positions 0..T-1 before attention):
    the transpose undoes the rotation; shifting every position by the same
    amount leaves O and LSE unchanged (the scores depend only on relative
    position) while dropping the rotation changes them; the backward through
    the rotation matches central finite differences of L = sum(dO * O) in the
    unrotated q and k; a packed variable-length batch equals dense runs on
    its slices (where each sequence's positions start is unobservable: only
    query-key position differences reach the scores)."""
    r = _rng(15)
    D, scale = 8, 0.4
    tab = _rope_table(64, D)
    x = r.standard_normal((3, 5, D))
    pos = r.integers(0, 64, (3, 5))
    np.testing.assert_allclose(oracle.rope_rotate_t(oracle.rope_rotate(x, pos, tab), pos, tab), x, atol=1e-13)
    B, Hq, Hkv, T = 2, 4, 2, 6
    q, do = r.standard_normal((B, Hq, T, D)), r.standard_normal((B, Hq, T, D))
    k, v = r.standard_normal((B, Hkv, T, D)), r.standard_normal((B, Hkv, T, D))
    o, l = oracle.rope_fwd(q, k, v, tab, scale=scale, lib=lib)
    o2, l2 = oracle.rope_fwd(q, k, v, tab[17:], scale=scale, lib=lib)   # every position + 17
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(l2, l, atol=1e-12)
    assert np.abs(oracle.fwd(q, k, v, scale=scale, lib=lib)[0] - o).max() > 1e-3
    g = oracle.rope_bwd(q, k, v, do, tab, scale=scale, lib=lib)
    np.testing.assert_allclose(g["o"], o, atol=1e-13)

    def loss(qq, kk, vv):
        return float((do * oracle.rope_fwd(qq, kk, vv, tab, scale=scale, lib=lib)[0]).sum())

    eps = 1e-6
    for name, which in (("dq", 0), ("dk", 1), ("dv", 2)):
        base = [q, k, v][which]
        for idx in list(np.ndindex(base.shape))[::5]:
            args_p = [q, k, v]
            a = base.copy()
            a[idx] += eps
            args_p[which] = a
            lp = loss(*args_p)
            a[idx] -= 2 * eps
            lm = loss(*args_p)
            num = (lp - lm) / (2 * eps)
            assert abs(num - g[name][idx]) <= 1e-6 * (1 + abs(num)), (name, idx, num, g[name][idx])
    cu = [0, 5, 6, 13]
    qv, dov = r.standard_normal((13, Hq, D)), r.standard_normal((13, Hq, D))
    kv, vv = r.standard_normal((13, Hkv, D)), r.standard_normal((13, Hkv, D))
    ov, lv = oracle.rope_varlen_fwd(qv, kv, vv, cu, tab, scale=scale, lib=lib)
    gv = oracle.rope_varlen_bwd(qv, kv, vv, dov, cu, tab, scale=scale, lib=lib)
    dense = lambda t: np.ascontiguousarray(t.transpose(1, 0, 2)[None])
    for a, b in zip(cu[:-1], cu[1:]):
        od, ld = oracle.rope_fwd(dense(qv[a:b]), dense(kv[a:b]), dense(vv[a:b]), tab, scale=scale, lib=lib)
        np.testing.assert_allclose(ov[a:b], od[0].transpose(1, 0, 2), atol=1e-13)
        np.testing.assert_allclose(lv[:, a:b], ld[0], atol=1e-13)
        gd = oracle.rope_bwd(dense(qv[a:b]), dense(kv[a:b]), dense(vv[a:b]), dense(dov[a:b]), tab, scale=scale,
                             lib=lib)
        for n in ("dq", "dk", "dv"):
            np.testing.assert_allclose(gv[n][a:b], gd[n][0].transpose(1, 0, 2), atol=1e-12)


PINS = [pin_hand_worked, pin_rows_sum_to_one, pin_single_token, pin_constant_keys, pin_shift_invariance,
        pin_gqa_equals_repeated_mha, pin_torch_sdpa, pin_finite_differences, pin_delta_identity,
        pin_varlen_equals_slices, pin_rounding_error_terms, pin_decode_is_dense_suffix,
        pin_paged_decode_is_contiguous_decode, pin_rope_decode, pin_fp8_decode, pin_rope_prefill]
