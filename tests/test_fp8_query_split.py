"""Precision of the three-part E4M3 query split used by the FP8 decode score
MMA, checked on the CPU.

Each query row q is carried as s (h0 + h1 + h2) with s = max|q| / 448 and,
for x = q / s, h0 = e4m3(x), h1 = e4m3(x - h0), h2 = e4m3(x - h0 - h1)
(round to nearest even).  One E4M3 rounding is off by at most 2^-4 of its
argument in the normal range and by at most 2^-10 (half the 2^-9 subnormal
step) below it, so three leave max(2^-12 |q|, 2^-10 max|q| / 448).  The
split is replayed here with PyTorch's float8_e4m3fn cast, which rounds the
same way.
"""
import numpy as np
import torch


def e4m3(x):
    return torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def split(q):
    amax = np.abs(q).max(axis=-1, keepdims=True)
    s = np.where(amax > 0, amax / 448.0, 1.0)
    x = (q / s).astype(np.float32).astype(np.float64)   # the kernel scales in f32
    parts = []
    for _ in range(3):
        h = e4m3(x)
        parts.append(h)
        x = x - h
    return s, parts


def test_three_parts_hold_q_to_the_stated_bound():
    r = np.random.default_rng(5)
    rows = [r.standard_normal((64, 128)),
            r.standard_normal((64, 128)) * np.exp(r.uniform(-12, 6, (64, 1))),   # any row scale
            r.standard_cauchy((64, 128)),                                         # heavy tails
            np.concatenate([r.standard_normal((64, 4)) * 1e3, r.standard_normal((64, 124)) * 1e-4], axis=1)]
    for q in rows:
        q = q.astype(np.float32).astype(np.float64)
        s, parts = split(q)
        for h in parts:
            assert np.all(np.abs(h) <= 448.0) and not np.isnan(h).any()
        err = np.abs(q - s * sum(parts))
        amax = np.abs(q).max(axis=-1, keepdims=True)
        bound = np.maximum(2.0 ** -12 * np.abs(q), 2.0 ** -10 * amax / 448.0)
        # the f32 scaling of q / s adds up to one f32 rounding of x (2^-24 relative)
        assert np.all(err <= bound * (1 + 1e-6) + 2.0 ** -23 * np.abs(q))


def test_one_or_two_parts_are_not_enough():
    """The third part matters: two parts leave errors near 2^-8 |q|."""
    q = np.random.default_rng(6).standard_normal((256, 128))
    s, parts = split(q)
    rel2 = np.abs(q - s * (parts[0] + parts[1])) / np.abs(q)
    rel3 = np.abs(q - s * sum(parts)) / np.abs(q)
    big = np.abs(q) > 0.25 * np.abs(q).max(axis=-1, keepdims=True)
    assert rel2[big].max() > 2.0 ** -11
    assert rel3[big].max() <= 2.0 ** -12 * (1 + 1e-6) + 2.0 ** -23
