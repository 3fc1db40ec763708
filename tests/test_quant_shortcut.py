"""The activation quantisation's shortcut, checked on the host.

The kernels take each e4m3 code from the product q = v * y, with y the
hardware's approximate reciprocal of the group scale s, instead of from the
IEEE quotient Q = v / s.  They send a group to the exact division whenever a
product is "undecided": its low 20 mantissa bits lie within 8 of 0x80000 (an
e4m3 rounding midpoint in e4m3's normal range), or |q| is below 2^-6 (e4m3's
subnormal range), or s's exponent field is outside [2, 252].  The claim is
that every product not flagged rounds to the same code as Q.

This test restates that rule in numpy and checks the claim for reciprocals up
to two ulps from the correctly rounded 1/s (the approximate reciprocal's error
is below that), over random groups and over values placed next to every
e4m3 midpoint.  The reference rounding is PyTorch's float8_e4m3fn cast of the
quotient clamped to +-448 (the kernels' conversion saturates).
"""
import numpy as np
import torch


def undecided(q: np.ndarray) -> np.ndarray:
    u = q.view(np.uint32) & np.uint32(0x7FFFFFFF)
    tiny = (u - np.uint32(1)) < np.uint32(0x3C800000 - 1)
    near_mid = ((u & np.uint32(0xFFFFF)) - np.uint32(0x7FFF8)) < np.uint32(16)
    return tiny | near_mid


def e4m3_codes(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.clip(v, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def shifted(y: np.ndarray, k: int) -> np.ndarray:
    """y moved k float32 steps (y > 0, away from the ends of the range)."""
    return (y.view(np.uint32).astype(np.int64) + k).astype(np.uint32).view(np.float32)


def check(v: np.ndarray, s: np.ndarray):
    """v, s float32 of the same shape; returns how many products were decided."""
    Q = (v.astype(np.float64) / s.astype(np.float64)).astype(np.float32)  # IEEE quotient
    want = e4m3_codes(Q)
    es = (s.view(np.uint32) >> np.uint32(23)) & np.uint32(0xFF)
    s_ok = (es >= 2) & (es <= 252)
    y0 = (1.0 / s.astype(np.float64)).astype(np.float32)
    decided = 0
    for k in (-2, -1, 0, 1, 2):
        q = (v * shifted(y0, k)).astype(np.float32)
        ok = s_ok & ~undecided(q)
        got = e4m3_codes(q)
        bad = np.nonzero(ok & (got != want))[0]
        assert bad.size == 0, (v[bad[:4]], s[bad[:4]], k)
        decided += int(ok.sum())
    return decided


def test_random_groups():
    rng = np.random.default_rng(0)
    n = 2_000_000
    amax = np.exp2(rng.uniform(-20, 20, n)).astype(np.float32)
    s = (amax.astype(np.float64) / 448.0).astype(np.float32)
    # values spread over twelve binades below the group amax, both signs,
    # rounded to bf16 for half of them (x is bf16; the SwiGLU rows are fp32)
    mag = amax * np.exp2(-rng.uniform(0, 12, n)).astype(np.float32)
    v = (mag * rng.choice([-1.0, 1.0], n)).astype(np.float32)
    half = rng.random(n) < 0.5
    v[half] = torch.from_numpy(v[half]).to(torch.bfloat16).float().numpy()
    v[::97] = amax[::97]  # the group maximum itself (code 0x7E)
    assert check(v, s) > 0.99 * 5 * n


def test_next_to_every_midpoint():
    """Quotients a few ulps either side of each e4m3 midpoint, for scales of
    many binades: the flagged window must cover every product that could
    round across the midpoint."""
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mags = np.unique(np.abs(table[np.isfinite(table)]))
    mids = 0.5 * (mags[:-1] + mags[1:])
    rng = np.random.default_rng(1)
    scales = np.exp2(rng.uniform(-30, 30, 64)).astype(np.float32)
    vs, ss = [], []
    for s in scales:
        for d in range(-12, 13):
            target = (mids * float(s)).astype(np.float32)
            v = (target.view(np.uint32).astype(np.int64) + d).astype(np.uint32).view(np.float32)
            vs.append(v)
            ss.append(np.full(v.size, s, np.float32))
    v = np.concatenate(vs)
    s = np.concatenate(ss)
    v = np.concatenate([v, -v])
    s = np.concatenate([s, s])
    check(v, s)


def test_window_is_needed():
    """Without the midpoint window some products round the other way, so the
    test above can see a mistake in it."""
    s = np.float32(1.0 / 3.0)
    y = shifted(np.array([1.0 / s], np.float32), 2)[0]
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mags = np.unique(np.abs(table[np.isfinite(table)]))
    mids = 0.5 * (mags[:-1] + mags[1:])
    target = (mids * float(s)).astype(np.float32)
    flips = 0
    for d in range(-3, 4):
        v = (target.view(np.uint32).astype(np.int64) + d).astype(np.uint32).view(np.float32)
        Q = (v.astype(np.float64) / float(s)).astype(np.float32)
        q = (v * y).astype(np.float32)
        flips += int(np.sum(e4m3_codes(q) != e4m3_codes(Q)))
    assert flips > 0
