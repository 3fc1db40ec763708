"""The decode kernels' two-level top-k, restated on the host.

For one row of E <= 32 * W fp32 logits (W warps of 32 experts), the kernels:
  1. map each logit to an order-preserving 32-bit key (-0 folded into +0;
     experts past E get key 0, below every real key);
  2. rank every expert within its warp by counting the keys there that beat
     it (larger, or equal with a lower index) and write the k best of each
     warp to slots [warp][rank];
  3. rank every candidate among all W * k candidates the same way and write
     the candidates ranked below k to the result, in rank order.
The claim is that this equals the k largest logits with ties to the lower
expert, in rank order, for every k <= 8 and k <= E.  This test restates the
three steps with numpy and compares them with a full stable sort on rows
full of ties, signed zeros and partially filled warps.
"""
import numpy as np
import pytest


def order_key(v: np.ndarray) -> np.ndarray:
    u = (v.astype(np.float32) + np.float32(0.0)).view(np.uint32)
    return np.where(u & np.uint32(0x80000000), ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def beats(ka, ia, kb, ib):
    return (ka > kb) | ((ka == kb) & (ia < ib))


def two_level(lg: np.ndarray, k: int, warps: int) -> list:
    E = lg.size
    n = 32 * warps
    keys = np.zeros(n, np.uint32)
    keys[:E] = order_key(lg)
    ids = np.arange(n)
    cand = {}
    for w in range(warps):
        kw, iw = keys[32 * w:32 * w + 32], ids[32 * w:32 * w + 32]
        for lane in range(32):
            r = int(np.sum(beats(kw, np.arange(32), kw[lane], lane)))
            if r < k:
                assert (w, r) not in cand
                cand[(w, r)] = (int(kw[lane]), int(iw[lane]))
    assert len(cand) == warps * k  # every slot below k is written
    ck = np.array([cand[(w, s)][0] for w in range(warps) for s in range(k)], np.uint64)
    ci = np.array([cand[(w, s)][1] for w in range(warps) for s in range(k)])
    out = [None] * k
    for K, D in zip(ck, ci):
        rank = int(np.sum(beats(ck, ci, K, D)))
        if rank < k:
            assert out[rank] is None
            out[rank] = int(D)
    return out


def full_sort(lg: np.ndarray, k: int) -> list:
    v = lg.astype(np.float32).astype(np.float64) + 0.0
    return [int(e) for e in np.lexsort((np.arange(lg.size), -v))[:k]]


def rows(rng, E):
    yield rng.standard_normal(E).astype(np.float32)
    yield rng.choice(np.float32([-1.0, 0.0, 0.5, 2.0]), E)          # heavy ties
    yield np.zeros(E, np.float32)                                     # all equal
    z = rng.choice(np.float32([0.0, -0.0, 1.0, -1.0]), E)             # signed zeros
    yield z
    yield np.float32(np.round(rng.standard_normal(E) * 4) / 4)       # coarse values
    big = rng.standard_normal(E).astype(np.float32) * np.float32(1e30)
    big[rng.integers(0, E, 3)] = -np.finfo(np.float32).max
    yield big


@pytest.mark.parametrize("E", [8, 16, 40, 100, 255, 256])
def test_two_level_equals_full_sort(E):
    rng = np.random.default_rng(E)
    for k in (1, 2, 4, 7, 8):
        if k > E:
            continue
        for lg in rows(rng, E):
            assert two_level(lg, k, 8) == full_sort(lg, k), (E, k, lg[:8])


def test_padding_keys_lose_to_every_real_key():
    extremes = np.float32([-np.inf, -np.finfo(np.float32).max, -1e-45, -0.0, 0.0])
    assert np.all(order_key(extremes) > 0)
    assert order_key(np.float32([-0.0]))[0] == order_key(np.float32([0.0]))[0]
