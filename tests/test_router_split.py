"""The prompt router's three-way bf16 split, checked on the host.

At load time the fp32 router weights become three bf16 parts: hi = bf16(w),
mid = bf16(w - hi), lo = bf16(w - hi - mid), each rounded to nearest even,
the differences taken in fp32.  The tensor-core router multiplies bf16 x by
each part (an 8-bit by 8-bit significand product, exact in fp32) and sums in
fp32, which needs w = hi + mid + lo exactly.  That holds while lo's lowest
bit stays above bf16's smallest subnormal, i.e. for |w| >= 2^-110 or so;
router weights are nowhere near that small.  This test restates the split
with PyTorch's bf16 cast (round to nearest even) and checks it.
"""
import numpy as np
import torch


def bf16(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16).float().numpy()


def split(w: np.ndarray):
    hi = bf16(w)
    r1 = (w - hi).astype(np.float32)
    mid = bf16(r1)
    lo = bf16((r1 - mid).astype(np.float32))
    return hi, mid, lo


def test_split_is_exact_over_the_fp32_range():
    rng = np.random.default_rng(0)
    n = 4_000_000
    bits = rng.integers(0, 1 << 23, n, dtype=np.uint32)          # every mantissa pattern
    exp = rng.integers(127 - 100, 127 + 100, n).astype(np.uint32)  # 2^-100 .. 2^100
    sign = rng.integers(0, 2, n).astype(np.uint32) << np.uint32(31)
    w = (sign | (exp << np.uint32(23)) | bits).view(np.float32)
    hi, mid, lo = split(w)
    total = hi.astype(np.float64) + mid.astype(np.float64) + lo.astype(np.float64)
    assert np.array_equal(total, w.astype(np.float64))


def test_router_scale_weights():
    """Weights drawn as the router's are (N(0, 0.02)), including exact zeros."""
    rng = np.random.default_rng(1)
    w = (0.02 * rng.standard_normal(2_000_000)).astype(np.float32)
    w[::1000] = 0.0
    hi, mid, lo = split(w)
    assert np.array_equal(hi.astype(np.float64) + mid + lo, w.astype(np.float64))


def test_products_with_bf16_inputs_are_exact_in_fp32():
    rng = np.random.default_rng(2)
    x = bf16(rng.standard_normal(1_000_000).astype(np.float32))
    w = (0.02 * rng.standard_normal(1_000_000)).astype(np.float32)
    for part in split(w):
        p32 = (x * part).astype(np.float32).astype(np.float64)
        assert np.array_equal(p32, x.astype(np.float64) * part.astype(np.float64))


def test_the_limit_is_real():
    """Far below 2^-110 the low part no longer fits: the documented limit."""
    w = np.float32([np.float32(1.2345678) * np.float32(2.0 ** -125)])
    hi, mid, lo = split(w)
    assert float(hi[0]) + float(mid[0]) + float(lo[0]) != float(w[0])
