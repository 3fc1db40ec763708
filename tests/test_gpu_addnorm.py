"""Residual add + RMS norm + FP8 groups (moe_add_rmsnorm_quantize) against the
CPU oracle, through the C ABI (needs a GB300).

The kernel computes the norm in fp32 (sum of squares, 1/sqrt, h * r * gamma)
and the oracle in double, so the value each bf16 rounding of xn sees differs
by about 1e-6 relative: a normed value may land one bf16 ulp away where it
sits that close to a rounding midpoint, about one element in 10^4.  The bars:
  - h (one bf16 add) bit for bit;
  - xn within one bf16 ulp everywhere, and identical in all but 1e-3 of the
    elements;
  - codes and scales bit for bit in every group whose xn agrees bit for bit,
    and elsewhere each code within one e4m3 step and each scale within a bf16
    ulp (the group's amax moved by at most one ulp);
  - codes and scales bit for bit equal to moe_quantize of the kernel's own xn,
    the separate quantisation launch the fused one replaces.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import bits

pytestmark = pytest.mark.gpu

m = pytest.importorskip("block_fp8_mixture_router_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    return torch.device("cuda", 0)


def _ctx(shape: W.MoEShape, dev, load: bool = True):
    """A context, with a layer loaded by default: the add-norm itself needs no
    weights, but the comparison with moe_quantize (which also forms the shared
    gate) does."""
    c = m.MoELayer(m.LayerShape(shape.hidden, shape.n_experts, shape.top_k, shape.inter,
                                shape.shared_inter, shape.group), max_rows=1024)
    if load:
        c.load(W.make_layer(shape, 1, device=dev, experts=[0]))
    return c


@pytest.fixture(scope="module")
def full_ctx(dev):
    c = _ctx(W.FULL, dev)
    yield c
    c.close()


@pytest.fixture(scope="module")
def tiny_ctx(dev):
    c = _ctx(W.TINY, dev)
    yield c
    c.close()


def _ulps_bf16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 steps between same-sign finite bf16 values (sign-magnitude)."""
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def check_addnorm(ctx, residual, x, gamma, eps, out):
    h, xn, codes, scales = [t.cpu() for t in out]
    rh, rxn, rc, rs = oracle.add_rmsnorm(bits(residual), bits(x), bits(gamma), eps)
    assert np.array_equal(bits(h), rh)
    gx = bits(xn)
    d = _ulps_bf16(gx, rxn)
    assert d.max() <= 1, d.max()
    assert (d > 0).mean() <= 1e-3, (d > 0).mean()
    T, H = gx.shape
    G = 128
    same_group = (d.reshape(T, H // G, G) == 0).all(-1)
    gc, gs = codes.numpy(), scales.numpy()
    gcg = gc.reshape(T, H // G, G)
    rcg = rc.reshape(T, H // G, G)
    assert np.array_equal(gcg[same_group], rcg[same_group])
    assert np.array_equal(gs[same_group], rs[same_group])
    if (~same_group).any():
        step = np.abs((gcg[~same_group] & 0x7F).astype(int) - (rcg[~same_group] & 0x7F))
        assert step.max() <= 1
        ratio = gs[~same_group] / rs[~same_group]
        assert np.all(np.abs(ratio - 1) <= 2.0 ** -8)
    # the same codes as the separate quantisation of the kernel's own bf16 rows
    if ctx is not None:
        qc, qs = ctx.quantize(out[1])
        torch.cuda.synchronize()
        assert np.array_equal(qc.cpu().numpy(), gc) and np.array_equal(qs.cpu().numpy(), gs)
    return int((d > 0).sum()), int((~same_group).sum())


@pytest.mark.parametrize("rows", [1, 11, 1024])
def test_addnorm_full(full_ctx, rows):
    r, x, g = W.make_addnorm(W.FULL, rows, 40 + rows, device="cuda")
    out = full_ctx.add_rmsnorm_quantize(r, x, g, W.NORM_EPS)
    torch.cuda.synchronize()
    n_el, n_gr = check_addnorm(full_ctx, r, x, g, W.NORM_EPS, out)
    print(f"rows={rows}: {n_el} xn elements one ulp apart, {n_gr} groups touched")


@pytest.mark.parametrize("rows", [3, 17])
def test_addnorm_tiny(tiny_ctx, rows):
    r, x, g = W.make_addnorm(W.TINY, rows, 7, device="cuda")
    out = tiny_ctx.add_rmsnorm_quantize(r, x, g, 1e-5)
    torch.cuda.synchronize()
    check_addnorm(tiny_ctx, r, x, g, 1e-5, out)


@pytest.mark.parametrize("hidden", [2560, 3072, 4096, 6144, 8192])
def test_addnorm_wide_rows(dev, hidden):
    """Rows wider than 2048 take two or four chunks per thread; 2560, 3072
    and 6144 leave the last chunk slot of some threads idle (a context with
    no weights: the add-norm needs none, so only the oracle is compared)."""
    shape = W.MoEShape(hidden=hidden, n_experts=16, top_k=4, inter=128, shared_inter=128)
    ctx = _ctx(shape, dev, load=False)
    try:
        r, x, g = W.make_addnorm(shape, 37, 11, device="cuda")
        out = ctx.add_rmsnorm_quantize(r, x, g, W.NORM_EPS)
        torch.cuda.synchronize()
        check_addnorm(None, r, x, g, W.NORM_EPS, out)
    finally:
        ctx.close()


def test_addnorm_in_place(full_ctx):
    """h_out = residual and xn_out = x give the out-of-place results."""
    r, x, g = W.make_addnorm(W.FULL, 64, 5, device="cuda")
    ref = [t.clone() for t in full_ctx.add_rmsnorm_quantize(r, x, g, W.NORM_EPS)]
    r2, x2 = r.clone(), x.clone()
    out = full_ctx.add_rmsnorm_quantize(r2, x2, g, W.NORM_EPS, h_out=r2, xn_out=x2)
    torch.cuda.synchronize()
    assert out[0].data_ptr() == r2.data_ptr() and out[1].data_ptr() == x2.data_ptr()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
    # the other way round: the new residual into x's buffer, xn into residual's
    r3, x3 = r.clone(), x.clone()
    out = full_ctx.add_rmsnorm_quantize(r3, x3, g, W.NORM_EPS, h_out=x3, xn_out=r3)
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)


def test_addnorm_degenerate_rows(full_ctx):
    """A zero row, a row whose residual cancels x, a constant row and a row of
    large values; eps > 0 keeps the zero rows finite (xn = 0, scale 1)."""
    r, x, g = W.make_addnorm(W.FULL, 4, 9, device="cuda")
    r[0] = 0
    x[0] = 0
    x[1] = -r[1]
    r[2] = 3.0
    x[2] = 0.5
    r[3] = r[3] * 4096
    out = full_ctx.add_rmsnorm_quantize(r, x, g, W.NORM_EPS)
    torch.cuda.synchronize()
    check_addnorm(full_ctx, r, x, g, W.NORM_EPS, out)
    h, xn, codes, scales = [t.cpu() for t in out]
    for t in (0, 1):
        assert not h[t].any() and not xn[t].any() and not codes[t].any()
        assert torch.all(scales[t] == 1.0)
    # constant row: xn = gamma * 3.5 / sqrt(3.5^2 + eps), within one ulp of gamma
    assert np.all(_ulps_bf16(bits(xn[2:3])[0], bits(g.cpu()[None])[0]) <= 1)


def test_addnorm_zero_rows_and_refusals(full_ctx):
    H = W.FULL.hidden
    r, x, g = W.make_addnorm(W.FULL, 8, 3, device="cuda")
    h = torch.empty_like(x)
    xn = torch.empty_like(x)
    codes = torch.empty((8, H), dtype=torch.uint8, device="cuda")
    scales = torch.empty((8, H // 128), dtype=torch.float32, device="cuda")
    call = lambda *a, **k: m.moe_add_rmsnorm_quantize(full_ctx.ctx, *a, **k)  # noqa: E731
    assert call(r, x, g, 1e-6, 0, h, xn, codes, scales) == m.MOE_OK
    assert call(r, x, g, -1.0, 8, h, xn, codes, scales) == m.MOE_ERR_INVALID_ARG
    assert call(r, x, g, float("nan"), 8, h, xn, codes, scales) == m.MOE_ERR_INVALID_ARG
    assert call(r, x, g, 1e-6, -1, h, xn, codes, scales) == m.MOE_ERR_INVALID_ARG
    assert call(r, x, None, 1e-6, 8, h, xn, codes, scales) == m.MOE_ERR_INVALID_ARG
    # outputs overlapping each other or a row input other than in place
    assert call(r, x, g, 1e-6, 8, h, h, codes, scales) == m.MOE_ERR_INVALID_ARG
    # (a nine-row buffer, so that the shifted output stays inside it either way)
    r9 = torch.cat([r, r[:1]])
    assert call(r9[:8], x, g, 1e-6, 8, r9[1:], xn, codes, scales) == m.MOE_ERR_INVALID_ARG
    assert call(r, x, g, 1e-6, 8, h, xn, codes, h) == m.MOE_ERR_INVALID_ARG
    # a bf16 pointer off the 16-byte grid
    off = ctypes.c_void_p(x.data_ptr() + 2)
    assert m.load_library().moe_add_rmsnorm_quantize(
        full_ctx.ctx, ctypes.c_void_p(r.data_ptr()), off, ctypes.c_void_p(g.data_ptr()),
        ctypes.c_float(1e-6), 4, ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(xn.data_ptr()),
        ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(scales.data_ptr()),
        None) == m.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
