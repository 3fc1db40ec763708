"""The layer taking the residual stream and the preceding block's output
(moe_forward_addnorm) against the oracle's add-norm followed by the oracle's
layer, through the C ABI (needs a GB300).

The pages fuse the residual add and RMS norm with the experts' FP8
activation quantisation (PR #925/#927 commit "add-norm fused with the routed
experts' FP8 activation quantization").  Here one row runs as one kernel,
the add-norm inside the layer's first pass; more rows run the add-norm kernel
and the grouped path scatters its codes.  The bars:
  - h bit for bit (one bf16 add);
  - xn within one bf16 ulp everywhere and identical in all but 1e-3 of the
    elements (the norm's fp32 sum of squares runs in another order than the
    oracle's double);
  - the codes and scales the experts read equal the oracle's quantisation of
    the GPU's own xn, bit for bit, for every (row, rank);
  - top-k, weights and y as for moe_forward, against the oracle's layer on
    the GPU's xn, and y also within the bar against the oracle's layer on the
    oracle's xn.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import bits, check_forward_codes, check_output, check_topk, oracle_rows

pytestmark = pytest.mark.gpu

m = pytest.importorskip("block_fp8_mixture_router_gb300")

from test_gpu_parity import Case  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    return torch.device("cuda", 0)


def _ulps_bf16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, -(u & 0x7FFF), u)
    return np.abs(ordered(a_bits) - ordered(b_bits))


@pytest.mark.parametrize("name,rows", [("decode_t1", 1), ("decode_t11", 11),
                                       ("prompt_t1024", 1024)])
def test_forward_addnorm_against_oracle(dev, name, rows):
    case = Case(W.WORKLOADS[name], max(rows, 16), dev)
    r, x, g = (t.to(dev) for t in W.make_addnorm(W.FULL, rows, 5100 + rows))
    h, xn, y = case.moe.forward_addnorm(r, x, g, W.NORM_EPS, keep_xn=True)
    fc, fs = case.moe.forward_codes(rows)
    idx, w = case.moe.route(xn)
    torch.cuda.synchronize()
    rh, rxn, _, _ = oracle.add_rmsnorm(bits(r), bits(x), bits(g), W.NORM_EPS)
    assert np.array_equal(bits(h), rh)
    d = _ulps_bf16(bits(xn), rxn)
    assert d.max() <= 1 and np.mean(d > 0) <= 1e-3, (int(d.max()), float(np.mean(d > 0)))
    # the layer on the GPU's own normed rows
    ref = oracle_rows(case.host, bits(xn), trace=True)
    check_forward_codes(fc.cpu().numpy(), fs.cpu().numpy(), ref.trace["xq"], ref.trace["sx"])
    near, differ = check_topk(idx.cpu().numpy(), ref.trace["logits"], W.FULL.top_k)
    assert differ.sum() <= max(1, 0.02 * rows)
    assert np.allclose(w.cpu().numpy()[~differ], ref.trace["w"][~differ], rtol=2e-5, atol=1e-7)
    check_output(bits(y), ref.y_ref, rows_mask=~differ)
    # and on the oracle's normed rows
    ref2 = oracle_rows(case.host, rxn)
    check_output(bits(y), ref2.y_ref, rows_mask=~differ)
    case.moe.close()


@pytest.mark.parametrize("rows", [1, 11, 300])
def test_forward_addnorm_equals_add_norm_then_forward(dev, rows):
    """The fused call gives what the add-norm entry point followed by
    moe_forward gives on the same inputs, bit for bit wherever the two
    normed rows agree (always above one row: the same add-norm kernel)."""
    case = Case(W.WORKLOADS["decode_t1"], 512, dev)
    r, x, g = (t.to(dev) for t in W.make_addnorm(W.FULL, rows, 5200 + rows))
    h1, xn1, y1 = case.moe.forward_addnorm(r, x, g, W.NORM_EPS, keep_xn=True)
    h2, xn2, _, _ = case.moe.add_rmsnorm_quantize(r, x, g, W.NORM_EPS)
    y2 = case.moe.forward(xn2)
    _, _, y3 = case.moe.forward_addnorm(r, x, g, W.NORM_EPS)  # without keeping xn
    torch.cuda.synchronize()
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    same = torch.all(xn1.view(torch.int16) == xn2.view(torch.int16), dim=1)
    if rows > 1:
        assert bool(same.all())
    assert torch.equal(y1[same].view(torch.int16), y2[same].view(torch.int16))
    case.moe.close()


def test_forward_addnorm_refusals(dev):
    case = Case(W.WORKLOADS["decode_t1"], 16, dev)
    ctx = case.moe.ctx
    r, x, g = (t.to(dev) for t in W.make_addnorm(W.FULL, 2, 5300))
    h, xn, y = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
    eps = W.NORM_EPS
    assert m.moe_forward_addnorm(ctx, r, x, g, eps, 2, h, xn, y) == m.MOE_OK
    assert m.moe_forward_addnorm(ctx, r, x, g, eps, 2, r, xn, y) == m.MOE_ERR_INVALID_ARG
    assert m.moe_forward_addnorm(ctx, r, x, g, eps, 2, h, h, y) == m.MOE_ERR_INVALID_ARG
    assert m.moe_forward_addnorm(ctx, r, x, g, eps, 2, h, xn, x) == m.MOE_ERR_INVALID_ARG
    assert m.moe_forward_addnorm(ctx, r, x, g, -1.0, 2, h, xn, y) == m.MOE_ERR_INVALID_ARG
    assert m.moe_forward_addnorm(ctx, r, x, g, float("nan"), 2, h, xn, y) == \
        m.MOE_ERR_INVALID_ARG
    assert m.moe_forward_addnorm(ctx, r, x, g, eps, 17, h, xn, y) == \
        m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_forward_addnorm(ctx, r, x, g, eps, 0, None, None, None) == m.MOE_OK
    assert m.moe_forward_addnorm(ctx, r, x, g, eps, 2, None, xn, y) == m.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert case.moe.device_status() == m.MOE_OK
    case.moe.close()
