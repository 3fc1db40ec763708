"""The router and quantisation variants the pages describe, against the
oracle's variants (needs a GB300).

- One activation scale per row (act_group == hidden): the literal reading of
  "dynamic per-row" activations, beside PR #939's "per row and per 128
  inputs" (section "Precision"), which stays the default.  Each row of x and
  each routed SwiGLU row takes one scale, amax / 448; the codes the forward
  feeds its experts must equal the oracle's per-row variant bit for bit.
- Router on bf16 logits (MOE_OPT_ROUTER_BF16): PR #939 ("drama3: Fish Audio
  Drama 3 text to speech on one CUDA GPU"), section "Fidelity against the
  PyTorch oracle": the reference's bf16 oracle routes on bf16 logits, where
  the 8th and 9th experts tie exactly.  The rows of the oracle's own pin meet
  such ties; the lower expert must come first, with no near-tie slack where
  the rounding to bf16 is unambiguous.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import bits, check_forward_codes, check_output, check_topk_bf16, oracle_rows
from test_gpu_parity import Case, run_and_check

pytestmark = pytest.mark.gpu

m = pytest.importorskip("block_fp8_mixture_router_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    return torch.device("cuda", 0)


def _net(layer, s, max_rows):
    net = m.MoELayer(m.LayerShape(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter,
                                  s.group), max_rows=max_rows)
    net.load(layer)
    return net


@pytest.fixture(scope="module")
def bf16_layer(dev):
    """The full-width layer whose router is the one of the oracle's bf16 pin
    (drawn on the host, as the pin draws it)."""
    s = W.FULL
    layer = W.make_layer(s, 21, device=dev)
    layer["router"] = W.make_router(s, 21).to(dev)
    net = _net(layer, s, 1024)
    host = W.to_numpy_layer(layer)
    yield layer, net, host
    net.close()


def _check_bf16(net, host, x, path, k):
    net.set_option(m.MOE_OPT_PATH, path)
    net.set_option(m.MOE_OPT_ROUTER_BF16, 1)
    try:
        T = x.shape[0]
        y = net.forward(x)
        fc, fs = net.forward_codes(T)
        idx, w = net.route(x)
        torch.cuda.synchronize()
    finally:
        net.set_option(m.MOE_OPT_ROUTER_BF16, 0)
        net.set_option(m.MOE_OPT_PATH, m.PATH_AUTO)
    xb = bits(x)
    ref = oracle_rows(host, xb, trace=True, router_bf16=True)
    lg64 = np.stack([oracle.router_row(xb[t], host["router"], k)[0] for t in range(T)])
    amb, differ = check_topk_bf16(idx.cpu().numpy(), lg64, k)
    assert differ.sum() <= max(1, 0.02 * T), differ.sum()
    same = ~amb
    assert np.array_equal(idx.cpu().numpy()[same], ref.trace["idx"][same])
    assert np.allclose(w.cpu().numpy()[same], ref.trace["w"][same], rtol=2e-5, atol=1e-7)
    check_forward_codes(fc.cpu().numpy(), fs.cpu().numpy(), ref.trace["xq"], ref.trace["sx"])
    check_output(bits(y), ref.y_ref, rows_mask=~differ)
    return ref


@pytest.mark.parametrize("rows,path", [(1, m.PATH_AUTO), (3, m.PATH_AUTO), (11, m.PATH_AUTO),
                                       (24, m.PATH_AUTO), (24, m.PATH_PROMPT_MMA),
                                       (1, m.PATH_DECODE_CHAINED), (11, m.PATH_DECODE_ROWS)])
def test_router_bf16_pin_rows(bf16_layer, dev, rows, path):
    """The pin's 24 rows (exact bf16 ties among the first k + 1 experts, and
    routings that differ from the fp32 router) on every kernel family."""
    layer, net, host = bf16_layer
    x = W.make_x(W.FULL, 24, 21).to(dev)[:rows].contiguous()
    ref = _check_bf16(net, host, x, path, W.FULL.top_k)
    if rows == 24:
        top = np.sort(ref.trace["logits"], axis=1)[:, ::-1][:, :9]
        assert np.any(top[:, 1:] == top[:, :-1]), "the pin's rows meet exact ties"


def test_router_bf16_prompt_t1024(bf16_layer, dev):
    layer, net, host = bf16_layer
    x = W.make_x(W.FULL, 1024, 21, tag="bf16p").to(dev)
    _check_bf16(net, host, x, m.PATH_AUTO, W.FULL.top_k)


def test_router_bf16_option_range(bf16_layer):
    _, net, _ = bf16_layer
    assert m.moe_set_option(net.ctx, m.MOE_OPT_ROUTER_BF16, 2) == m.MOE_ERR_INVALID_ARG
    assert m.moe_set_option(net.ctx, m.MOE_OPT_ROUTER_BF16, 0) == m.MOE_OK


# ---- one activation scale per row --------------------------------------------

PER_ROW = {"act_per_row": True}


@pytest.fixture(scope="module")
def per_row_full(dev):
    c = Case(W.WORKLOADS["decode_t11"], 1024, dev, act_group=W.FULL.hidden)
    yield c
    c.moe.close()


@pytest.mark.parametrize("rows", [1, 2, 5, 11, 16, 17, 64, 1024])
def test_per_row_scales_full_layer(per_row_full, rows):
    """1 row on the one-row kernel, 2..16 on the role-split multi-row kernel,
    more on the tcgen05 kernels (with the row quantiser of the SwiGLU rows)."""
    x = per_row_full.x(rows, tag=f"pr{rows}")
    run_and_check(per_row_full, x, oracle_kw=PER_ROW)


def test_per_row_scales_codes_are_one_per_row(per_row_full):
    x = per_row_full.x(3, tag="pr_codes")
    per_row_full.moe.forward(x)
    codes, scales = per_row_full.moe.forward_codes(3)
    q_codes, q_scales = per_row_full.moe.quantize(x)
    torch.cuda.synchronize()
    s = scales.cpu().numpy()
    assert np.all(s == s[:, :, :1])  # every group of a row has the row's scale
    assert np.array_equal(q_codes.cpu().numpy(), codes.cpu().numpy()[:, 0])
    assert np.array_equal(q_scales.cpu().numpy(), s[:, 0])


@pytest.mark.parametrize("rows", [1, 4, 40])
def test_per_row_scales_tiny_layer(dev, rows):
    case = Case(W.WORKLOADS["tiny_t4"], 64, dev, act_group=W.TINY.hidden)
    run_and_check(case, case.x(rows, tag=f"prt{rows}"), oracle_kw=PER_ROW)
    case.moe.close()


def test_per_row_scales_refusals(per_row_full, dev):
    ctx = per_row_full.moe.ctx
    assert m.moe_set_option(ctx, m.MOE_OPT_PATH, m.PATH_DECODE_CHAINED) == \
        m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_set_option(ctx, m.MOE_OPT_PATH, m.PATH_PROMPT_MMA) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_set_option(ctx, m.MOE_OPT_PATH, m.PATH_PROMPT) == m.MOE_OK
    assert m.moe_set_option(ctx, m.MOE_OPT_PATH, m.PATH_AUTO) == m.MOE_OK
    H = W.FULL.hidden
    z = torch.zeros((1, H), dtype=torch.bfloat16, device=dev)
    g = torch.ones((H,), dtype=torch.bfloat16, device=dev)
    c = torch.empty((1, H), dtype=torch.uint8, device=dev)
    sc = torch.empty((1, H // 128), dtype=torch.float32, device=dev)
    assert m.moe_add_rmsnorm_quantize(ctx, z, z.clone(), g, 1e-6, 1, torch.empty_like(z),
                                      torch.empty_like(z), c, sc) == m.MOE_ERR_UNSUPPORTED_SHAPE
