"""moe_route_static (router on the library's fixed scratch, no allocation)
against moe_route on the same inputs, two calls in a row.  The file name
sorts last so the test also runs after every other GPU test."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

m = pytest.importorskip("block_fp8_mixture_router_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    return torch.device("cuda", 0)


def _layer(name, dev, max_rows):
    wl = W.WORKLOADS[name]
    s = wl.shape
    seed = W.layer_seed(wl, 0)
    layer = W.make_layer(s, seed, wl.x_kind, device=dev)
    moe = m.MoELayer(m.LayerShape(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter,
                                  s.group), max_rows=max_rows)
    moe.load(layer)
    # moe_route on the router kernels moe_route_static also runs (the
    # CUDA-core router of the warp-MMA prompt path)
    moe.set_option(m.MOE_OPT_PATH, m.PATH_PROMPT_MMA)
    return wl, seed, layer, moe


def _route_static(layer, s, x):
    T = x.shape[0]
    idx = torch.full((T, s.top_k), -1, dtype=torch.int32, device=x.device)
    w = torch.full((T, s.top_k), -1.0, dtype=torch.float32, device=x.device)
    rc = m.moe_route_static(x, layer["router"], T, s.hidden, s.n_experts, s.top_k, idx, w)
    return rc, idx, w


@pytest.mark.parametrize("name,rows", [("decode_t1", 1), ("decode_t1", 17), ("decode_t1", 1024),
                                       ("tiny_t4", 40), ("tiny_t4", 3000)])
def test_two_consecutive_calls_match_moe_route(dev, name, rows):
    wl, seed, layer, moe = _layer(name, dev, max_rows=rows)
    s = wl.shape
    for tag in ("first", "second"):
        x = W.make_x(s, rows, seed, wl.x_kind, device="cuda", tag=tag)
        rc, idx, w = _route_static(layer, s, x)
        assert rc == m.MOE_OK, m.status_string(rc)
        idx_ref, w_ref = moe.route(x)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), idx_ref.cpu().numpy()), tag
        assert np.allclose(w.cpu().numpy(), w_ref.cpu().numpy(), rtol=1e-6, atol=0.0), tag
    moe.close()


def test_refuses_more_logits_than_the_scratch_holds(dev):
    wl = W.WORKLOADS["decode_t1"]
    s = wl.shape
    layer = W.make_layer(s, W.layer_seed(wl, 0), wl.x_kind, device=dev)
    rows = m.MOE_ROUTE_STATIC_MAX_LOGITS // s.n_experts + 1
    x = torch.zeros((rows, s.hidden), dtype=torch.bfloat16, device=dev)
    rc, idx, w = _route_static(layer, s, x)
    torch.cuda.synchronize()
    assert rc == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert bool((idx == -1).all()) and bool((w == -1.0).all())
    assert m.moe_route_static(x, layer["router"], 0, s.hidden, s.n_experts, s.top_k, None,
                              None) == m.MOE_OK
