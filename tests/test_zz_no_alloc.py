"""moe_route_static: the router for callers that cannot allocate device
memory (a runtime whose memory pool has already claimed the device, or a
latency-critical loop that must not pay for cudaMalloc's implicit
synchronisation).  Its logits live in a fixed scratch array of the library.

Checked on two calls in a row: against the oracle's router (the definition),
and against moe_route on the same inputs (the context-owning entry point,
same bar as every other GPU test).  The device's free memory is read around
the second call and must not change.  The file name sorts last so the test
also runs after every other GPU test; it passes alone in a fresh process too.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import bits, check_topk

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


def _route_static(layer, s, x, idx=None, w=None):
    T = x.shape[0]
    if idx is None:
        idx = torch.full((T, s.top_k), -1, dtype=torch.int32, device=x.device)
        w = torch.full((T, s.top_k), -1.0, dtype=torch.float32, device=x.device)
    rc = m.moe_route_static(x, layer["router"], T, s.hidden, s.n_experts, s.top_k, idx, w)
    return rc, idx, w


def _check_against_oracle(x, router_host, k, idx, w):
    """Ordered top-k bit-exact outside near ties, weights within the bar of
    the other router tests, against the oracle's router row by row."""
    xb = bits(x)
    T = xb.shape[0]
    logits = np.zeros((T, router_host.shape[0]))
    w_ref = np.zeros((T, k))
    for t in range(T):
        logits[t], _, w_ref[t] = oracle.router_row(xb[t], router_host, k)
    near, differ = check_topk(idx, logits, k)
    assert differ.sum() <= max(1, 0.02 * T), f"{differ.sum()} rows routed differently"
    assert np.allclose(w[~differ], w_ref[~differ], rtol=2e-5, atol=1e-7)


@pytest.mark.parametrize("name,rows", [("decode_t1", 1), ("decode_t1", 17), ("decode_t1", 1024),
                                       ("tiny_t4", 40), ("tiny_t4", 3000)])
def test_two_consecutive_calls(dev, name, rows):
    wl, seed, layer, moe = _layer(name, dev, max_rows=rows)
    s = wl.shape
    router_host = layer["router"].cpu().numpy()
    idx = torch.full((rows, s.top_k), -1, dtype=torch.int32, device=dev)
    w = torch.full((rows, s.top_k), -1.0, dtype=torch.float32, device=dev)
    for tag in ("first", "second"):
        x = W.make_x(s, rows, seed, wl.x_kind, device="cuda", tag=tag)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info(dev)[0]
        rc, _, _ = _route_static(layer, s, x, idx, w)
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info(dev)[0]
        assert rc == m.MOE_OK, m.status_string(rc)
        if tag == "second":
            # set-up is done: this call takes no device memory
            assert free1 == free0, (free0, free1)
        gi, gw = idx.cpu().numpy().copy(), w.cpu().numpy().copy()
        _check_against_oracle(x, router_host, s.top_k, gi, gw)
        idx_ref, w_ref = moe.route(x)
        torch.cuda.synchronize()
        assert np.array_equal(gi, idx_ref.cpu().numpy()), tag
        assert np.allclose(gw, w_ref.cpu().numpy(), rtol=1e-6, atol=0.0), tag
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
