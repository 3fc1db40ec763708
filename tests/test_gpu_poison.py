"""No kernel depends on what an earlier call left in the workspace: its value
buffers filled with NaN bytes (0xFF: NaN in bf16, fp32 and e4m3), zeros or
0x7F between two forwards leave the output bits unchanged, on every path.

The pages have no such test; it checks this implementation (stale or
never-written workspace read by mistake would change the second output)."""
from __future__ import annotations

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

m = pytest.importorskip("block_fp8_mixture_router_gb300")


@pytest.fixture(scope="module")
def net():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = W.WORKLOADS["decode_t1"]
    s = wl.shape
    dev = torch.device("cuda", 0)
    layer = W.make_layer(s, W.layer_seed(wl, 0), wl.x_kind, device=dev)
    n = m.MoELayer(m.LayerShape(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, s.group),
                   max_rows=1024)
    n.load(layer)
    yield wl, n
    n.close()


@pytest.mark.parametrize("rows,path", [(1, m.PATH_AUTO), (3, m.PATH_AUTO), (11, m.PATH_AUTO),
                                       (11, m.PATH_DECODE_CHAINED), (11, m.PATH_DECODE_ROWS),
                                       (64, m.PATH_AUTO), (1024, m.PATH_AUTO)])
def test_forward_ignores_stale_workspace(net, rows, path):
    wl, n = net
    x = W.make_x(wl.shape, rows, wl.seed, wl.x_kind, device="cuda", tag=f"poison{rows}")
    n.set_option(m.MOE_OPT_PATH, path)
    try:
        y0 = n.forward(x).clone()
        for byte in (0xFF, 0x00, 0x7F):
            n.poison_workspace(byte)
            y1 = n.forward(x)
            torch.cuda.synchronize()
            assert torch.equal(y1.view(torch.int16), y0.view(torch.int16)), (rows, path, byte)
    finally:
        n.set_option(m.MOE_OPT_PATH, m.PATH_AUTO)
    assert n.device_status() == m.MOE_OK


@pytest.mark.parametrize("rows", [1, 11, 1024])
def test_forward_addnorm_ignores_stale_workspace(net, rows):
    wl, n = net
    r, x, g = W.make_addnorm(wl.shape, rows, seed=3, device="cuda")
    h0, xn0, y0 = n.forward_addnorm(r, x, g, 1e-6)
    y0 = y0.clone()
    n.poison_workspace(0xFF)
    h1, xn1, y1 = n.forward_addnorm(r, x, g, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y0.view(torch.int16)), rows
    assert torch.equal(h1.view(torch.int16), h0.view(torch.int16)), rows
