"""Layers in sequence (moe_chain_*), the backbone's 40 MoE layers with one
row passed through them (needs a GB300).

At one row the chain runs as one launch of the one-row kernel looping over
the layers (PR #939 "drama3: Fish Audio Drama 3 text to speech on one CUDA
GPU", section "What it adds": the frame step runs the next backbone row as
one CUDA graph; PR #927 "drama: the backbone chain launches with programmatic
dependent launch").  Its arithmetic per layer is the one-row forward's, so:
  - every layer's output equals moe_forward of that layer on the previous
    layer's output, bit for bit;
  - every layer, teacher forced (on the GPU's own input to that layer),
    matches the oracle: routing bit-exact outside near ties, y within the bar.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import bits, check_output, check_topk

pytestmark = pytest.mark.gpu

m = pytest.importorskip("block_fp8_mixture_router_gb300")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    return torch.device("cuda", 0)


def _layers(n, dev, max_rows=16):
    wl = W.WORKLOADS["sweep40"]
    s = wl.shape
    layers, nets = [], []
    for l in range(n):
        layer = W.make_layer(s, W.layer_seed(wl, l), wl.x_kind, device=dev)
        net = m.MoELayer(m.LayerShape(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter,
                                      s.group), max_rows=max_rows)
        net.load(layer)
        layers.append(layer)
        nets.append(net)
    x = W.make_x(s, 1, W.layer_seed(wl, 0), wl.x_kind, device="cuda", tag="chain")
    return layers, nets, x


def _host_subset(layer: dict, experts) -> dict:
    """The oracle's numpy layer with only `experts` copied from the device
    (the other experts stay zero pages that are never touched)."""
    out = {}
    for n, v in layer.items():
        if not isinstance(v, torch.Tensor):
            out[n] = v
        elif n in ("w13", "s13", "w2", "s2"):
            a = np.zeros(tuple(v.shape), dtype=W.to_numpy_layer({n: v[:1]})[n].dtype)
            for e in experts:
                a[e] = W.to_numpy_layer({n: v[e:e + 1]})[n][0]
            out[n] = a
        else:
            out[n] = W.to_numpy_layer({n: v})[n]
    return out


def test_chain_one_row_equals_layer_by_layer(dev):
    layers, nets, x = _layers(4, dev)
    chain = m.MoEChain(nets)
    y_all = chain.forward(x).clone()
    y_again = chain.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(y_all.view(torch.int16), y_again.view(torch.int16))
    src = x
    for l, net in enumerate(nets):
        y = net.forward(src)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_all[l].view(torch.int16)), l
        src = y_all[l]
    # more rows: each layer's forward in order
    x3 = W.make_x(W.FULL, 3, 1234, device="cuda", tag="chain3")
    y3 = chain.forward(x3)
    src = x3
    for l, net in enumerate(nets):
        y = net.forward(src)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y3[l].view(torch.int16)), l
        src = y3[l]
    chain.close()
    for net in nets:
        net.close()


def test_chain_40_layers_teacher_forced(dev):
    layers, nets, x = _layers(40, dev)
    chain = m.MoEChain(nets)
    y_all = chain.forward(x)
    torch.cuda.synchronize()
    assert nets[0].device_status() == m.MOE_OK
    s = W.FULL
    for l, (layer, net) in enumerate(zip(layers, nets)):
        xl = x if l == 0 else y_all[l - 1]
        idx, _ = net.route(xl)
        torch.cuda.synchronize()
        host = _host_subset(layer, sorted(set(idx.cpu().numpy().ravel().tolist())))
        ref = oracle.moe_rows(host, bits(xl), trace=True)
        near, differ = check_topk(idx.cpu().numpy(), ref.trace["logits"], s.top_k)
        if differ.any():  # a near tie ordered the other way: the experts differ
            continue
        check_output(bits(y_all[l]), ref.y_ref)
    chain.close()
    for net in nets:
        net.close()


def test_chain_refusals(dev):
    layers, nets, x = _layers(2, dev)
    tiny = m.MoELayer(m.LayerShape(256, 16, 4, 128, 128), max_rows=4)
    tiny.load(W.make_layer(W.TINY, 0, device=dev))
    rc, h = m.moe_chain_create([nets[0].ctx, tiny.ctx])
    assert rc == m.MOE_ERR_UNSUPPORTED_SHAPE and not h.value
    rc, h = m.moe_chain_create([])
    assert rc == m.MOE_ERR_INVALID_ARG
    unloaded = m.MoELayer(m.LayerShape(), max_rows=4)
    rc, h = m.moe_chain_create([nets[0].ctx, unloaded.ctx])
    assert rc == m.MOE_ERR_NOT_LOADED
    chain = m.MoEChain(nets)
    y = torch.empty((2, 1, W.FULL.hidden), dtype=torch.bfloat16, device=dev)
    assert m.moe_chain_forward(chain.chain, x, y, 17) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_chain_forward(chain.chain, y[0], y, 1) == m.MOE_ERR_INVALID_ARG
    assert m.moe_chain_forward(chain.chain, x, y, 0) == m.MOE_OK
    chain.close()
    for net in nets + [tiny, unloaded]:
        net.close()


def test_chain_across_the_tag_clear(dev):
    """A chain launch uses one launch tag per layer; started just below the
    clearing threshold it crosses it, clears the exchange words at its end and
    restarts the tags: the outputs stay bit for bit the same."""
    layers, nets, x = _layers(3, dev)
    chain = m.MoEChain(nets)
    ref = chain.forward(x).clone()
    torch.cuda.synchronize()
    nets[0].set_option(m.MOE_OPT_LAUNCH_EPOCH, m.TAG_CLEAR - 2)
    outs = [chain.forward(x).clone() for _ in range(3)]
    y0 = nets[0].forward(x)
    torch.cuda.synchronize()
    for y in outs:
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(y0.view(torch.int16), ref[0].view(torch.int16))
    assert nets[0].device_status() == m.MOE_OK
    chain.close()
    for net in nets:
        net.close()
