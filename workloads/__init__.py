"""Seeded synthetic inputs for the block-FP8 MoE layer.

This module only draws numbers: it holds none of the layer's arithmetic and is
the one thing the CUDA path and the CPU oracle share.  The shapes and value
distributions follow the workloads the Drama 3 pages describe (one-row decode
steps, one frame's eleven rows, prompt chunks of up to 1024 rows, the 40-layer
backbone); no dataset or trained checkpoint is involved.

Weights are drawn in fp32 from N(0, 0.02) and stored the way a block-FP8
checkpoint stores them: e4m3 codes plus one fp32 scale (block amax / 448) per
128 x 128 block.  That conversion is checkpoint preparation, done once with
PyTorch's own float8 cast; the layer itself never requantises weights.

Every tensor has its own generator seed, derived from (layer seed, tensor
name, expert), so any one expert of any layer can be regenerated alone.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import torch

GROUP = 128
WEIGHT_STD = 0.02


@dataclass(frozen=True)
class MoEShape:
    hidden: int = 2048        # H
    n_experts: int = 256      # E
    top_k: int = 8            # k
    inter: int = 512          # I, routed SwiGLU width
    shared_inter: int = 512   # Is, shared SwiGLU width
    group: int = GROUP        # activation group = weight block edge


FULL = MoEShape()
TINY = MoEShape(hidden=256, n_experts=16, top_k=4, inter=128, shared_inter=128)


@dataclass(frozen=True)
class Workload:
    name: str
    shape: MoEShape
    rows: int
    seed: int
    x_kind: str = "normal"        # normal | shared_plus_noise | bias_skew
    layers: int = 1
    description: str = ""


WORKLOADS = {
    "tiny_t4": Workload("tiny_t4", TINY, 4, 0, "normal", 1,
                        "T=4, H=256, 16 experts top-4, I=Is=128"),
    "decode_t1": Workload("decode_t1", FULL, 1, 1, "normal", 1,
                          "one-row decode step, H=2048, 256 experts top-8, I=Is=512"),
    "decode_t11": Workload("decode_t11", FULL, 11, 2, "shared_plus_noise", 1,
                           "eleven rows of one frame, overlapping expert sets"),
    "prompt_t1024": Workload("prompt_t1024", FULL, 1024, 3, "bias_skew", 1,
                             "1024-row prompt chunk, per-expert router bias N(0,1)"),
    "prompt_t16384": Workload("prompt_t16384", FULL, 16384, 4, "bias_skew", 1,
                              "16384 rows, compute-bound prompt shape"),
    "sweep40": Workload("sweep40", FULL, 1, 1000, "normal", 40,
                        "40 independent layers, one batch passed through all"),
}
SWEEP_ROWS = (1, 4, 16, 64, 256, 1024)


def _seed(*parts) -> int:
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


def _randn(shape, device, *parts) -> torch.Tensor:
    return torch.randn(shape, generator=_gen(device, *parts), device=device,
                       dtype=torch.float32)


def quantize_blocks(w: torch.Tensor, group: int = GROUP):
    """fp32 [..., R, C] -> (e4m3 codes as uint8 [..., R, C], fp32 scales [..., R/g, C/g]).

    Checkpoint preparation: scale = block amax / 448, codes = PyTorch's float8
    cast of w / scale (round to nearest even; |w / scale| <= 448 by construction).
    """
    *lead, R, C = w.shape
    b = w.reshape(*lead, R // group, group, C // group, group)
    amax = b.abs().amax(dim=(-3, -1))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (b / scale[..., :, None, :, None]).reshape(*lead, R, C)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.contiguous()


def make_router(shape: MoEShape, seed: int, x_kind: str = "normal", device="cpu"):
    wr = _randn((shape.n_experts, shape.hidden), device, seed, "router") * WEIGHT_STD
    if x_kind == "bias_skew":
        # a per-expert bias b ~ N(0,1), carried by the last input coordinate (fixed to 1)
        wr[:, -1] = _randn((shape.n_experts,), device, seed, "router_bias")
    return wr.contiguous()


def make_expert(shape: MoEShape, seed: int, e: int, device="cpu"):
    """One routed expert: (w13 codes [2I,H], s13 [2I/g,H/g], w2 codes [H,I], s2 [H/g,I/g])."""
    w13 = _randn((2 * shape.inter, shape.hidden), device, seed, "w13", e) * WEIGHT_STD
    w2 = _randn((shape.hidden, shape.inter), device, seed, "w2", e) * WEIGHT_STD
    c13, s13 = quantize_blocks(w13, shape.group)
    c2, s2 = quantize_blocks(w2, shape.group)
    return c13, s13, c2, s2


def make_shared(shape: MoEShape, seed: int, device="cpu"):
    ws13 = (_randn((2 * shape.shared_inter, shape.hidden), device, seed, "ws13")
            * WEIGHT_STD).to(torch.bfloat16)
    ws2 = (_randn((shape.hidden, shape.shared_inter), device, seed, "ws2")
           * WEIGHT_STD).to(torch.bfloat16)
    gate = (_randn((shape.hidden,), device, seed, "shared_gate") * WEIGHT_STD).to(torch.bfloat16)
    return ws13, ws2, gate


def make_layer(shape: MoEShape, seed: int, x_kind: str = "normal", device="cpu",
               experts=None) -> dict:
    """All weights of one layer as torch tensors on `device`.

    `experts`: iterable of expert ids to generate; the others stay zero (used by
    CPU tests that only need the experts a few rows select).
    """
    E, H, I, g = shape.n_experts, shape.hidden, shape.inter, shape.group
    w13 = torch.zeros((E, 2 * I, H), dtype=torch.uint8, device=device)
    s13 = torch.ones((E, 2 * I // g, H // g), dtype=torch.float32, device=device)
    w2 = torch.zeros((E, H, I), dtype=torch.uint8, device=device)
    s2 = torch.ones((E, H // g, I // g), dtype=torch.float32, device=device)
    for e in (range(E) if experts is None else sorted(set(int(v) for v in experts))):
        c13, sc13, c2, sc2 = make_expert(shape, seed, e, device)
        w13[e], s13[e], w2[e], s2[e] = c13, sc13, c2, sc2
    ws13, ws2, gate = make_shared(shape, seed, device)
    return dict(w13=w13, s13=s13, w2=w2, s2=s2,
                router=make_router(shape, seed, x_kind, device),
                ws13=ws13, ws2=ws2, shared_gate=gate, top_k=shape.top_k)


def make_x(shape: MoEShape, rows: int, seed: int, x_kind: str = "normal", device="cpu",
           tag: str = "x") -> torch.Tensor:
    """Layer input [rows, H] bf16."""
    H = shape.hidden
    if x_kind == "shared_plus_noise":
        # every row = one shared N(0,1) vector + 0.5 * its own N(0,1) noise, so the
        # rows' router logits share a component and their expert sets overlap
        a = _randn((1, H), device, seed, tag, "shared")
        n = _randn((rows, H), device, seed, tag, "noise")
        x = a + 0.5 * n
    else:
        x = _randn((rows, H), device, seed, tag)
        if x_kind == "bias_skew":
            x[:, -1] = 1.0
    return x.to(torch.bfloat16).contiguous()


NORM_EPS = 1e-6


def make_addnorm(shape: MoEShape, rows: int, seed: int, device="cpu"):
    """Inputs of the residual add + RMS norm in front of the layer, all bf16:
    the residual stream [rows, H] ~ N(0, 1), the preceding block's output
    [rows, H] ~ N(0, 0.5^2), and the norm weight gamma [H] ~ 1 + N(0, 0.1^2)."""
    H = shape.hidden
    residual = _randn((rows, H), device, seed, "residual").to(torch.bfloat16).contiguous()
    x = (0.5 * _randn((rows, H), device, seed, "block_out")).to(torch.bfloat16).contiguous()
    gamma = (1.0 + 0.1 * _randn((H,), device, seed, "norm_gamma")).to(torch.bfloat16)
    return residual, x, gamma.contiguous()


def layer_seed(workload: Workload, layer: int) -> int:
    return workload.seed + layer if workload.layers > 1 else workload.seed


def to_numpy_layer(layer: dict) -> dict:
    """Torch layer -> numpy arrays in the oracle's convention (bf16 as uint16 bits)."""
    out = {}
    for n, v in layer.items():
        if isinstance(v, torch.Tensor):
            t = v.detach().cpu()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
                out[n] = t.numpy().view("uint16")
            else:
                out[n] = t.numpy()
        else:
            out[n] = v
    return out


def bf16_bits(x: torch.Tensor):
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
