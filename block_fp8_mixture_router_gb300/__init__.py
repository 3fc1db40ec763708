"""Python binding of the block-FP8 MoE layer's C ABI (include/moe.h).

Argument marshalling only: every step of the layer runs in the CUDA kernels of
`lib/libmoe_gb300.so`.  PyTorch provides device memory and streams.  There is
no CPU fallback: if the library is missing or fails to load, importing the
binding's entry points raises.

Low-level functions carry the C names (`moe_create`, `moe_forward`, ...) and
return the C status; `MoELayer` wraps them and raises `MoEError`.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED_SHAPE = -2
MOE_ERR_NOT_LOADED = -3
MOE_ERR_ALLOC_LIMIT = -4
MOE_ERR_CUDA = -5
MOE_ERR_DEVICE_TIMEOUT = -6

MOE_OPT_PATH = 1
MOE_OPT_PDL = 2
MOE_OPT_POLL_LIMIT = 3
MOE_OPT_LAUNCH_EPOCH = 4
MOE_OPT_BATCH_INVARIANT = 5
MOE_OPT_ROUTER_BF16 = 6
TAG_WRAP = 0x7FFFFFFF
TAG_CLEAR = TAG_WRAP - 4096  # tags of the role-split decode kernels stay below TAG_WRAP
PATH_AUTO, PATH_DECODE, PATH_PROMPT, PATH_DECODE_CHAINED, PATH_PROMPT_MMA = 0, 1, 2, 3, 4
PATH_DECODE_ROWS = 6  # the role-split multi-row decode kernel for 2..16 rows

EXPORTED = ("moe_create", "moe_load_weights", "moe_forward", "moe_forward_host", "moe_route",
            "moe_quantize", "moe_expert_activations", "moe_set_option", "moe_required_bytes",
            "moe_last_device_status", "moe_destroy", "moe_status_string",
            "moe_profile_forward", "moe_route_static", "moe_add_rmsnorm_quantize",
            "moe_forward_codes", "moe_forward_addnorm", "moe_chain_create",
            "moe_chain_forward", "moe_chain_destroy", "moe_debug_poison_workspace")

MOE_ROUTE_STATIC_MAX_LOGITS = 262144


class moe_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("inter", ctypes.c_int), ("shared_inter", ctypes.c_int),
                ("act_group", ctypes.c_int), ("max_rows", ctypes.c_int),
                ("workspace_cap_bytes", ctypes.c_size_t)]


class moe_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w13", "s13", "w2", "s2", "router", "ws13", "ws2", "shared_gate")]


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def load_library(path: str = LIB_PATH):
    """Load the shared library; raises if it is missing (no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
    L = ctypes.CDLL(path)
    vp, i, ip = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p)
    L.moe_create.argtypes = [ctypes.POINTER(moe_config), i, ip]
    L.moe_load_weights.argtypes = [vp, ctypes.POINTER(moe_weights), i, vp]
    L.moe_forward.argtypes = [vp, vp, vp, i, vp]
    L.moe_forward_host.argtypes = [vp, vp, vp, i, vp]
    L.moe_route.argtypes = [vp, vp, i, vp, vp, vp]
    L.moe_quantize.argtypes = [vp, vp, i, vp, vp, vp]
    L.moe_add_rmsnorm_quantize.argtypes = [vp, vp, vp, vp, ctypes.c_float, i, vp, vp, vp, vp,
                                           vp]
    L.moe_route_static.argtypes = [vp, vp, i, i, i, i, vp, vp, vp]
    L.moe_expert_activations.argtypes = [vp, i, vp, vp, vp]
    L.moe_forward_codes.argtypes = [vp, i, vp, vp, vp]
    L.moe_forward_addnorm.argtypes = [vp, vp, vp, vp, ctypes.c_float, i, vp, vp, vp, vp]
    L.moe_chain_create.argtypes = [ctypes.POINTER(ctypes.c_void_p), i, ip]
    L.moe_chain_forward.argtypes = [vp, vp, vp, i, vp]
    L.moe_chain_destroy.argtypes = [vp]
    L.moe_chain_destroy.restype = None
    L.moe_set_option.argtypes = [vp, i, i]
    L.moe_debug_poison_workspace.argtypes = [vp, i, vp]
    L.moe_profile_forward.argtypes = [vp, vp, vp, i, vp, vp, i, ctypes.POINTER(ctypes.c_int), vp]
    L.moe_required_bytes.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(ctypes.c_size_t)]
    L.moe_last_device_status.argtypes = [vp]
    L.moe_destroy.argtypes = [vp]
    L.moe_destroy.restype = None
    L.moe_status_string.argtypes = [i]
    L.moe_status_string.restype = ctypes.c_char_p
    for n in EXPORTED:
        if n not in ("moe_destroy", "moe_status_string", "moe_chain_destroy"):
            getattr(L, n).restype = ctypes.c_int
    _lib = L
    return L


def status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


# ---- C names, thin wrappers (status returned as is) ------------------------

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return ctypes.c_void_p(t.data_ptr())
    return ctypes.c_void_p(int(t))


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def moe_create(cfg: moe_config, device: int = 0):
    h = ctypes.c_void_p()
    rc = load_library().moe_create(ctypes.byref(cfg), device, ctypes.byref(h))
    return rc, h


def moe_load_weights(ctx, w: moe_weights, pointers_on_device: int, stream=None) -> int:
    return load_library().moe_load_weights(ctx, ctypes.byref(w), pointers_on_device,
                                           _stream(stream))


def moe_forward(ctx, x, y, rows: int, stream=None) -> int:
    return load_library().moe_forward(ctx, _ptr(x), _ptr(y), rows, _stream(stream))


def moe_forward_host(ctx, x, y, rows: int, stream=None) -> int:
    return load_library().moe_forward_host(ctx, _ptr(x), _ptr(y), rows, _stream(stream))


def moe_debug_poison_workspace(ctx, byte: int, stream=None) -> int:
    """Fills the context's data workspace with `byte` (a test of the
    kernels' independence from earlier calls' leftovers)."""
    return load_library().moe_debug_poison_workspace(ctx, byte, _stream(stream))


def moe_route(ctx, x, rows: int, idx, w, stream=None) -> int:
    return load_library().moe_route(ctx, _ptr(x), rows, _ptr(idx), _ptr(w), _stream(stream))


def moe_route_static(x, router, rows: int, hidden: int, n_experts: int, top_k: int, idx, w,
                     stream=None) -> int:
    """The router on the library's fixed scratch (allocates nothing); calls on
    one device must not overlap."""
    return load_library().moe_route_static(_ptr(x), _ptr(router), rows, hidden, n_experts,
                                           top_k, _ptr(idx), _ptr(w), _stream(stream))


def moe_quantize(ctx, x, rows: int, codes, scales, stream=None) -> int:
    return load_library().moe_quantize(ctx, _ptr(x), rows, _ptr(codes), _ptr(scales),
                                       _stream(stream))


def moe_add_rmsnorm_quantize(ctx, residual, x, gamma, eps: float, rows: int, h_out, xn_out,
                             codes, scales, stream=None) -> int:
    return load_library().moe_add_rmsnorm_quantize(
        ctx, _ptr(residual), _ptr(x), _ptr(gamma), float(eps), rows, _ptr(h_out), _ptr(xn_out),
        _ptr(codes), _ptr(scales), _stream(stream))


def moe_expert_activations(ctx, rows: int, hq, sh, stream=None) -> int:
    return load_library().moe_expert_activations(ctx, rows, _ptr(hq), _ptr(sh), _stream(stream))


def moe_forward_addnorm(ctx, residual, x, gamma, eps: float, rows: int, h_out, xn_out, y,
                        stream=None) -> int:
    return load_library().moe_forward_addnorm(ctx, _ptr(residual), _ptr(x), _ptr(gamma),
                                              float(eps), rows, _ptr(h_out), _ptr(xn_out),
                                              _ptr(y), _stream(stream))


def moe_chain_create(ctxs):
    arr = (ctypes.c_void_p * len(ctxs))(*[c.value if isinstance(c, ctypes.c_void_p) else c
                                          for c in ctxs])
    h = ctypes.c_void_p()
    rc = load_library().moe_chain_create(arr, len(ctxs), ctypes.byref(h))
    return rc, h


def moe_chain_forward(chain, x, y_all, rows: int, stream=None) -> int:
    return load_library().moe_chain_forward(chain, _ptr(x), _ptr(y_all), rows, _stream(stream))


def moe_chain_destroy(chain) -> None:
    load_library().moe_chain_destroy(chain)


def moe_forward_codes(ctx, rows: int, codes, scales, stream=None) -> int:
    return load_library().moe_forward_codes(ctx, rows, _ptr(codes), _ptr(scales),
                                            _stream(stream))


def moe_profile_forward(ctx, x, y, rows: int, stream=None, capacity: int = 16):
    """-> (status, [(stage name, device ms), ...])"""
    ms = (ctypes.c_float * capacity)()
    names = (ctypes.c_char_p * capacity)()
    n = ctypes.c_int()
    rc = load_library().moe_profile_forward(ctx, _ptr(x), _ptr(y), rows, ctypes.cast(ms, ctypes.c_void_p),
                                            ctypes.cast(names, ctypes.c_void_p), capacity,
                                            ctypes.byref(n), _stream(stream))
    return rc, [(names[i].decode(), float(ms[i])) for i in range(n.value)]


def moe_set_option(ctx, option: int, value: int) -> int:
    return load_library().moe_set_option(ctx, option, value)


def moe_required_bytes(cfg: moe_config):
    n = ctypes.c_size_t()
    rc = load_library().moe_required_bytes(ctypes.byref(cfg), ctypes.byref(n))
    return rc, n.value


def moe_last_device_status(ctx) -> int:
    return load_library().moe_last_device_status(ctx)


def moe_destroy(ctx) -> None:
    load_library().moe_destroy(ctx)


def moe_status_string(status: int) -> str:
    return status_string(status)


# ---- convenience wrapper ---------------------------------------------------

@dataclass
class LayerShape:
    hidden: int = 2048
    n_experts: int = 256
    top_k: int = 8
    inter: int = 512
    shared_inter: int = 512
    act_group: int = 128


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoEError(rc, what)


class MoELayer:
    """One layer on one GPU: owns a context, its device weights and workspace."""

    def __init__(self, shape: LayerShape, max_rows: int = 1024, device: int = 0,
                 workspace_cap_bytes: int = 0):
        self.shape = shape
        self.max_rows = max_rows
        self.device = device
        cfg = moe_config(shape.hidden, shape.n_experts, shape.top_k, shape.inter,
                         shape.shared_inter, shape.act_group, max_rows, workspace_cap_bytes)
        rc, h = moe_create(cfg, device)
        _check(rc, "moe_create")
        self.ctx = h

    def close(self):
        if getattr(self, "ctx", None):
            moe_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load(self, layer: dict, stream=None):
        """Weights as torch tensors (see include/moe.h for names, dtypes, layouts)."""
        names = ("w13", "s13", "w2", "s2", "router", "ws13", "ws2", "shared_gate")
        ts = [layer[n].contiguous() for n in names]
        on_dev = {t.is_cuda for t in ts}
        if len(on_dev) != 1:
            raise ValueError("weights must be all on the device or all on the host")
        w = moe_weights(*[t.data_ptr() for t in ts])
        _check(moe_load_weights(self.ctx, w, 1 if ts[0].is_cuda else 0, stream),
               "moe_load_weights")
        self._keep = ts  # alive until the synchronous copy returned

    def set_option(self, option: int, value: int):
        _check(moe_set_option(self.ctx, option, value), "moe_set_option")

    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2:
            raise ValueError("x must be a 2-D bf16 CUDA tensor")
        x = x.contiguous()
        if y is None:
            y = torch.empty_like(x)
        _check(moe_forward(self.ctx, x, y, x.shape[0], stream), "moe_forward")
        return y

    def forward_addnorm(self, residual: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor,
                        eps: float, keep_xn: bool = False, stream=None):
        """Residual add + RMS norm + the layer: returns (h, xn or None, y)."""
        for t in (residual, x, gamma):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("residual, x and gamma must be contiguous bf16 CUDA tensors")
        T, H = x.shape
        h = torch.empty_like(x)
        xn = torch.empty_like(x) if keep_xn else None
        y = torch.empty_like(x)
        _check(moe_forward_addnorm(self.ctx, residual, x, gamma, eps, T, h, xn, y, stream),
               "moe_forward_addnorm")
        return h, xn, y

    def forward_host(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None):
        if x.dtype != torch.bfloat16 or x.is_cuda:
            raise ValueError("x must be a host bf16 tensor")
        if y is None:
            y = torch.empty_like(x)
        _check(moe_forward_host(self.ctx, x, y, x.shape[0], stream), "moe_forward_host")
        return y

    def poison_workspace(self, byte: int = 0xFF, stream=None):
        _check(moe_debug_poison_workspace(self.ctx, byte, stream), "moe_debug_poison_workspace")

    def route(self, x: torch.Tensor, stream=None):
        T = x.shape[0]
        idx = torch.empty((T, self.shape.top_k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, self.shape.top_k), dtype=torch.float32, device=x.device)
        _check(moe_route(self.ctx, x.contiguous(), T, idx, w, stream), "moe_route")
        return idx, w

    def quantize(self, x: torch.Tensor, stream=None):
        T, H = x.shape
        codes = torch.empty((T, H), dtype=torch.uint8, device=x.device)
        scales = torch.empty((T, H // 128), dtype=torch.float32, device=x.device)
        _check(moe_quantize(self.ctx, x.contiguous(), T, codes, scales, stream), "moe_quantize")
        return codes, scales

    def add_rmsnorm_quantize(self, residual: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor,
                             eps: float, h_out=None, xn_out=None, stream=None):
        """Residual add + RMS norm + the normed rows' FP8 groups, one launch.
        Returns (h, xn, codes, scales); h_out / xn_out may be `residual` or `x`
        for an in-place update."""
        for t in (residual, x, gamma):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("residual, x and gamma must be contiguous bf16 CUDA tensors")
        T, H = x.shape
        if residual.shape != x.shape or gamma.shape != (H,):
            raise ValueError("residual and x must be [rows, H] and gamma [H]")
        h_out = torch.empty_like(x) if h_out is None else h_out
        xn_out = torch.empty_like(x) if xn_out is None else xn_out
        codes = torch.empty((T, H), dtype=torch.uint8, device=x.device)
        scales = torch.empty((T, H // 128), dtype=torch.float32, device=x.device)
        _check(moe_add_rmsnorm_quantize(self.ctx, residual, x, gamma, eps, T, h_out, xn_out,
                                        codes, scales, stream), "moe_add_rmsnorm_quantize")
        return h_out, xn_out, codes, scales

    def expert_activations(self, rows: int, stream=None):
        k, I = self.shape.top_k, self.shape.inter
        dev = torch.device("cuda", self.device)
        hq = torch.empty((rows, k, I), dtype=torch.uint8, device=dev)
        sh = torch.empty((rows, k, I // 128), dtype=torch.float32, device=dev)
        _check(moe_expert_activations(self.ctx, rows, hq, sh, stream), "moe_expert_activations")
        return hq, sh

    def forward_codes(self, rows: int, stream=None):
        """The e4m3 codes and group scales of x that the experts of the most
        recent forward read: ([rows, k, H] uint8, [rows, k, H/128] fp32)."""
        k, H = self.shape.top_k, self.shape.hidden
        dev = torch.device("cuda", self.device)
        codes = torch.empty((rows, k, H), dtype=torch.uint8, device=dev)
        scales = torch.empty((rows, k, H // 128), dtype=torch.float32, device=dev)
        _check(moe_forward_codes(self.ctx, rows, codes, scales, stream), "moe_forward_codes")
        return codes, scales

    def profile(self, x: torch.Tensor, y: torch.Tensor, stream=None):
        rc, stages = moe_profile_forward(self.ctx, x, y, x.shape[0], stream)
        _check(rc, "moe_profile_forward")
        return stages

    def device_status(self) -> int:
        return moe_last_device_status(self.ctx)


class MoEChain:
    """Layers in sequence (each a MoELayer that must outlive the chain): the
    output of layer l is the input of layer l + 1."""

    def __init__(self, layers):
        self.layers = list(layers)
        rc, h = moe_chain_create([net.ctx for net in self.layers])
        _check(rc, "moe_chain_create")
        self.chain = h

    def close(self):
        if getattr(self, "chain", None):
            moe_chain_destroy(self.chain)
            self.chain = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x: torch.Tensor, y_all: torch.Tensor | None = None, stream=None):
        """x [rows, H] bf16 -> every layer's output [n_layers, rows, H]."""
        if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2:
            raise ValueError("x must be a 2-D bf16 CUDA tensor")
        x = x.contiguous()
        if y_all is None:
            y_all = torch.empty((len(self.layers),) + tuple(x.shape), dtype=x.dtype,
                                device=x.device)
        _check(moe_chain_forward(self.chain, x, y_all, x.shape[0], stream), "moe_chain_forward")
        return y_all
