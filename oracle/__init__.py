"""CPU oracle of the block-FP8 MoE layer (test infrastructure only).

The oracle is the plain, slow definition of what the layer computes
(`moe_oracle.c`, single-threaded, double accumulation).  Only the test suite,
`__graft_entry__.smoke()` and the benchmark's CPU-baseline leg may import this
package; the CUDA library never does, and the two share no code.

`build()` compiles the C file with gcc into `oracle/_build/`.  Compilation uses
`-ffp-contract=off` so that x86-64 and aarch64 hosts give the same doubles.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

# planted-mistake selectors (see moe_oracle.c)
MUT_NONE = 0
MUT_TIE_HIGH = 1
MUT_SCALE_447 = 2
MUT_ENC_TRUNC = 3
MUT_DROP_EXPERT = 4
MUT_SWAP_GATE_UP = 5
MUT_SCALE_TRANSPOSE = 6
MUT_GATE_SIGN = 7
MUT_NO_RENORM = 8
MUT_ENC_TIE_UP = 9
MUT_NORM_EPS_OUTSIDE = 10
MUT_NORM_NO_RESIDUAL = 11
MUT_NORM_GAMMA_PLUS_ONE = 12
MUT_NORM_QUANT_UNROUNDED = 13
MUT_ROUTER_BF16_IGNORED = 14
MUT_PER_ROW_IGNORED = 15


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Layer(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("k", ctypes.c_int),
                ("I", ctypes.c_int), ("Is", ctypes.c_int), ("G", ctypes.c_int),
                ("w13", ctypes.c_void_p), ("s13", ctypes.c_void_p),
                ("w2", ctypes.c_void_p), ("s2", ctypes.c_void_p),
                ("wr", ctypes.c_void_p), ("ws13", ctypes.c_void_p),
                ("ws2", ctypes.c_void_p), ("gate", ctypes.c_void_p),
                ("router_bf16", ctypes.c_int), ("act_per_row", ctypes.c_int)]


class _Trace(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("logits", "idx", "w", "xq", "sx", "z", "hq", "sh", "d",
                 "zs", "hs", "ds", "gamma")]


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        L.orc_set_mutation.argtypes = [ctypes.c_int]
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_e4m3_table.argtypes = [ctypes.c_void_p]
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.orc_bf16_from_double_array.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                                 ctypes.c_void_p]
        L.orc_bf16_from_double.argtypes = [ctypes.c_double]
        L.orc_bf16_from_double.restype = ctypes.c_uint16
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_double.restype = ctypes.c_double
        L.orc_quant_row.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_void_p, ctypes.c_void_p]
        L.orc_add_rmsnorm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]
        L.orc_router.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                 ctypes.c_void_p, ctypes.c_void_p]
        L.orc_router_bf16.argtypes = L.orc_router.argtypes
        L.orc_block_fp8_dot.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
        L.orc_block_fp8_dot.restype = ctypes.c_double
        L.orc_moe_rows.argtypes = [ctypes.POINTER(_Layer), ctypes.c_void_p, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.POINTER(_Trace)]
        L.orc_moe_rows.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


class mutation:
    """Context manager that plants one mistake in the oracle (tests only)."""

    def __init__(self, m: int):
        self.m = m

    def __enter__(self):
        lib().orc_set_mutation(self.m)
        return self

    def __exit__(self, *exc):
        lib().orc_set_mutation(MUT_NONE)
        return False


# ---- scalar / row helpers -------------------------------------------------

def e4m3_table() -> np.ndarray:
    out = np.zeros(256, np.float64)
    lib().orc_e4m3_table(_p(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    v = _c(values, np.float32).ravel()
    out = np.zeros(v.size, np.uint8)
    lib().orc_e4m3_encode_array(_p(v), v.size, _p(out))
    return out


def bf16_from_double(values) -> np.ndarray:
    v = _c(values, np.float64).ravel()
    out = np.zeros(v.size, np.uint16)
    lib().orc_bf16_from_double_array(_p(v), v.size, _p(out))
    return out


def quant_row(values, group: int = 128):
    """Quantise one row of fp32 values in groups -> (codes uint8, scales f32)."""
    v = _c(values, np.float32).ravel()
    n = v.size
    codes = np.zeros(n, np.uint8)
    scales = np.zeros(n // group, np.float32)
    lib().orc_quant_row(_p(v), n, group, _p(codes), _p(scales))
    return codes, scales


def add_rmsnorm(residual_bits, x_bits, gamma_bits, eps: float, group: int = 128):
    """Residual add, plain-gamma RMS norm and the FP8 groups of the normed rows.

    bf16 bit arrays residual, x [T, H] and gamma [H] -> (h uint16 [T, H],
    xn uint16 [T, H], codes uint8 [T, H], scales f32 [T, H/group]).
    """
    r = _c(residual_bits, np.uint16)
    x = _c(x_bits, np.uint16)
    g = _c(gamma_bits, np.uint16).ravel()
    T, H = x.shape
    assert r.shape == x.shape and g.size == H and H % group == 0
    h = np.zeros((T, H), np.uint16)
    xn = np.zeros((T, H), np.uint16)
    codes = np.zeros((T, H), np.uint8)
    scales = np.zeros((T, H // group), np.float32)
    lib().orc_add_rmsnorm(_p(r), _p(x), _p(g), T, H, group, float(eps), _p(h), _p(xn),
                          _p(codes), _p(scales))
    return h, xn, codes, scales


def router_row(x_bf16_bits, wr, k: int, bf16_logits: bool = False):
    """Router for one row -> (logits f64 [E], idx int32 [k], w f64 [k]).
    bf16_logits: the variant that routes on bf16-rounded logits."""
    x = _c(x_bf16_bits, np.uint16).ravel()
    wr = _c(wr, np.float32)
    E, H = wr.shape
    logits = np.zeros(E, np.float64)
    idx = np.zeros(k, np.int32)
    w = np.zeros(k, np.float64)
    fn = lib().orc_router_bf16 if bf16_logits else lib().orc_router
    fn(_p(x), H, _p(wr), E, k, _p(logits), _p(idx), _p(w))
    return logits, idx, w


def block_fp8_dot(a_codes, a_scales, w_codes, w_scales, group: int = 128) -> float:
    a = _c(a_codes, np.uint8).ravel()
    s = _c(a_scales, np.float32).ravel()
    w = _c(w_codes, np.uint8).ravel()
    ws = _c(w_scales, np.float32).ravel()
    return lib().orc_block_fp8_dot(_p(a), _p(s), _p(w), _p(ws), a.size, group)


# ---- the layer ------------------------------------------------------------

@dataclass
class OracleResult:
    y_bf16: np.ndarray     # uint16 bits [T, H]
    y_ref: np.ndarray      # float64 [T, H]
    trace: dict | None


def moe_rows(layer: dict, x_bf16_bits, act_quant: bool = True, trace: bool = False,
             group: int = 128, router_bf16: bool = False,
             act_per_row: bool = False) -> OracleResult:
    """Run the layer on T rows.

    `layer` holds numpy arrays with the names of the C-ABI weight struct:
    w13 uint8 [E,2I,H], s13 f32 [E,2I/G,H/G], w2 uint8 [E,H,I], s2 f32 [E,H/G,I/G],
    router f32 [E,H], ws13 uint16(bf16) [2Is,H], ws2 uint16 [H,Is],
    shared_gate uint16 [H], and the scalar `top_k`.
    Variants: router_bf16 routes on bf16-rounded logits; act_per_row gives x
    and the SwiGLU rows one activation scale per row instead of per 1 x group.
    """
    x = _c(x_bf16_bits, np.uint16)
    T, H = x.shape
    w13 = _c(layer["w13"], np.uint8)
    E, I2, H_ = w13.shape
    assert H_ == H
    I = I2 // 2
    ws13 = _c(layer["ws13"], np.uint16)
    Is = ws13.shape[0] // 2
    k = int(layer["top_k"])
    arrs = dict(w13=w13, s13=_c(layer["s13"], np.float32), w2=_c(layer["w2"], np.uint8),
                s2=_c(layer["s2"], np.float32), wr=_c(layer["router"], np.float32),
                ws13=ws13, ws2=_c(layer["ws2"], np.uint16),
                gate=_c(layer["shared_gate"], np.uint16))
    L = _Layer(H, E, k, I, Is, group, *[_p(arrs[n]) for n in
                                         ("w13", "s13", "w2", "s2", "wr", "ws13", "ws2", "gate")],
               1 if router_bf16 else 0, 1 if act_per_row else 0)
    y = np.zeros((T, H), np.uint16)
    yr = np.zeros((T, H), np.float64)
    tr_arrays = None
    tr = _Trace()
    if trace:
        G = group
        tr_arrays = dict(
            logits=np.zeros((T, E), np.float64), idx=np.zeros((T, k), np.int32),
            w=np.zeros((T, k), np.float64), xq=np.zeros((T, H), np.uint8),
            sx=np.zeros((T, H // G), np.float32), z=np.zeros((T, k, 2 * I), np.uint16),
            hq=np.zeros((T, k, I), np.uint8), sh=np.zeros((T, k, I // G), np.float32),
            d=np.zeros((T, k, H), np.uint16), zs=np.zeros((T, 2 * Is), np.uint16),
            hs=np.zeros((T, Is), np.uint16), ds=np.zeros((T, H), np.uint16),
            gamma=np.zeros(T, np.float64))
        for n, a in tr_arrays.items():
            setattr(tr, n, _p(a))
    rc = lib().orc_moe_rows(ctypes.byref(L), _p(x), T, 1 if act_quant else 0,
                            _p(y), _p(yr), ctypes.byref(tr))
    if rc != 0:
        raise ValueError(f"oracle refused the layer shape (rc={rc})")
    return OracleResult(y, yr, tr_arrays)
