"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin ties one part of the oracle to a closed form, a standard, a library
routine it does not use, or a brute-force restatement on tiny inputs.  The
planted-mistake test at the end runs every pin with one error planted in the
oracle at a time and requires at least one pin to turn red for each.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- independent helpers (library routines, not the oracle) --------------

def torch_e4m3_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(codes, np.uint8).copy()).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_e4m3_encode(v: np.ndarray) -> np.ndarray:
    """PyTorch's float8 cast (RNE); defined here only for |v| < 464."""
    t = torch.from_numpy(np.asarray(v, np.float32).copy())
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def np_bf16_round(v) -> np.ndarray:
    """Round doubles in the bf16 normal range to 8 significant bits, ties to even."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)
    nz = v != 0
    assert np.all(np.abs(v[nz]) > 2.0 ** -120) and np.all(np.abs(v) < 2.0 ** 120)
    return np.where(nz, np.ldexp(np.round(m * 256.0), e - 8), v)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16).copy()).view(
        torch.bfloat16).to(torch.float64).numpy()


def torch_quant_groups(v32: np.ndarray, group=128):
    """Quantise fp32 rows in groups with PyTorch fp32 ops and its float8 cast."""
    t = torch.from_numpy(np.asarray(v32, np.float32).copy())
    *lead, n = t.shape
    g = t.reshape(*lead, n // group, group)
    amax = g.abs().amax(-1)
    s = torch.where(amax > 0, amax / torch.tensor(448.0), torch.ones_like(amax))
    q = (g / s[..., None]).to(torch.float8_e4m3fn)
    return (q.view(torch.uint8).reshape(*lead, n).numpy(), s.numpy(),
            (q.to(torch.float64) * s.to(torch.float64)[..., None]).reshape(*lead, n).numpy())


def silu(a):
    return a / (1.0 + np.exp(-a))


def brute_force_layer(layer: dict, x_bits: np.ndarray, group=128, act_per_row=False):
    """Dense restatement on tiny shapes: every expert for every row, masked by a
    top-k found by scanning all k-subsets; quantisation through PyTorch's cast
    (one scale per row of x and of h when act_per_row)."""
    x = bits_to_f64(x_bits)
    T, H = x.shape
    E, I2, _ = layer["w13"].shape
    I = I2 // 2
    k = layer["top_k"]
    wr = layer["router"].astype(np.float64)
    logits = x @ wr.T
    lf = logits.astype(np.float32)
    # dequantised weights
    dec = torch_e4m3_decode(np.arange(256))
    w13 = dec[layer["w13"]] * np.repeat(np.repeat(layer["s13"], group, 1), group, 2)
    w2 = dec[layer["w2"]] * np.repeat(np.repeat(layer["s2"], group, 1), group, 2)
    ws13 = bits_to_f64(layer["ws13"])
    ws2 = bits_to_f64(layer["ws2"])
    gate = bits_to_f64(layer["shared_gate"])
    _, _, xd = torch_quant_groups(x.astype(np.float32), H if act_per_row else group)
    out = np.zeros((T, H))
    sel_all = []
    for t in range(T):
        chosen = None
        for S in itertools.combinations(range(E), k):
            Sset = set(S)
            ok = all((lf[t, e] > lf[t, f]) or (lf[t, e] == lf[t, f] and e < f)
                     for e in S for f in range(E) if f not in Sset)
            if ok:
                assert chosen is None
                chosen = S
        order = sorted(chosen, key=lambda e: (-lf[t, e], e))
        sel_all.append(order)
        ls = logits[t, order]
        wts = np.exp(ls - ls.max())
        wts = wts / wts.sum()
        for j, e in enumerate(order):
            z = np_bf16_round(w13[e] @ xd[t])
            h = (silu(z[:I]) * z[I:]).astype(np.float32)
            _, _, hd = torch_quant_groups(h[None, :], I if act_per_row else group)
            d = np_bf16_round(w2[e] @ hd[0])
            out[t] += wts[j] * d
        zs = np_bf16_round(ws13 @ x[t])
        Is = zs.size // 2
        hs = np_bf16_round(silu(zs[:Is]) * zs[Is:])
        ds = np_bf16_round(ws2 @ hs)
        gam = 1.0 / (1.0 + np.exp(-(x[t] @ gate)))
        out[t] += gam * ds
    return out, np.array(sel_all)


def tiny_layer(seed=0, T=4):
    L = W.to_numpy_layer(W.make_layer(W.TINY, seed))
    x = W.bf16_bits(W.make_x(W.TINY, T, seed))
    return L, x


# ---- pins ------------------------------------------------------------------

def pin_e4m3_table_vs_torch():
    t = oracle.e4m3_table()
    ref = torch_e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(t), nan)
    assert np.array_equal(t[~nan], ref[~nan])
    assert np.array_equal(np.signbit(t[~nan]), np.signbit(ref[~nan]))


def pin_e4m3_spec_points():
    t = oracle.e4m3_table()
    with open(os.path.join(GOLDEN, "e4m3_ocp_points.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            c, v = int(code, 16), float(val)
            if math.isnan(v):
                assert math.isnan(t[c])
            else:
                assert t[c] == v and math.copysign(1, t[c]) == math.copysign(1, v), (code, t[c])


def pin_e4m3_roundtrip():
    t = oracle.e4m3_table()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(t[codes]), codes)


def pin_e4m3_boundaries():
    t = oracle.e4m3_table()
    pos = t[:0x7F]  # 0x00..0x7E increasing
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2  # exact: at most 5 significant bits
    mid32 = mid.astype(np.float32)
    assert np.array_equal(mid32.astype(np.float64), mid)
    codes_lo = np.arange(0x7E, dtype=np.uint8)
    even = np.where(codes_lo % 2 == 0, codes_lo, codes_lo + 1).astype(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(mid32), even)
    assert np.array_equal(oracle.e4m3_encode(-mid32), even | 0x80)
    below = np.nextafter(mid32, np.float32(-np.inf))
    above = np.nextafter(mid32, np.float32(np.inf))
    assert np.array_equal(oracle.e4m3_encode(below), codes_lo)
    assert np.array_equal(oracle.e4m3_encode(above), codes_lo + 1)
    sat = np.array([448, 449, 463.99, 464, 465, 1e9, np.inf, 3.0e38], np.float32)
    assert np.all(oracle.e4m3_encode(sat) == 0x7E)
    assert np.all(oracle.e4m3_encode(-sat) == 0xFE)
    assert oracle.e4m3_encode([np.nan])[0] == 0x7F
    assert oracle.e4m3_encode([-0.0])[0] == 0x80
    assert oracle.e4m3_encode([2.0 ** -10])[0] == 0x00
    assert oracle.e4m3_encode([-(2.0 ** -10)])[0] == 0x80
    assert oracle.e4m3_encode([np.nextafter(np.float32(2.0 ** -10), np.float32(1))])[0] == 0x01


def pin_e4m3_random_vs_torch():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-14, 9, 200_000))).astype(np.float32)
    v = v[np.abs(v) < 460]
    assert np.array_equal(oracle.e4m3_encode(v), torch_e4m3_encode(v))


def pin_bf16_vs_torch():
    rng = np.random.default_rng(2)
    f = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-60, 60, 200_000))).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_from_double(f.astype(np.float64)), ref)
    # midpoints between adjacent bf16 values (exact doubles) go to the even one
    b = np.arange(0x0080, 0x7F7F, 7, dtype=np.uint16)
    lo, hi = bits_to_f64(b), bits_to_f64(b + 1)
    even = np.where(b % 2 == 0, b, b + 1).astype(np.uint16)
    assert np.array_equal(oracle.bf16_from_double((lo + hi) / 2), even)
    # just off the midpoint by far less than a float32 ulp: a single rounding
    eps = (hi - lo) * 2.0 ** -30
    assert np.array_equal(oracle.bf16_from_double((lo + hi) / 2 + eps), b + 1)
    assert np.array_equal(oracle.bf16_from_double((lo + hi) / 2 - eps), b)
    assert np.array_equal(oracle.bf16_from_double(np_bf16_round(f[np.abs(f) > 1e-30]
                                                                .astype(np.float64))),
                          oracle.bf16_from_double(f[np.abs(f) > 1e-30].astype(np.float64)))


def pin_quant_special_cases():
    t = oracle.e4m3_table()
    rng = np.random.default_rng(3)
    # the amax element always lands on +-448
    for _ in range(50):
        v = (rng.standard_normal(128) * 10 ** rng.uniform(-3, 3)).astype(np.float32)
        c, s = oracle.quant_row(v)
        i = np.argmax(np.abs(v))
        assert c[i] == (0xFE if v[i] < 0 else 0x7E)
    # a group whose max is 448 and whose values are e4m3 values: scale 1, codes exact
    codes = rng.integers(0, 0x7E, 128).astype(np.uint8) | (rng.integers(0, 2, 128) * 0x80).astype(np.uint8)
    codes[17] = 0x7E
    v = t[codes].astype(np.float32)
    c, s = oracle.quant_row(v)
    assert s[0] == 1.0 and np.array_equal(c, codes)
    # powers of two: value 2^p with amax 2^q: x/s = 448 * 2^(p-q)
    v = np.zeros(128, np.float32)
    v[0] = 4.0
    v[1] = 1.0
    v[2] = -0.25
    c, s = oracle.quant_row(v)
    assert s[0] == np.float32(4.0) / np.float32(448.0)
    assert t[c[0]] == 448 and t[c[1]] == 112 and t[c[2]] == -28
    # all-zero group: scale 1, zero codes (signs kept)
    v = np.zeros(128, np.float32)
    v[5] = -0.0
    c, s = oracle.quant_row(v)
    assert s[0] == 1.0 and np.all(c[np.arange(128) != 5] == 0) and c[5] == 0x80
    # one non-zero value
    v = np.zeros(256, np.float32)
    v[200] = -3.5
    c, s = oracle.quant_row(v)
    assert s[0] == 1.0 and s[1] == np.float32(3.5) / np.float32(448)
    assert c[200] == 0xFE and np.count_nonzero(c) == 1


def pin_quant_vs_torch():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((64, 512)).astype(np.float32)
    v[3] *= 1e-20
    v[7] *= 1e20
    ref_c, ref_s, _ = torch_quant_groups(v)
    for r in range(v.shape[0]):
        c, s = oracle.quant_row(v[r])
        assert np.array_equal(s, ref_s[r]) and np.array_equal(c, ref_c[r]), r


def pin_router_topk_vs_full_sort():
    rng = np.random.default_rng(5)
    E, H = 32, 256
    for trial in range(20):
        wr = (rng.standard_normal((E, H)) * 0.02).astype(np.float32)
        if trial % 2:
            wr[5] = wr[9]     # duplicate rows -> exactly equal logits
            wr[20] = wr[3]
            wr[31] = wr[0]
        x = W.bf16_bits(torch.from_numpy(rng.standard_normal((1, H)).astype(np.float32))
                        .to(torch.bfloat16))[0]
        for k in (1, 4, 8, E):
            logits, idx, w = oracle.router_row(x, wr, k)
            ref_logits = bits_to_f64(x) @ wr.astype(np.float64).T
            assert np.allclose(logits, ref_logits, rtol=1e-12, atol=1e-15)
            full = sorted(range(E), key=lambda e: (-np.float32(logits[e]), e))
            assert list(idx) == full[:k]
    # all logits equal -> the first k indices, equal weights
    logits, idx, w = oracle.router_row(np.zeros(H, np.uint16), np.zeros((E, H), np.float32), 8)
    assert list(idx) == list(range(8)) and np.all(w == 0.125)


def pin_router_softmax():
    import scipy.special
    rng = np.random.default_rng(6)
    E, H = 16, 256
    wr = (rng.standard_normal((E, H)) * 0.05).astype(np.float32)
    x = W.bf16_bits(torch.from_numpy(rng.standard_normal((1, H)).astype(np.float32))
                    .to(torch.bfloat16))[0]
    logits, idx, w = oracle.router_row(x, wr, 4)
    assert abs(w.sum() - 1.0) < 1e-15
    p = scipy.special.softmax(logits)
    assert np.allclose(w, p[idx] / p[idx].sum(), rtol=1e-13)
    logits, idx, w = oracle.router_row(x, wr, E)
    assert np.allclose(w, p[idx], rtol=1e-13)


def pin_block_fp8_dot():
    rng = np.random.default_rng(7)
    dec = torch_e4m3_decode(np.arange(256))
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    for K in (128, 512, 2048):
        a = rng.choice(finite, K).astype(np.uint8)
        w = rng.choice(finite, K).astype(np.uint8)
        sa = rng.uniform(0.001, 0.1, K // 128).astype(np.float32)
        sw = rng.uniform(0.001, 0.1, K // 128).astype(np.float32)
        got = oracle.block_fp8_dot(a, sa, w, sw)
        ref = float(np.dot(dec[a] * np.repeat(sa, 128), dec[w] * np.repeat(sw, 128)))
        assert abs(got - ref) <= 1e-12 * np.sum(np.abs(dec[a] * np.repeat(sa, 128) * dec[w] *
                                                      np.repeat(sw, 128)))
        # unit scales and codes in {0, +1, -1}: small exact integers
        a = rng.choice(np.array([0x00, 0x38, 0xB8], np.uint8), K)
        w = rng.choice(np.array([0x00, 0x38, 0xB8], np.uint8), K)
        one = np.ones(K // 128, np.float32)
        assert oracle.block_fp8_dot(a, one, w, one) == float(np.dot(dec[a], dec[w]))


def pin_layer_brute_force():
    for seed, T in ((0, 4), (11, 3)):
        L, x = tiny_layer(seed, T)
        r = oracle.moe_rows(L, x, trace=True)
        ref, sel = brute_force_layer(L, x)
        assert np.array_equal(r.trace["idx"], sel)
        assert np.allclose(r.y_ref, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())


def pin_layer_brute_force_per_row_scale():
    """The one-scale-per-row variant against the dense restatement quantising
    each row of x and of h as a single group; it must differ from 1 x 128."""
    L, x = tiny_layer(7, 3)
    r = oracle.moe_rows(L, x, trace=True, act_per_row=True)
    ref, sel = brute_force_layer(L, x, act_per_row=True)
    assert np.array_equal(r.trace["idx"], sel)
    assert np.allclose(r.y_ref, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())
    assert np.all(r.trace["sx"] == r.trace["sx"][:, :1])
    assert not np.array_equal(r.y_ref, oracle.moe_rows(L, x).y_ref)


def pin_layer_closed_form_all_selected():
    """E = k, zero router -> every weight 1/k; identical experts -> the routed
    sum is one dense block-FP8 SwiGLU; zero shared weights -> gamma * 0."""
    shape = W.MoEShape(hidden=256, n_experts=4, top_k=4, inter=128, shared_inter=128)
    L = W.to_numpy_layer(W.make_layer(shape, 5, experts=[0]))
    for e in range(1, 4):
        for n in ("w13", "s13", "w2", "s2"):
            L[n][e] = L[n][0]
    L["router"][:] = 0
    L["ws13"][:] = 0
    L["ws2"][:] = 0
    x = W.bf16_bits(W.make_x(shape, 3, 5))
    r = oracle.moe_rows(L, x, trace=True)
    assert np.all(r.trace["w"] == 0.25)
    assert np.array_equal(r.trace["idx"], np.tile(np.arange(4), (3, 1)))
    # the dense SwiGLU of one expert, restated with library routines
    dec = torch_e4m3_decode(np.arange(256))
    w13 = dec[L["w13"][0]] * np.repeat(np.repeat(L["s13"][0], 128, 0), 128, 1)
    w2 = dec[L["w2"][0]] * np.repeat(np.repeat(L["s2"][0], 128, 0), 128, 1)
    _, _, xd = torch_quant_groups(bits_to_f64(x).astype(np.float32))
    for t in range(3):
        z = np_bf16_round(w13 @ xd[t])
        h = (silu(z[:128]) * z[128:]).astype(np.float32)
        _, _, hd = torch_quant_groups(h[None])
        d = np_bf16_round(w2 @ hd[0])
        assert np.array_equal(r.y_ref[t], d)   # 4 * (1/4) * d, exactly


def pin_layer_shared_only():
    """Zero routed weights and a zero gate vector: y = sigmoid(0) * shared = ds / 2."""
    L, x = tiny_layer(3, 2)
    L["w13"][:] = 0
    L["shared_gate"][:] = 0
    r = oracle.moe_rows(L, x)
    xf = bits_to_f64(x)
    zs = np_bf16_round(xf @ bits_to_f64(L["ws13"]).T)
    hs = np_bf16_round(silu(zs[:, :128]) * zs[:, 128:])
    ds = np_bf16_round(hs @ bits_to_f64(L["ws2"]).T)
    assert np.array_equal(r.y_ref, 0.5 * ds)


def pin_router_bf16_logits():
    """The bf16-logit router variant: logits from numpy's float64 products,
    rounded to fp32 and then bf16 by PyTorch's casts; the k largest by a full
    stable sort of (-logit, expert); weights by scipy's softmax over the
    selection.  On these rows the variant must meet exact ties among the first
    k + 1 and pick differently from the fp32 router at least once."""
    from scipy.special import softmax
    shape = W.FULL
    E, k = shape.n_experts, shape.top_k
    wr = W.make_router(shape, 21).numpy()
    xb = W.bf16_bits(W.make_x(shape, 24, 21))
    lg = bits_to_f64(xb) @ wr.astype(np.float64).T
    lb = torch.from_numpy(lg).float().to(torch.bfloat16).double().numpy()
    differs = ties = 0
    for t in range(xb.shape[0]):
        _, idx, w = oracle.router_row(xb[t], wr, k, bf16_logits=True)
        order = np.lexsort((np.arange(E), -lb[t]))
        assert np.array_equal(idx, order[:k])
        assert np.allclose(w, softmax(lb[t][order[:k]]), rtol=1e-12, atol=0)
        top = lb[t][order[:k + 1]]
        ties += int(np.any(top[1:] == top[:-1]))
        differs += int(not np.array_equal(idx, oracle.router_row(xb[t], wr, k)[1]))
    assert ties > 0 and differs > 0, (ties, differs)


def _addnorm_expected_from_xn(xn_bits):
    """Codes and scales of bf16 rows, through the PyTorch restatement."""
    codes, scales, _ = torch_quant_groups(bits_to_f64(xn_bits).astype(np.float32))
    return codes, scales


def pin_addnorm_constant_rows():
    """Constant rows with eps = 0 normalise to sign(h) exactly, so xn is
    +-gamma bit for bit and its FP8 groups are gamma's."""
    H = 256
    res = np.array([-3.0, 0.5, 2.0])[:, None] * np.ones((1, H))
    x = np.array([1.0, 0.25, -6.0])[:, None] * np.ones((1, H))
    gam = torch.from_numpy(1.0 + 0.1 * np.random.default_rng(4).standard_normal(H))
    gbits = W.bf16_bits(gam.to(torch.bfloat16))
    rb = W.bf16_bits(torch.from_numpy(res).to(torch.bfloat16))
    xb = W.bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    h, xn, codes, scales = oracle.add_rmsnorm(rb, xb, gbits, 0.0)
    assert np.array_equal(bits_to_f64(h), res + x)
    want = np.sign(res + x) * bits_to_f64(gbits)[None, :]
    assert np.array_equal(bits_to_f64(xn), want)
    c, s = _addnorm_expected_from_xn(W.bf16_bits(torch.from_numpy(want).to(torch.bfloat16)))
    assert np.array_equal(codes, c) and np.array_equal(scales, s)


def pin_addnorm_eps_inside_root():
    """h = 2 everywhere and eps = 3 * 2^2: 1 / sqrt(4 + 12) = 1/4, so xn = gamma / 2."""
    H = 256
    gam = torch.from_numpy(1.0 + 0.1 * np.random.default_rng(5).standard_normal(H))
    gbits = W.bf16_bits(gam.to(torch.bfloat16))
    rb = W.bf16_bits(torch.full((1, H), 2.0, dtype=torch.bfloat16))
    xb = W.bf16_bits(torch.zeros((1, H), dtype=torch.bfloat16))
    _, xn, _, _ = oracle.add_rmsnorm(rb, xb, gbits, 12.0)
    assert np.array_equal(bits_to_f64(xn)[0], bits_to_f64(gbits) / 2)


def pin_addnorm_vs_library():
    """Seeded rows against PyTorch's float64 RMS norm (torch.nn.functional.rms_norm),
    numpy's bf16 rounding of the sums, and the PyTorch group quantiser."""
    shape = W.FULL
    r, x, g = W.make_addnorm(shape, 5, 7)
    h, xn, codes, scales = oracle.add_rmsnorm(W.bf16_bits(r), W.bf16_bits(x), W.bf16_bits(g),
                                              W.NORM_EPS)
    hs = np_bf16_round(r.double().numpy() + x.double().numpy())
    assert np.array_equal(bits_to_f64(h), hs)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(hs), (shape.hidden,),
                                       weight=g.double(), eps=W.NORM_EPS).numpy()
    assert np.array_equal(bits_to_f64(xn), np_bf16_round(ref))
    c, s = _addnorm_expected_from_xn(xn)
    assert np.array_equal(codes, c) and np.array_equal(scales, s)


PINS = [pin_e4m3_table_vs_torch, pin_e4m3_spec_points, pin_e4m3_roundtrip,
        pin_e4m3_boundaries, pin_e4m3_random_vs_torch, pin_bf16_vs_torch,
        pin_quant_special_cases, pin_quant_vs_torch, pin_router_topk_vs_full_sort,
        pin_router_softmax, pin_block_fp8_dot, pin_layer_brute_force,
        pin_layer_closed_form_all_selected, pin_layer_shared_only,
        pin_addnorm_constant_rows, pin_addnorm_eps_inside_root, pin_addnorm_vs_library,
        pin_router_bf16_logits, pin_layer_brute_force_per_row_scale]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


@pytest.mark.parametrize("mut", [oracle.MUT_TIE_HIGH, oracle.MUT_SCALE_447,
                                 oracle.MUT_ENC_TRUNC, oracle.MUT_DROP_EXPERT,
                                 oracle.MUT_SWAP_GATE_UP, oracle.MUT_SCALE_TRANSPOSE,
                                 oracle.MUT_GATE_SIGN, oracle.MUT_NO_RENORM,
                                 oracle.MUT_ENC_TIE_UP, oracle.MUT_NORM_EPS_OUTSIDE,
                                 oracle.MUT_NORM_NO_RESIDUAL, oracle.MUT_NORM_GAMMA_PLUS_ONE,
                                 oracle.MUT_NORM_QUANT_UNROUNDED,
                                 oracle.MUT_ROUTER_BF16_IGNORED, oracle.MUT_PER_ROW_IGNORED])
def test_planted_mistake_turns_a_pin_red(mut):
    failed = []
    with oracle.mutation(mut):
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
    assert failed, f"mutation {mut} went unnoticed by every pin"


def test_e4m3_encode_exhaustive_range():
    """Every fp32 value in [2^-12, 448) and its negative, against PyTorch's cast."""
    start = np.float32(2.0 ** -12).view(np.uint32)
    stop = np.float32(448.0).view(np.uint32)
    step = 1 << 22
    for a in range(int(start), int(stop), step):
        bits = np.arange(a, min(a + step, int(stop)), dtype=np.uint32)
        v = bits.view(np.float32)
        ref = torch_e4m3_encode(v)
        got = oracle.e4m3_encode(v)
        assert np.array_equal(got, ref), hex(a)
        assert np.array_equal(oracle.e4m3_encode(-v[::97]), ref[::97] | 0x80)


def test_quantisation_effect_matches_pages():
    """The Precision section of the one-GPU pull request says that skipping the
    activation quantisation moves each MoE block's output by about 1e-2
    relative.  Full-width layer (H=2048, 256 experts top-8, I=512), one row."""
    shape = W.FULL
    wr = W.make_router(shape, 1)
    x = W.make_x(shape, 1, 1)
    _, idx, _ = oracle.router_row(W.bf16_bits(x)[0], wr.numpy(), shape.top_k)
    L = W.to_numpy_layer(W.make_layer(shape, 1, experts=idx))
    xb = W.bf16_bits(x)
    on = oracle.moe_rows(L, xb).y_ref
    off = oracle.moe_rows(L, xb, act_quant=False).y_ref
    rel = np.linalg.norm(on - off) / np.linalg.norm(off)
    assert 2e-3 < rel < 5e-2, rel
