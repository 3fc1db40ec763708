"""CUDA path against the CPU oracle, through the C ABI (needs a GB300)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity import (bits, check_forward_codes, check_output, check_topk, hq_agreement,
                    oracle_rows)

pytestmark = pytest.mark.gpu

m = pytest.importorskip("block_fp8_mixture_router_gb300")


def _shape(s: W.MoEShape) -> "m.LayerShape":
    return m.LayerShape(s.hidden, s.n_experts, s.top_k, s.inter, s.shared_inter, s.group)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    return torch.device("cuda", 0)


class Case:
    """A layer built on the GPU, loaded into a context, plus its host copy."""

    def __init__(self, wl: W.Workload, max_rows: int, dev, layer_idx: int = 0,
                 act_group: int | None = None):
        self.wl = wl
        self.shape = wl.shape
        seed = W.layer_seed(wl, layer_idx)
        self.layer = W.make_layer(wl.shape, seed, wl.x_kind, device=dev)
        shape = _shape(wl.shape)
        if act_group is not None:
            shape.act_group = act_group
        self.moe = m.MoELayer(shape, max_rows=max_rows)
        self.moe.load(self.layer)
        self._host = None
        self.seed = seed

    @property
    def host(self):
        if self._host is None:
            self._host = W.to_numpy_layer(self.layer)
        return self._host

    def x(self, rows, tag="x"):
        return W.make_x(self.shape, rows, self.seed, self.wl.x_kind, device="cuda", tag=tag)


# bar for the re-quantised SwiGLU codes (order-dependent, so not bit-exact):
# at least this fraction identical, and within one e4m3 step wherever the
# group scale agrees
HQ_SAME_MIN = 0.98
HQ_MAX_STEP = 1


def run_and_check(case: Case, x: torch.Tensor, sample_rows=None, path=m.PATH_AUTO,
                  threads=None, oracle_kw=None):
    """One forward on `path`, then every check against the oracle on the
    sampled rows (all rows by default): the FP8 codes and scales of x that the
    forward's experts read (read back from the forward itself, every rank's
    copy, bit-exact), the routing (bit-exact outside near ties), the routing
    weights, the re-quantised SwiGLU codes (held to a bar) and y."""
    case.moe.set_option(m.MOE_OPT_PATH, path)
    T = x.shape[0]
    y = case.moe.forward(x)
    fcodes, fscales = case.moe.forward_codes(T)
    hq, sh = case.moe.expert_activations(T)
    idx, w = case.moe.route(x)
    codes, scales = case.moe.quantize(x)
    torch.cuda.synchronize()
    rows = np.arange(T) if sample_rows is None else np.asarray(sample_rows)
    xb = bits(x)[rows]
    ref = oracle_rows(case.host, xb, threads=threads, trace=True, **(oracle_kw or {}))
    check_forward_codes(fcodes.cpu().numpy()[rows], fscales.cpu().numpy()[rows],
                        ref.trace["xq"], ref.trace["sx"])
    near, differ = check_topk(idx.cpu().numpy()[rows], ref.trace["logits"], case.shape.top_k)
    assert differ.sum() <= max(1, 0.02 * rows.size), f"{differ.sum()} rows routed differently"
    exact = ~differ
    assert np.array_equal(codes.cpu().numpy()[rows], ref.trace["xq"])
    assert np.array_equal(scales.cpu().numpy()[rows], ref.trace["sx"])
    wg = w.cpu().numpy()[rows]
    assert np.allclose(wg[exact], ref.trace["w"][exact], rtol=2e-5, atol=1e-7)
    same, step, s_ok = hq_agreement(hq.cpu().numpy()[rows], sh.cpu().numpy()[rows],
                                    ref.trace["hq"], ref.trace["sh"], rows_mask=exact)
    assert same >= HQ_SAME_MIN and step <= HQ_MAX_STEP, (same, step, s_ok)
    rel, mx = check_output(bits(y)[rows], ref.y_ref, rows_mask=exact)
    return y, ref, rel, mx


# ---- the tiny layer (H=256, 16 experts top-4, I=Is=128) ----------------------

@pytest.mark.parametrize("rows", [1, 4, 5, 16, 17, 40])
def test_tiny_layer(dev, rows):
    case = Case(W.WORKLOADS["tiny_t4"], 64, dev)
    x = case.x(rows)
    run_and_check(case, x)


@pytest.mark.parametrize("path", [m.PATH_AUTO, m.PATH_PROMPT, m.PATH_DECODE_CHAINED])
@pytest.mark.parametrize("rows", [1, 4, 9, 16])
def test_tiny_layer_every_path(dev, path, rows):
    case = Case(W.WORKLOADS["tiny_t4"], 64, dev)
    run_and_check(case, case.x(rows, tag=f"p{rows}"), path=path)


@pytest.mark.parametrize("path", [m.PATH_PROMPT, m.PATH_DECODE_CHAINED, m.PATH_DECODE_ROWS])
def test_full_layer_other_paths(full_case, path):
    x = full_case.x(11, tag="paths")
    try:
        run_and_check(full_case, x, path=path)
    finally:
        full_case.moe.set_option(m.MOE_OPT_PATH, m.PATH_AUTO)


# ---- full-width layers --------------------------------------------------------

@pytest.fixture(scope="module")
def full_case(dev):
    return Case(W.WORKLOADS["decode_t1"], 1024, dev)


def test_quantize_rounding_edges(full_case):
    """Groups whose quotients v/s fall exactly on e4m3 rounding midpoints (ties
    to even), on e4m3 values, in e4m3's subnormal range, and all-zero groups:
    the kernels' codes and scales equal the oracle's bit for bit."""
    H = full_case.shape.hidden
    rng = np.random.default_rng(11)
    table = oracle.e4m3_table()
    mags = np.unique(np.abs(table[np.isfinite(table)]))
    mids = 0.5 * (mags[:-1] + mags[1:])
    rows = 16
    x = np.zeros((rows, H), np.float64)
    for t in range(rows):
        for g in range(H // 128):
            scale = 2.0 ** int(rng.integers(-8, 8))  # amax = 448 * scale: s = scale exactly
            kind = (t + g) % 4
            if kind == 0:
                vals = rng.choice(mids, 128)
            elif kind == 1:
                vals = rng.choice(mags, 128)
            elif kind == 2:
                vals = rng.choice(np.concatenate([mids[:10], mags[:10]]), 128)
            else:
                vals = np.zeros(128) if g % 2 else rng.choice(mids, 128)
            vals = vals * scale * rng.choice([-1.0, 1.0], 128)
            if kind != 3 or g % 2 == 0:
                vals[int(rng.integers(0, 128))] = 448.0 * scale
            x[t, g * 128:(g + 1) * 128] = vals
    xt = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)
    assert np.array_equal(xt.float().numpy().astype(np.float64), x)  # exact in bf16
    codes, scales = full_case.moe.quantize(xt.cuda())
    torch.cuda.synchronize()
    for t in range(rows):
        rc, rs = oracle.quant_row(x[t].astype(np.float32))
        assert np.array_equal(codes[t].cpu().numpy(), rc), t
        assert np.array_equal(scales[t].cpu().numpy(), rs), t


def test_decode_t1(full_case):
    x = full_case.x(1)
    run_and_check(full_case, x)


def test_decode_t1_many_rows_one_by_one(full_case):
    x = full_case.x(8, tag="many")
    for r in range(8):
        run_and_check(full_case, x[r:r + 1].contiguous())


@pytest.mark.parametrize("path", [m.PATH_DECODE_ROWS, m.PATH_DECODE_CHAINED, m.PATH_PROMPT])
def test_decode_t1_other_kernels(full_case, path):
    """One row on the multi-row decode kernel, the chained decode kernels and
    the prompt kernels (the automatic path takes the one-row kernel)."""
    x = full_case.x(3, tag="t1paths")
    try:
        for r in range(3):
            run_and_check(full_case, x[r:r + 1].contiguous(), path=path)
    finally:
        full_case.moe.set_option(m.MOE_OPT_PATH, m.PATH_AUTO)


def test_decode_t1_repeated_launches_bitwise(full_case):
    """Back-to-back one-row forwards (launch tags advance every launch) give
    identical outputs."""
    x = full_case.x(1, tag="rep1")
    ys = [full_case.moe.forward(x).clone() for _ in range(6)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
    assert full_case.moe.device_status() == m.MOE_OK


@pytest.mark.parametrize("rows", [1, 3, 11, 64])
def test_plain_launches_match_chained(full_case, rows):
    """With programmatic dependent launch off (MOE_OPT_PDL = 0) every path
    gives bit-identical outputs to the chained launches, and matches the
    oracle."""
    x = full_case.x(rows, tag=f"pdl{rows}")
    y_on = full_case.moe.forward(x).clone()
    full_case.moe.set_option(m.MOE_OPT_PDL, 0)
    try:
        y_off = full_case.moe.forward(x).clone()
        torch.cuda.synchronize()
        assert torch.equal(y_on, y_off)
        run_and_check(full_case, x, sample_rows=[0, rows - 1])
    finally:
        full_case.moe.set_option(m.MOE_OPT_PDL, 1)


@pytest.fixture(scope="module")
def tie_layer(dev):
    """A full-width layer whose router repeats rows: experts 100 and 200 copy
    expert 3's row, 7 and 250 copy expert 5's, so their logits tie exactly
    on both sides for every input."""
    s = W.FULL
    layer = W.make_layer(s, 4242, device=dev)
    wr = layer["router"]
    for a, b in ((3, 100), (3, 200), (5, 7), (5, 250)):
        wr[b] = wr[a]
    net = m.MoELayer(_shape(s), max_rows=64)
    net.load(layer)
    return layer, net, W.to_numpy_layer(layer)


@pytest.mark.parametrize("rows,path", [(1, m.PATH_AUTO), (1, m.PATH_DECODE_ROWS),
                                       (1, m.PATH_DECODE_CHAINED), (3, m.PATH_AUTO),
                                       (8, m.PATH_AUTO), (8, m.PATH_DECODE_ROWS),
                                       (40, m.PATH_AUTO), (40, m.PATH_PROMPT_MMA)])
def test_exact_ties(tie_layer, rows, path):
    """Exact ties take the lower expert first at every rank, with no near-tie
    slack: rows along router row 3 put the tie group {3, 100, 200} on top,
    rows along rows 5 and 3 put {5, 7, 250} first, and all-zero rows tie all
    256 experts (experts 0..7, equal weights, zero codes with scale 1)."""
    layer, net, host = tie_layer
    wr = layer["router"].float().cpu()
    x = torch.zeros((rows, wr.shape[1]))
    for t in range(rows):
        if t % 3 == 1:
            x[t] = wr[3] * 40.0
        elif t % 3 == 2:
            x[t] = wr[5] * 40.0 + wr[3] * 10.0
    x = x.to(torch.bfloat16).cuda()
    net.set_option(m.MOE_OPT_PATH, path)
    try:
        y = net.forward(x)
        idx, w = net.route(x)
        codes, scales = net.quantize(x)
        torch.cuda.synchronize()
    finally:
        net.set_option(m.MOE_OPT_PATH, m.PATH_AUTO)
    ref = oracle.moe_rows(host, bits(x), trace=True)
    gi = idx.cpu().numpy()
    for t in range(rows):
        if t % 3 == 0:
            assert gi[t].tolist() == list(range(8)), (t, gi[t])
            assert np.allclose(w.cpu().numpy()[t], 0.125, rtol=0, atol=1e-7)
        elif t % 3 == 1:
            assert gi[t][:3].tolist() == [3, 100, 200], (t, gi[t])
        else:
            assert gi[t][:3].tolist() == [5, 7, 250], (t, gi[t])
    near, differ = check_topk(gi, ref.trace["logits"], 8)
    assert not differ.any()
    assert np.array_equal(gi, ref.trace["idx"])
    assert np.array_equal(codes.cpu().numpy(), ref.trace["xq"])
    assert np.array_equal(scales.cpu().numpy(), ref.trace["sx"])
    check_output(bits(y), ref.y_ref)


@pytest.fixture(scope="module")
def t11_case(dev):
    return Case(W.WORKLOADS["decode_t11"], 64, dev)


@pytest.mark.parametrize("path", [m.PATH_AUTO, m.PATH_DECODE_ROWS, m.PATH_PROMPT])
def test_decode_t11(t11_case, path):
    """Eleven rows with overlapping expert sets on the automatic path (the
    chained decode kernels), the role-split multi-row kernel and the grouped
    tcgen05 kernels."""
    x = t11_case.x(11)
    try:
        run_and_check(t11_case, x, path=path)
        idx, _ = t11_case.moe.route(x)
    finally:
        t11_case.moe.set_option(m.MOE_OPT_PATH, m.PATH_AUTO)
    distinct = len(set(idx.cpu().numpy().ravel().tolist()))
    assert distinct < 11 * 8, "rows were meant to share experts"


def test_path_option_range(t11_case):
    assert t11_case.moe.ctx is not None
    assert m.moe_set_option(t11_case.moe.ctx, m.MOE_OPT_PATH, 7) == m.MOE_ERR_INVALID_ARG
    assert m.moe_set_option(t11_case.moe.ctx, m.MOE_OPT_PATH, -1) == m.MOE_ERR_INVALID_ARG
    assert m.moe_set_option(t11_case.moe.ctx, m.MOE_OPT_PATH, 5) == m.MOE_ERR_INVALID_ARG
    assert m.moe_set_option(t11_case.moe.ctx, m.MOE_OPT_PATH, m.PATH_DECODE_ROWS) == m.MOE_OK
    assert m.moe_set_option(t11_case.moe.ctx, m.MOE_OPT_PATH, m.PATH_AUTO) == m.MOE_OK


@pytest.mark.parametrize("rows", [2, 3, 4, 5, 6, 15, 16, 17, 64, 128, 129, 255, 1023])
def test_ragged_rows(full_case, rows):
    """Both sides of every automatic path boundary (1 | 2..4 | 5..), of the
    one-block schedule (up to 128 rows) and of the token tiles."""
    x = full_case.x(rows, tag=f"r{rows}")
    sample = sorted(set([0, rows - 1] + list(range(0, rows, max(1, rows // 6)))))
    run_and_check(full_case, x, sample_rows=sample)


def test_prompt_t1024_sampled(dev):
    wl = W.WORKLOADS["prompt_t1024"]
    case = Case(wl, 1024, dev)
    x = case.x(1024)
    idx, _ = case.moe.route(x)
    counts = np.bincount(idx.cpu().numpy().ravel(), minlength=256)
    assert counts.max() > 100 and (counts == 0).sum() >= 1, counts
    # every one of the 1024 rows against the oracle (over all host cores)
    run_and_check(case, x)
    case.moe.close()


def _rows_covering_every_expert(idx: np.ndarray, n: int) -> list:
    """At least one row for every expert some row selected (the first such
    row), then evenly spaced rows up to n in all."""
    first = {}
    for t, row in enumerate(idx):
        for e in row:
            first.setdefault(int(e), t)
    rows = set(first.values())
    T = idx.shape[0]
    spread = [int(t) for t in np.linspace(0, T - 1, n).astype(int)]
    spread += [int(t) for t in np.random.default_rng(0).permutation(T)]
    for t in spread:
        if len(rows) >= n:
            break
        rows.add(t)
    return sorted(rows)


def test_prompt_t16384_sampled(dev):
    """The compute-bound prompt shape (16384 rows, about 512 rows per expert):
    rows covering every selected expert, plus evenly spaced ones, at least 512
    in all, against the oracle."""
    wl = W.WORKLOADS["prompt_t16384"]
    case = Case(wl, 16384, dev)
    x = case.x(16384)
    idx, _ = case.moe.route(x)
    torch.cuda.synchronize()
    gi = idx.cpu().numpy()
    counts = np.bincount(gi.ravel(), minlength=256)
    assert counts.max() > 1000, counts.max()
    sample = _rows_covering_every_expert(gi, 512)
    assert len(sample) >= 512
    covered = set(gi[sample].ravel().tolist())
    assert covered == set(np.nonzero(counts)[0].tolist())
    run_and_check(case, x, sample_rows=sample)
    case.moe.close()


def test_repeat_bitwise(full_case):
    for rows in (1, 11, 300):
        x = full_case.x(rows, tag=f"rep{rows}")
        ys = [full_case.moe.forward(x).clone() for _ in range(5)]
        torch.cuda.synchronize()
        for y in ys[1:]:
            assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))


@pytest.mark.parametrize("rows", [1, 3, 64])
def test_forward_host_matches_device(full_case, rows):
    """moe_forward_host gives moe_forward's bits: with pinned buffers (the
    same pair with new contents, another pair, after an option change) and
    with pageable ones."""
    net = full_case.moe

    def check(xh, yh, x):
        net.forward_host(xh, yh)
        y_dev = net.forward(x)
        torch.cuda.synchronize()
        assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))

    xh = full_case.x(rows, tag=f"host{rows}").cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    for tag in ("a", "b"):  # the same buffers with new contents
        x = full_case.x(rows, tag=f"host{tag}{rows}")
        xh.copy_(x.cpu())
        check(xh, yh, x)
    xh2, yh2 = xh.clone().pin_memory(), torch.empty_like(xh).pin_memory()
    check(xh2, yh2, x)
    net.set_option(m.MOE_OPT_PDL, 0)
    try:
        check(xh, yh, x)
    finally:
        net.set_option(m.MOE_OPT_PDL, 1)
    check(xh, yh, x)
    xp, yp = x.cpu(), torch.empty((rows, x.shape[1]), dtype=torch.bfloat16)
    assert not xp.is_pinned() and not yp.is_pinned()
    check(xp, yp, x)


# ---- boundary behaviour ------------------------------------------------------

def test_errors(full_case, dev):
    ctx = full_case.moe.ctx
    x = full_case.x(2, tag="err")
    y = torch.empty_like(x)
    assert m.moe_forward(ctx, x, y, 0) == m.MOE_OK
    assert m.moe_forward(ctx, x, y, -1) == m.MOE_ERR_INVALID_ARG
    assert m.moe_forward(ctx, x, y, 1025) == m.MOE_ERR_UNSUPPORTED_SHAPE
    assert m.moe_forward(ctx, x, x, 2) == m.MOE_ERR_INVALID_ARG
    assert m.moe_forward(ctx, None, y, 2) == m.MOE_ERR_INVALID_ARG
    fresh = m.MoELayer(_shape(W.TINY), max_rows=4)
    xt = torch.zeros((1, 256), dtype=torch.bfloat16, device=dev)
    assert m.moe_forward(fresh.ctx, xt, torch.empty_like(xt), 1) == m.MOE_ERR_NOT_LOADED
    cfg = m.moe_config(2048, 256, 8, 512, 512, 128, 1024, 1 << 20)
    rc, h = m.moe_create(cfg, 0)
    assert rc == m.MOE_ERR_ALLOC_LIMIT and not h.value
    for bad in (m.moe_config(2000, 256, 8, 512, 512, 128, 16, 0),
                m.moe_config(2048, 256, 8, 500, 512, 128, 16, 0),
                m.moe_config(2048, 300, 8, 512, 512, 128, 16, 0),
                m.moe_config(2048, 4, 8, 512, 512, 128, 16, 0),
                m.moe_config(2048, 256, 8, 512, 512, 64, 16, 0)):
        rc, h = m.moe_create(bad, 0)
        assert rc == m.MOE_ERR_UNSUPPORTED_SHAPE and not h.value
    assert m.moe_last_device_status(ctx) == m.MOE_OK
    fresh.close()


def test_max_rows(dev):
    case = Case(W.WORKLOADS["tiny_t4"], 1024, dev)
    x = case.x(1024, tag="max")
    run_and_check(case, x, sample_rows=[0, 333, 1023])


# ---- layers in sequence (the 40-layer backbone sweep, shortened) --------------

@pytest.mark.parametrize("rows", [1, 17])
def test_chained_layers_teacher_forced(dev, rows):
    """Rows passed through three distinct layers, x_{l+1} = y_l, each layer on
    its own context with launches chained on one stream; every layer's output
    is checked against the oracle on that layer's GPU input (teacher forced)."""
    wl = W.WORKLOADS["sweep40"]
    s = wl.shape
    layers = [W.make_layer(s, W.layer_seed(wl, l), wl.x_kind, device=dev) for l in range(3)]
    nets = []
    for layer in layers:
        net = m.MoELayer(_shape(s), max_rows=64)
        net.load(layer)
        nets.append(net)
    xs = [W.make_x(s, rows, W.layer_seed(wl, 0), wl.x_kind, device="cuda", tag="chain")]
    for net in nets:
        xs.append(net.forward(xs[-1]))
    routes = [net.route(x) for net, x in zip(nets, xs[:-1])]
    torch.cuda.synchronize()
    sample = sorted({0, rows - 1})
    for l, layer in enumerate(layers):
        host = W.to_numpy_layer(layer)
        ref = oracle.moe_rows(host, bits(xs[l])[sample], trace=True)
        idx = routes[l][0].cpu().numpy()[sample]
        near, differ = check_topk(idx, ref.trace["logits"], s.top_k)
        assert differ.sum() == 0 or (differ & near).all(), f"layer {l} routed differently"
        rel, mx = check_output(bits(xs[l + 1])[sample], ref.y_ref, rows_mask=~differ)
    for net in nets:
        net.close()
