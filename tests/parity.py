"""Comparison rules between the CUDA path and the oracle (test infrastructure).

Bars, from the layer's specification:
  - top-k indices: bit-exact, ordered, for every row whose fp32 logit margins
    at each rank boundary up to the (k+1)-th exceed tau = 2^-10 * max|logit|.
    Near-ties (the pages report 8th/9th experts 6e-5 apart and exactly tied)
    may reorder only within their tie group; such rows are counted and left
    out of the output comparison;
  - activation codes and scales: bit-exact;
  - y: relative L2 <= 5e-3 and max-abs <= 1e-2 * max|y_ref| against the
    oracle's double-precision output.
"""
from __future__ import annotations

import numpy as np
import torch

REL_L2_TOL = 5e-3
MAX_ABS_FRAC = 1e-2
TAU_FRAC = 2.0 ** -10


def tie_groups(lf_row: np.ndarray, k: int):
    """Oracle order of one row and the tie-group id of each position < k+1."""
    E = lf_row.size
    order = sorted(range(E), key=lambda e: (-lf_row[e], e))
    tau = TAU_FRAC * float(np.max(np.abs(lf_row)))
    group = [0] * min(E, k + 1)
    for r in range(1, len(group)):
        gap = float(lf_row[order[r - 1]]) - float(lf_row[order[r]])
        group[r] = group[r - 1] + (0 if gap <= tau else 1)
    return order, group


def check_topk(gpu_idx: np.ndarray, oracle_logits: np.ndarray, k: int):
    """Asserts the rule; returns (near_tie_rows, differing_rows) masks.

    near_tie_rows: rows with a tie group at some rank boundary up to k+1.
    differing_rows: near-tie rows whose GPU order differs from the oracle's
    (allowed only inside tie groups); the output check leaves them out."""
    T = gpu_idx.shape[0]
    near = np.zeros(T, bool)
    differ = np.zeros(T, bool)
    lf = oracle_logits.astype(np.float32)
    for t in range(T):
        order, group = tie_groups(lf[t], k)
        has_tie = any(group[r] == group[r - 1] for r in range(1, len(group)))
        got = [int(v) for v in gpu_idx[t]]
        if not has_tie:
            assert got == order[:k], (t, got, order[:k])
            continue
        near[t] = True
        members = {}
        for r, gid in enumerate(group):
            members.setdefault(gid, set()).add(order[r])
        for r in range(k):
            assert got[r] in members[group[r]], (t, r)
        assert len(set(got)) == k
        differ[t] = got != order[:k]
    return near, differ


def check_output(y_gpu_bits: np.ndarray, y_ref: np.ndarray, rows_mask=None):
    y = torch.from_numpy(y_gpu_bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    if rows_mask is not None:
        y, y_ref = y[rows_mask], y_ref[rows_mask]
    err = y - y_ref
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-300))
    mx = float(np.max(np.abs(err))) if err.size else 0.0
    ref_max = float(np.max(np.abs(y_ref))) if y_ref.size else 0.0
    assert np.all(np.isfinite(y)), "non-finite GPU output"
    assert rel <= REL_L2_TOL, f"relative L2 {rel:.3e} > {REL_L2_TOL}"
    assert mx <= MAX_ABS_FRAC * ref_max, f"max abs {mx:.3e} > {MAX_ABS_FRAC} * {ref_max:.3e}"
    return rel, mx / max(ref_max, 1e-300)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bits (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ---- the oracle over several host threads ------------------------------------

def oracle_rows(host: dict, xb: np.ndarray, threads: int | None = None, **kw):
    """oracle.moe_rows on the rows of xb, split over host threads (the oracle
    is C behind ctypes, which releases the GIL during each call; its only
    mutable state is a table built before the threads start).  Returns one
    OracleResult whose arrays are the per-chunk results concatenated in row
    order, exactly as one call over all rows would give them."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    T = xb.shape[0]
    if threads is None:
        try:
            threads = len(os.sched_getaffinity(0))
        except (AttributeError, OSError):
            threads = os.cpu_count() or 1
    threads = max(1, min(threads, T))
    if threads == 1:
        return oracle.moe_rows(host, xb, **kw)
    oracle.moe_rows(host, xb[:1], **kw)  # builds the e4m3 table before the threads start
    bounds = np.linspace(0, T, threads + 1).astype(int)
    parts = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        res = list(ex.map(lambda ab: oracle.moe_rows(host, xb[ab[0]:ab[1]], **kw), parts))
    trace = None
    if res[0].trace is not None:
        trace = {n: np.concatenate([r.trace[n] for r in res], axis=0) for n in res[0].trace}
    return oracle.OracleResult(np.concatenate([r.y_bf16 for r in res], axis=0),
                               np.concatenate([r.y_ref for r in res], axis=0), trace)


# ---- FP8 codes read back from the forward ------------------------------------

def check_forward_codes(codes: np.ndarray, scales: np.ndarray, ref_xq: np.ndarray,
                        ref_sx: np.ndarray):
    """The codes and group scales every (row, rank) pair's expert read in the
    forward ([T, k, H] and [T, k, H/128]) equal the oracle's quantisation of
    the row, bit for bit, for every rank's copy."""
    T, k, H = codes.shape
    assert ref_xq.shape == (T, H) and ref_sx.shape == (T, scales.shape[2])
    for j in range(k):
        bad = np.nonzero(np.any(codes[:, j] != ref_xq, axis=1))[0]
        assert bad.size == 0, f"rank {j}: codes differ in rows {bad[:8].tolist()}"
        bad = np.nonzero(np.any(scales[:, j].view(np.uint32) != ref_sx.view(np.uint32), axis=1))[0]
        assert bad.size == 0, f"rank {j}: scales differ in rows {bad[:8].tolist()}"


def e4m3_steps(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in e4m3 code steps between two code arrays (the codes are
    sign-magnitude and the magnitude field is monotonic in the value)."""
    def ordered(c):
        c = c.astype(np.int32)
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def hq_agreement(hq: np.ndarray, sh: np.ndarray, ref_hq: np.ndarray, ref_sh: np.ndarray,
                 rows_mask=None):
    """Agreement of the re-quantised SwiGLU rows with the oracle's: (fraction of
    identical codes, largest code-step distance in groups whose scale agrees
    bit for bit, fraction of groups whose scale agrees).  These codes depend
    on the fp32 accumulation order of the gate/up sums, so they are reported
    and held to a bar, not bit-exact."""
    if rows_mask is not None:
        hq, sh, ref_hq, ref_sh = hq[rows_mask], sh[rows_mask], ref_hq[rows_mask], ref_sh[rows_mask]
    if hq.size == 0:
        return 1.0, 0, 1.0
    same = float(np.mean(hq == ref_hq))
    G = hq.shape[-1] // sh.shape[-1]
    s_ok = sh.view(np.uint32) == ref_sh.view(np.uint32)
    steps = e4m3_steps(hq, ref_hq).reshape(*sh.shape, G)
    max_step = int(steps[s_ok].max()) if s_ok.any() else 0
    return same, max_step, float(np.mean(s_ok))


# ---- the bf16-logit router variant ---------------------------------------------

def _bf16_round(v32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(v32, np.float32)).to(torch.bfloat16) \
        .float().numpy()


def bf16_route_alternatives(logits64: np.ndarray, rel_eps: float = 2.0 ** -14):
    """The bf16 values the variant routes on, from the oracle's double logits
    of one row ([E]): (b, alt) where b is the fp32-rounded logit rounded to
    bf16 and alt[e] is the other bf16 neighbour when the fp32 logit lies
    within rel_eps (relative) of the bf16 rounding midpoint between them,
    else NaN.  The GPU sums the fp32 logit in another order, so an expert
    whose fp32 logit sits that close to a midpoint may round either way."""
    l32 = logits64.astype(np.float32)
    b = _bf16_round(l32)
    # the two bf16 neighbours around l32 and the midpoint between them
    up = _bf16_round(np.nextafter(b, np.float32(np.inf)) + np.abs(b) * 2.0 ** -8)
    dn = _bf16_round(np.nextafter(b, np.float32(-np.inf)) - np.abs(b) * 2.0 ** -8)
    other = np.where(l32 >= b, up, dn)
    mid = 0.5 * (b.astype(np.float64) + other.astype(np.float64))
    near = np.abs(l32.astype(np.float64) - mid) <= rel_eps * np.abs(l32.astype(np.float64))
    alt = np.where(near & (other != b), other, np.nan).astype(np.float32)
    return b, alt


def _order(vals: np.ndarray, k: int):
    return [int(e) for e in np.lexsort((np.arange(vals.size), -vals.astype(np.float64)))[:k]]


def check_topk_bf16(gpu_idx: np.ndarray, logits64: np.ndarray, k: int, max_alts: int = 8):
    """The bf16-logit variant's ordered top-k, bit-exact (ties to the lower
    expert) for every row whose decisive experts all round unambiguously to
    bf16; a row with ambiguous experts must equal the order under one of the
    roundings those experts allow.  Returns (ambiguous_rows, differing_rows)."""
    T = gpu_idx.shape[0]
    amb = np.zeros(T, bool)
    differ = np.zeros(T, bool)
    for t in range(T):
        b, alt = bf16_route_alternatives(logits64[t])
        ref = _order(b, k)
        got = [int(v) for v in gpu_idx[t]]
        # experts that can matter: any whose value, either way, reaches the
        # (k+1)-th largest value
        lo = np.sort(np.fmin(b, np.where(np.isnan(alt), b, alt)))[::-1][k]
        cand = [e for e in np.nonzero(~np.isnan(alt))[0] if max(b[e], alt[e]) >= lo]
        if not cand:
            assert got == ref, (t, got, ref)
            continue
        amb[t] = True
        assert len(cand) <= max_alts, (t, len(cand))
        ok = False
        for mask in range(1 << len(cand)):
            v = b.copy()
            for i, e in enumerate(cand):
                if mask >> i & 1:
                    v[e] = alt[e]
            if _order(v, k) == got:
                ok = True
                break
        assert ok, (t, got, ref, cand)
        differ[t] = got != ref
    return amb, differ
