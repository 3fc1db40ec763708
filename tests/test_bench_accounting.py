"""The algorithmic work bench.py divides by, against the closed forms of the
layer (no GPU).

Per touched expert: 2I*H + H*I bytes of e4m3 weights plus fp32 128x128 block
scales.  Per layer: the fp32 router [E, H], the bf16 shared expert
[2Is, H] + [H, Is], the bf16 gate vector [H], and bf16 x and y.  FP8 flops:
2 * T * k * (2I*H + H*I).
"""
from __future__ import annotations

import bench
import workloads as W


def test_one_row_layer_bytes():
    s = W.FULL
    per_expert = 3 * 512 * 2048 + 4 * (8 * 16 + 16 * 4)
    assert per_expert == 3_146_496
    fixed = 4 * 256 * 2048 + 2 * 3 * 512 * 2048 + 2 * 2048
    assert bench.layer_bytes(s, 1, 8) == 8 * per_expert + fixed + 2 * 2 * 2048
    assert bench.layer_bytes(s, 1, 8) == 33_572_864


def test_layer_bytes_grow_with_rows_and_experts():
    s = W.FULL
    base = bench.layer_bytes(s, 11, 29)
    assert bench.layer_bytes(s, 12, 29) - base == 2 * 2 * 2048       # x and y of one row
    assert bench.layer_bytes(s, 11, 30) - base == 3_146_496          # one more expert


def test_fp8_flops():
    s = W.FULL
    assert bench.fp8_flops(s, 1) == 2 * 8 * (2 * 512 * 2048 + 2048 * 512)
    assert bench.fp8_flops(s, 1024) == 1024 * bench.fp8_flops(s, 1)


def test_stage_bytes_cover_every_timed_stage():
    """Every stage name a forward can report has a byte count; the stages
    that only read and write workspace (top-k, schedule) have none."""
    s = W.FULL
    sb = bench.stage_bytes(s, 1024, 173.3)
    for name in ("decode_row", "decode_rows", "route_decode", "gateup_decode",
                 "down_combine_decode", "router_tc", "quant_scatter",
                 "shared_gateup_tc", "gateup_tc", "shared_down_tc", "down_tc", "combine"):
        assert name in sb and sb[name] > 0, name
    assert sb["topk"] == 0 and sb["schedule"] == 0
    # the whole-layer kernels move the layer's bytes
    assert sb["decode_row"] == bench.layer_bytes(s, 1024, 173.3)


def test_expert_gemm_stages_count_weights_only():
    """The routed GEMMs' algorithmic bytes are the touched experts' weights and
    block scales: the gathered codes, the SwiGLU rows and the expert outputs
    they also move are workspace traffic."""
    s = W.FULL
    U = 200
    sb = bench.stage_bytes(s, 1024, U)
    assert sb["gateup_tc"] == U * (2 * 512 * 2048 + 4 * 8 * 16)
    assert sb["down_tc"] == U * (2048 * 512 + 4 * 16 * 4)
    assert sb["shared_down_tc"] == 2 * 2048 * 512
    # weights + layer input bytes + layer output bytes over all stages of the
    # tcgen05 forward = the layer's bytes
    tc = ("router_tc", "quant_scatter", "shared_gateup_tc", "gateup_tc", "shared_down_tc",
          "down_tc", "combine")
    x_reads = 3 * 2 * 1024 * 2048  # router, quantisation and the shared gate/up read x
    assert sum(sb[n] for n in tc) - x_reads + 2 * 1024 * 2048 == bench.layer_bytes(s, 1024, U)


def test_rows_per_second_is_whole_job():
    assert bench.rows_per_second(1, 100, 11, 0.5) == 100 * 11 / 0.5
    assert bench.rows_per_second(4, 100, 11, 0.5) == 4 * 100 * 11 / 0.5


def test_addnorm_bytes():
    """Per row: residual and x read, new residual and normed row written (bf16),
    codes (e4m3) and 16 group scales (fp32); gamma once per launch."""
    H = 2048
    assert bench.addnorm_bytes(H, 1) == 4 * 2 * H + H + 4 * 16 + 2 * H
    assert bench.addnorm_bytes(H, 1024) - bench.addnorm_bytes(H, 1023) == 18_496


def test_threaded_oracle_matches_one_thread():
    """The all-cores oracle leg calls the same C oracle from several threads:
    its outputs equal the single-threaded ones, row by row."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    L = W.to_numpy_layer(W.make_layer(W.TINY, 3))
    xb = W.bf16_bits(W.make_x(W.TINY, 12, 3))
    one = [oracle.moe_rows(L, xb[r:r + 1]).y_bf16 for r in range(12)]
    with ThreadPoolExecutor(max_workers=4) as ex:
        many = list(ex.map(lambda r: oracle.moe_rows(L, xb[r:r + 1]).y_bf16, range(12)))
    for a, b in zip(one, many):
        assert np.array_equal(a, b)
    v, n = bench.cpu_baseline_threads(L, xb, 0.2, 3)
    assert n >= 3 and v > 0


def test_quantiles_interpolate():
    import numpy as np
    vals = sorted(np.random.default_rng(0).random(57).tolist())
    for q in (0.1, 0.5, 0.9):
        assert abs(bench.per_quantile(vals, q) - float(np.quantile(vals, q))) < 1e-12


def test_replay_quantiles_logic(monkeypatch):
    """The per-replay event bookkeeping, with host stand-ins for CUDA events:
    replay i takes (i + 1) ms, so per-step times are (i + 1) / steps."""
    import contextlib

    import torch

    clock = [0.0]

    class FakeEvent:
        def __init__(self, enable_timing=False):
            self.t = None

        def record(self, stream=None):
            self.t = clock[0]

        def elapsed_time(self, other):
            return other.t - self.t

        def synchronize(self):
            pass

    class FakeGraph:
        def __init__(self):
            self.n = 0

        def replay(self):
            self.n += 1
            clock[0] += float(self.n)

    monkeypatch.setattr(torch.cuda, "Event", FakeEvent)
    monkeypatch.setattr(torch.cuda, "stream", lambda s: contextlib.nullcontext())
    q = bench.replay_quantiles(FakeGraph(), None, 4, 11)
    per = [(i + 1) / 4 for i in range(11)]
    assert q["replays"] == 11 and q["steps_per_replay"] == 4
    assert abs(q["median"] - per[5]) < 1e-12
    assert abs(q["p10"] - bench.per_quantile(per, 0.1)) < 1e-12
    assert "unavailable" in bench.replay_quantiles(FakeGraph(), None, 4, 2)
    assert "unavailable" in bench.replay_quantiles(None, None, 4, 50)


def _reference_line(*extra, env_extra=None):
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", *extra], cwd=root,
                       capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    return [json.loads(ln) for ln in lines]


def _check_reference_contract(d):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_layer():
    (d,) = _reference_line("--steps", "1", "--warmup", "0")
    _check_reference_contract(d)
    assert d["metric"] == bench.METRIC and d["config"]["workload"] == "decode_t1"
    assert d["warmup"] == 0


def test_reference_arm_addnorm():
    (d,) = _reference_line("--workload", "addnorm_t1", "--steps", "2", "--cpu-seconds", "0.4")
    _check_reference_contract(d)
    assert d["metric"] == bench.ADDNORM_METRIC


def test_reference_arm_other_ranks_print_nothing():
    assert _reference_line("--steps", "1", env_extra={"RANK": "1", "WORLD_SIZE": "2"}) == []


def test_threaded_oracle_rows_equal_one_call():
    """The parity tests' multi-threaded oracle helper returns exactly what one
    call over all rows returns (outputs and every trace array)."""
    import numpy as np

    import oracle
    from parity import oracle_rows
    L = W.to_numpy_layer(W.make_layer(W.TINY, 5))
    xb = W.bf16_bits(W.make_x(W.TINY, 13, 5))
    one = oracle.moe_rows(L, xb, trace=True)
    many = oracle_rows(L, xb, threads=4, trace=True)
    assert np.array_equal(one.y_bf16, many.y_bf16)
    assert np.array_equal(one.y_ref, many.y_ref)
    for n in one.trace:
        assert np.array_equal(one.trace[n], many.trace[n]), n
