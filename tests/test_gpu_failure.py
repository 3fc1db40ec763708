"""Failure and wrap-around paths of the role-split decode kernels, made to run
without faulting anything (needs a GB300).

- A poll of another CTA's exchange word that gives up: a checking option
  lowers the poll limit, so a normal one-row forward's polls give up.  The
  forward must finish, moe_last_device_status must report
  MOE_ERR_DEVICE_TIMEOUT (and restart the counters), and the next forward at
  the normal limit must match the oracle.  Only polls give up early: the
  kernel's waits for its own copies keep the built-in limit, so no copy is
  left in flight.  Every index the one-row kernel takes from a polled value
  comes out of its top-k over the expert range, so garbage values stay in
  bounds.
- The launch tag's wrap-around: the epoch is set just below the wrap, and
  forwards on both role-split kernels run across it; every output must equal
  the same forward's output away from the wrap, bit for bit.
"""
from __future__ import annotations

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

m = pytest.importorskip("block_fp8_mixture_router_gb300")

from test_gpu_parity import Case, run_and_check  # noqa: E402


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.load_library()
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def case(dev):
    c = Case(W.WORKLOADS["decode_t1"], 16, dev)
    yield c
    c.moe.close()


def test_poll_limit_option_range(case):
    ctx = case.moe.ctx
    assert m.moe_set_option(ctx, m.MOE_OPT_POLL_LIMIT, -1) == m.MOE_ERR_INVALID_ARG
    assert m.moe_set_option(ctx, m.MOE_OPT_LAUNCH_EPOCH, -1) == m.MOE_ERR_INVALID_ARG
    assert m.moe_set_option(ctx, m.MOE_OPT_LAUNCH_EPOCH, m.TAG_CLEAR) == m.MOE_ERR_INVALID_ARG
    assert m.moe_set_option(ctx, m.MOE_OPT_POLL_LIMIT, 0) == m.MOE_OK


def test_forced_poll_timeout_reports_and_recovers(case):
    x = case.x(1, tag="timeout")
    assert case.moe.device_status() == m.MOE_OK
    case.moe.set_option(m.MOE_OPT_POLL_LIMIT, 1)
    try:
        case.moe.forward(x)
        torch.cuda.synchronize()
        assert case.moe.device_status() == m.MOE_ERR_DEVICE_TIMEOUT
        # the flag was read and cleared; the counters start afresh
        assert case.moe.device_status() == m.MOE_OK
    finally:
        case.moe.set_option(m.MOE_OPT_POLL_LIMIT, 0)
    run_and_check(case, x)
    assert case.moe.device_status() == m.MOE_OK


def test_launch_tags_across_the_wrap(case):
    xs = {1: case.x(1, tag="wrap1"), 3: case.x(3, tag="wrap3"), 4: case.x(4, tag="wrap4")}
    ref = {T: case.moe.forward(x).clone() for T, x in xs.items()}
    torch.cuda.synchronize()
    case.moe.set_option(m.MOE_OPT_LAUNCH_EPOCH, m.TAG_CLEAR - 3)
    # tags C-2, C-1, C (clears the words; epoch back to 0), then 1, 2, 3, ...
    order = [1, 3, 4, 3, 1, 4, 1, 3]
    outs = [(T, case.moe.forward(xs[T]).clone()) for T in order]
    torch.cuda.synchronize()
    for i, (T, y) in enumerate(outs):
        assert torch.equal(y.view(torch.int16), ref[T].view(torch.int16)), (i, T)
    assert case.moe.device_status() == m.MOE_OK
    run_and_check(case, xs[3])
