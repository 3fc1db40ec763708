"""Layers wider than the pages' 2048: hidden widths that make the row kernels
take more than one pass over a row (the quantise-scatter's 2048-value passes,
the decode kernels' per-warp slices) and K-block counts of the block-FP8
GEMMs other than 16, every path against the oracle (needs a GB300)."""
from __future__ import annotations

import pytest

import workloads as W
from test_gpu_parity import Case, dev, run_and_check  # noqa: F401  (dev: fixture)

pytestmark = pytest.mark.gpu

m = pytest.importorskip("block_fp8_mixture_router_gb300")


def _wide(hidden: int) -> W.Workload:
    shape = W.MoEShape(hidden=hidden, n_experts=16, top_k=4, inter=256, shared_inter=128)
    return W.Workload(f"wide_h{hidden}", shape, 8, 23 + hidden, "normal", 1,
                      f"H={hidden}, 16 experts top-4, I=256, Is=128")


@pytest.mark.parametrize("hidden", [2560, 4096])
@pytest.mark.parametrize("rows", [1, 3, 40])
def test_wide_layer(dev, hidden, rows):  # noqa: F811
    case = Case(_wide(hidden), 64, dev)
    try:
        run_and_check(case, case.x(rows, tag=f"w{rows}"))
    finally:
        case.moe.close()


@pytest.mark.parametrize("hidden", [2560, 4096])
def test_wide_layer_grouped_path_few_rows(dev, hidden):  # noqa: F811
    """Three rows on the grouped tcgen05 kernels (the automatic path takes the
    decode kernels there)."""
    case = Case(_wide(hidden), 64, dev)
    try:
        run_and_check(case, case.x(3, tag="g3"), path=m.PATH_PROMPT)
    finally:
        case.moe.close()
