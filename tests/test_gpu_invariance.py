"""Batch-invariant rows (needs a GB300): with MOE_OPT_BATCH_INVARIANT a row's
output is bit-identical whatever rows share its forward.

The pages disagree on whether their path has this property: PR #920 ("drama:
Drama 3 (fishaudio/drama-3) text-to-speech on CUDA", section "Receipt")
reports backbone outputs hash-identical at chunk sizes 1, 7 and 128, and
PR #939 ("drama3: Fish Audio Drama 3 text to speech on one CUDA GPU", section
"Determinism and request state") reports that prompt chunk seams fail.  Here
it is an option: every row count runs on the grouped tcgen05 kernels with a
fixed router K split, so each output element is computed by the same
sequence of operations at every row count and position.
"""
from __future__ import annotations

import numpy as np
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


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name", ["decode_t1", "prompt_t1024"])
def test_row_identical_across_batch_sizes(dev, name):
    case = Case(W.WORKLOADS[name], 1024, dev)
    case.moe.set_option(m.MOE_OPT_BATCH_INVARIANT, 1)
    x = case.x(1024, tag="inv")
    y_all = case.moe.forward(x).clone()
    for T in (1, 7, 11, 64, 128, 255):
        y = case.moe.forward(x[:T].contiguous())
        torch.cuda.synchronize()
        assert _same(y, y_all[:T]), T
    # the same rows in another order, and a row alone at other positions
    perm = torch.from_numpy(np.random.default_rng(7).permutation(64)).cuda()
    y = case.moe.forward(x[:64][perm].contiguous())
    torch.cuda.synchronize()
    assert _same(y, y_all[:64][perm])
    for r in (5, 500, 1023):
        y = case.moe.forward(x[r:r + 1].contiguous())
        torch.cuda.synchronize()
        assert _same(y, y_all[r:r + 1]), r
    # and the mode computes the layer: oracle parity on a few row counts
    for T in (1, 11):
        run_and_check(case, x[:T].contiguous())
    case.moe.close()


def test_invariant_option_range(dev):
    case = Case(W.WORKLOADS["tiny_t4"], 16, dev)
    assert m.moe_set_option(case.moe.ctx, m.MOE_OPT_BATCH_INVARIANT, 2) == m.MOE_ERR_INVALID_ARG
    assert m.moe_set_option(case.moe.ctx, m.MOE_OPT_BATCH_INVARIANT, 1) == m.MOE_OK
    assert m.moe_set_option(case.moe.ctx, m.MOE_OPT_BATCH_INVARIANT, 0) == m.MOE_OK
    case.moe.close()
