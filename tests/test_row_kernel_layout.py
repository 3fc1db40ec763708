"""The index arithmetic of two kernels restated on the CPU (no GPU needed).

k_quant_scatter (csrc/k_slots.cu): 128 threads per row, thread rt takes the
16 values at 16*rt + 2048*p in pass p.  A 1 x 128 group's amax is reduced by
shuffles within an aligned block of 8 lanes, so each group must sit in one
pass on exactly one such block, and the 16-byte loads and stores need 16-value
alignment.

The block-FP8 GEMMs' scale-product table (csrc/k_prompt_tc.cu): with
n_k % 4 == 0, vector v of the item's token scales is token t = v // (n_k/4),
K blocks 4*kq .. 4*kq+3 with kq = v % (n_k/4); every (token, K block) entry
of the table is written exactly once.
"""
from __future__ import annotations

import numpy as np
import pytest

ROW_THREADS = 128
PER_THREAD = 16
PASS = PER_THREAD * ROW_THREADS
GROUP = 128


def scatter_map(H: int):
    """(value index -> (pass, thread)) as the kernel walks a row."""
    owner = np.full((H, 2), -1, np.int64)
    for rt in range(ROW_THREADS):
        base = PER_THREAD * rt
        p = 0
        while base < H:
            assert base % PER_THREAD == 0  # 16-byte codes, 32-byte bf16 loads
            for i in range(PER_THREAD):
                assert owner[base + i, 0] == -1, "value covered twice"
                owner[base + i] = (p, rt)
            base += PASS
            p += 1
    return owner


@pytest.mark.parametrize("H", [128, 256, 1920, 2048, 2176, 2560, 3072, 4096, 6144, 8192, 65536])
def test_quant_scatter_covers_every_value_once(H):
    owner = scatter_map(H)
    assert (owner[:, 0] >= 0).all(), "a value no thread takes"


@pytest.mark.parametrize("H", [128, 256, 1920, 2048, 2176, 2560, 3072, 4096, 6144, 8192, 65536])
def test_quant_scatter_groups_on_aligned_eight_lanes(H):
    owner = scatter_map(H)
    for g in range(H // GROUP):
        p = owner[g * GROUP:(g + 1) * GROUP, 0]
        rt = owner[g * GROUP:(g + 1) * GROUP, 1]
        assert (p == p[0]).all(), "a group split over passes"
        threads = np.unique(rt)
        assert threads.size == GROUP // PER_THREAD == 8
        lanes = threads % 32
        # one aligned block of 8 lanes in one warp: the shuffle mask
        # 0xFF << (lane & 24) names exactly these lanes
        assert (threads // 32 == threads[0] // 32).all()
        assert lanes.min() % 8 == 0 and lanes.max() == lanes.min() + 7
        mask = 0xFF << (int(lanes[0]) & 24)
        assert all((mask >> int(l)) & 1 for l in lanes)
        # every lane of an active block is active in that pass: a pass
        # starts at 16 * rt, so a group's first lane is a multiple of 8
        assert (g * GROUP - PASS * p[0]) % (8 * PER_THREAD) == 0


@pytest.mark.parametrize("n_k", [4, 8, 16, 20, 32, 96])
@pytest.mark.parametrize("kN", [64, 128])
@pytest.mark.parametrize("threads", [512])
def test_scale_table_vector_map(n_k, kN, threads):
    nq = n_k // 4
    hits = np.zeros((n_k, kN), np.int64)
    reads = []
    for tid in range(threads):
        v = tid
        while v < kN * nq:
            t, kq = divmod(v, nq)
            reads.append(t * n_k + 4 * kq)  # float offset of the float4 read
            for r in range(4):
                hits[4 * kq + r, t] += 1
            v += threads
    assert (hits == 1).all()
    # every float4 read starts on a 16-byte boundary of the token-major rows
    assert all(o % 4 == 0 for o in reads)
    # consecutive threads read consecutive float4s (no bank conflicts)
    first = [tid for tid in range(min(32, kN * nq))]
    offs = [(tid // nq) * n_k + 4 * (tid % nq) for tid in first]
    assert offs == [4 * i for i in range(len(first))]
