"""The prompt path's token-to-expert schedule, restated on the host.

The kernels cut the T rows into blocks of 128.  In each block a bitmap per
expert marks the rows that selected it; a (row, rank) pair's rank among its
expert's rows in the block is the number of marked rows before it, and each
block publishes its per-expert counts.  The pair's slot is then
    off[e] + (rows of e in earlier blocks) + rank,
with off[] the exclusive prefix sum of the experts' totals, and each expert's
rows are cut into chunks of at most 16.  The claims: the slots are a
permutation of the T*k pairs, ordered by (expert, row); the chunks tile every
expert's rows exactly and their number stays within the workspace bound
ceil(T*k/16) + E.  This test restates the steps block by block with numpy and
checks those claims on uniform and skewed routings.  The chained decode
path (at most 16 rows) schedules with one row mask per expert instead; its
restatement below is held to the same claims.
"""
import numpy as np
import pytest

ROWS_PER_BLOCK = 128
CHUNK = 16


def schedule(idx: np.ndarray, E: int):
    T, k = idx.shape
    nb = -(-T // ROWS_PER_BLOCK)
    rank = np.zeros(T * k, np.int64)
    blk_cnt = np.zeros((nb, E), np.int64)
    for b in range(nb):
        t0, nt = b * ROWS_PER_BLOCK, min(ROWS_PER_BLOCK, T - b * ROWS_PER_BLOCK)
        marked = np.zeros((E, ROWS_PER_BLOCK), bool)
        for tl in range(nt):
            marked[idx[t0 + tl], tl] = True
        blk_cnt[b] = marked.sum(1)
        for tl in range(nt):
            for j in range(k):
                e = idx[t0 + tl, j]
                rank[(t0 + tl) * k + j] = int(marked[e, :tl].sum())
    tot = blk_cnt.sum(0)
    off = np.concatenate([[0], np.cumsum(tot)])
    chs = -(-tot // CHUNK)
    ch_off = np.concatenate([[0], np.cumsum(chs)])
    slot_of_pair = np.zeros(T * k, np.int64)
    for p in range(T * k):
        t, e = p // k, idx[p // k, p % k]
        pre = blk_cnt[:t // ROWS_PER_BLOCK, e].sum()
        slot_of_pair[p] = off[e] + pre + rank[p]
    chunks = []
    for e in range(E):
        for c in range(chs[e]):
            chunks.append((e, off[e] + c * CHUNK, min(CHUNK, tot[e] - c * CHUNK), ch_off[e] + c))
    return slot_of_pair, off, chunks, int(ch_off[E])


def routing(rng, T, E, k, skew):
    logits = rng.standard_normal((T, E)) + (skew * rng.standard_normal(E))[None, :]
    return np.argsort(-logits, axis=1, kind="stable")[:, :k]


@pytest.mark.parametrize("T", [1, 17, 128, 129, 300, 1024])
@pytest.mark.parametrize("E,k", [(16, 4), (256, 8), (8, 1)])
@pytest.mark.parametrize("skew", [0.0, 3.0])
def test_schedule_claims(T, E, k, skew):
    rng = np.random.default_rng(T * 1000 + E + int(skew))
    idx = routing(rng, T, E, k, skew)
    slot_of_pair, off, chunks, n_chunks = schedule(idx, E)
    P = T * k
    # a permutation of the pairs
    assert np.array_equal(np.sort(slot_of_pair), np.arange(P))
    pair_of_slot = np.empty(P, np.int64)
    pair_of_slot[slot_of_pair] = np.arange(P)
    # ordered by (expert, row)
    experts = idx.reshape(-1)[pair_of_slot]
    rows = pair_of_slot // k
    key = experts * (T + 1) + rows
    assert np.all(np.diff(key) > 0)
    # every expert's slots are [off[e], off[e+1])
    for e in range(E):
        assert np.all(experts[off[e]:off[e + 1]] == e)
    # chunks tile each expert's rows in order, at most 16 rows each
    covered = np.zeros(P, np.int64)
    for i, (e, first, n, pos) in enumerate(chunks):
        assert pos == i and 1 <= n <= CHUNK
        assert off[e] <= first and first + n <= off[e + 1]
        covered[first:first + n] += 1
    assert np.all(covered == 1)
    assert n_chunks == len(chunks) <= -(-P // CHUNK) + E


def decode_schedule(idx: np.ndarray, E: int):
    """The chained decode path's schedule (rows <= 16): one row mask per
    expert, one chunk per selected expert, slots by an exclusive scan of the
    masks' popcounts and, inside an expert, in row order."""
    T, k = idx.shape
    mask = np.zeros(E, np.int64)
    for p in range(T * k):
        mask[idx[p // k, p % k]] |= 1 << (p // k)
    cnt = np.array([bin(int(m)).count("1") for m in mask])
    slot0 = np.concatenate([[0], np.cumsum(cnt)])[:-1]
    used = np.concatenate([[0], np.cumsum(cnt > 0)])[:-1]
    slot_of_pair = np.full(T * k, -1, np.int64)
    chunks = {}
    for e in range(E):
        if cnt[e] == 0:
            continue
        chunks[int(used[e])] = (e, int(slot0[e]), int(cnt[e]))
        for r, t in enumerate(t for t in range(T) if mask[e] >> t & 1):
            j = int(np.nonzero(idx[t] == e)[0][0])
            slot_of_pair[t * k + j] = slot0[e] + r
    return slot_of_pair, chunks, int((cnt > 0).sum())


@pytest.mark.parametrize("T", [1, 2, 6, 11, 16])
@pytest.mark.parametrize("E,k", [(16, 4), (256, 8)])
def test_decode_schedule_claims(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    for skew in (0.0, 3.0):
        idx = routing(rng, T, E, k, skew)
        slot_of_pair, chunks, n_used = decode_schedule(idx, E)
        P = T * k
        assert np.array_equal(np.sort(slot_of_pair), np.arange(P))
        pair_of_slot = np.empty(P, np.int64)
        pair_of_slot[slot_of_pair] = np.arange(P)
        key = idx.reshape(-1)[pair_of_slot] * (T + 1) + pair_of_slot // k
        assert np.all(np.diff(key) > 0)
        assert sorted(chunks) == list(range(n_used))
        covered = np.zeros(P, np.int64)
        for e, first, n in chunks.values():
            assert 1 <= n <= min(T, CHUNK)
            assert np.all(idx.reshape(-1)[pair_of_slot[first:first + n]] == e)
            covered[first:first + n] += 1
        assert np.all(covered == 1)
