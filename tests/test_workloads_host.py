"""Host checks of the seeded input generators the parity tests and the bench
share: the prefix-hit workload's recipe, and the gather of a sequence's keys
out of the paged pool (used to build the contiguous twin of that workload)."""
import math

import numpy as np

import workloads as wl


def test_prefix_workload_recipe():
    pre = wl.config_prefix()
    assert pre.prefix.size == pre.new.size == 16
    assert np.all(pre.prefix % wl.BLOCK_SIZE == 0)
    assert pre.prefix.min() >= 256 and pre.prefix.max() <= 4096
    assert pre.new.min() >= 128 and pre.new.max() <= 1024
    lk = pre.prefix + pre.new
    assert np.array_equal(np.diff(pre.cu_seqlens_k), lk)
    assert np.array_equal(np.diff(pre.cu_seqlens_q), pre.new)
    assert pre.q.shape == (int(pre.new.sum()), pre.shape.hq, 128)
    used = []
    for b, L in enumerate(lk):
        nblk = math.ceil(int(L) / wl.BLOCK_SIZE)
        ids = pre.block_tables[b, :nblk]
        assert np.all(ids >= 0) and np.all(pre.block_tables[b, nblk:] == -1)
        used.extend(ids.tolist())
    assert len(used) == len(set(used)) == pre.pool.num_blocks, "every block used once"
    # the same seed gives the same bits
    again = wl.config_prefix()
    assert np.array_equal(again.q, pre.q) and np.array_equal(again.pool.k, pre.pool.k)


def test_gather_paged_follows_the_block_table():
    g = np.random.default_rng(7)
    bs, hkv, d = wl.BLOCK_SIZE, 2, 128
    lengths = np.array([1, 256, 257, 700])
    nb = int(sum(math.ceil(int(L) / bs) for L in lengths)) + 3
    bt = wl.carve_block_tables(g.permutation(nb).astype(np.int32), lengths)
    pool = wl.make_pool(8, nb, bt[bt >= 0], hkv)
    k, v = wl.gather_paged(pool, bt, lengths)
    assert k.shape == (int(lengths.sum()), hkv, d)
    row = 0
    for b, L in enumerate(lengths):
        for j in range(int(L)):
            blk, off = bt[b, j // bs], j % bs
            assert np.array_equal(k[row], pool.k[blk, off])
            assert np.array_equal(v[row], pool.v[blk, off])
            row += 1
