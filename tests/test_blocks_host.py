"""Copy-on-write and swap bookkeeping of the host allocator, and the
reference block copy, on the CPU."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_226_gb300 import inputs as pin


def test_oracle_copy_blocks_matches_numpy_assignment():
    rng = np.random.default_rng(0)
    src_k = rng.integers(0, 1 << 16, size=(6, 16, 2, 64), dtype=np.uint16)
    src_v = rng.integers(0, 1 << 16, size=(6, 16, 2, 64), dtype=np.uint16)
    dst_k = rng.integers(0, 1 << 16, size=(9, 16, 2, 64), dtype=np.uint16)
    dst_v = rng.integers(0, 1 << 16, size=(9, 16, 2, 64), dtype=np.uint16)
    mapping = np.array([[0, 8], [5, 2], [3, 3], [7, 1], [1, -1]], dtype=np.int64)
    kd, vd, bad = oracle.copy_blocks(src_k, src_v, dst_k, dst_v, mapping)
    assert bad == 2
    wk, wv = dst_k.copy(), dst_v.copy()
    for s, d in mapping[:3]:
        wk[d], wv[d] = src_k[s], src_v[s]
    assert np.array_equal(kd, wk) and np.array_equal(vd, wv)


def test_fork_shares_then_copies_on_write():
    pool = pin.BlockPool(8, 4, order=list(range(8))[::-1])     # pops 0, 1, 2, ...
    a = pin.PagedKVAllocator(pool)
    a.add_sequence(0)
    slots = [a.append_token(0) for _ in range(6)]               # blocks 0, 1; block 1 half full
    assert slots == [0, 1, 2, 3, 4, 5] and a.page_tables[0] == [0, 1]
    a.fork(0, 1)
    assert pool.ref_count[0] == 2 and pool.ref_count[1] == 2
    s_child = a.append_token(1)                                 # writes into shared block 1
    assert a.take_copies() == [(1, 2)]
    assert a.page_tables[1] == [0, 2] and s_child == 2 * 4 + 2
    assert pool.ref_count[1] == 1 and pool.ref_count[2] == 1 and pool.ref_count[0] == 2
    s_parent = a.append_token(0)                                # block 1 is the parent's alone now
    assert a.take_copies() == [] and s_parent == 1 * 4 + 2
    a.free_sequence(1)
    assert pool.ref_count[0] == 1 and pool.ref_count[2] == 0


def test_fork_at_a_block_boundary_needs_no_copy():
    pool = pin.BlockPool(8, 4)
    a = pin.PagedKVAllocator(pool)
    a.add_sequence(0)
    a.extend(0, 8)                                              # two full blocks
    a.fork(0, 1)
    a.append_token(1)
    assert a.take_copies() == []
    assert a.page_tables[1][:2] == a.page_tables[0] and len(a.page_tables[1]) == 3


def test_swap_out_and_in_round_trip():
    dev_pool = pin.BlockPool(6, 16)
    host_pool = pin.BlockPool(4, 16)
    a = pin.PagedKVAllocator(dev_pool)
    a.add_sequence(7)
    a.extend(7, 40)                                             # 3 blocks
    before = list(a.page_tables[7])
    out_pairs = a.swap_out(7, host_pool)
    assert [p for p, _ in out_pairs] == before
    assert dev_pool.num_free == 6 and host_pool.num_free == 1
    in_pairs = a.swap_in(7)
    assert [h for h, _ in in_pairs] == [h for _, h in out_pairs]
    assert a.page_tables[7] == [p for _, p in in_pairs]
    assert host_pool.num_free == 4 and dev_pool.num_free == 3
    a.fork(7, 8)
    with pytest.raises(ValueError):
        a.swap_out(7, host_pool)
