"""GPU parity of pa_copy_blocks: device-to-device copies, copy-on-write of a
forked request, and swapping blocks out to pinned host memory and back."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_226_gb300 import build, lib
from paged_kv_cache_226_gb300 import inputs as pin
from parity_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib.load()
    d = torch.device("cuda:0")
    lib.read_device_errors(d)
    return d


@pytest.mark.parametrize("dtype,bs,hkv,d", [("fp16", 16, 8, 128), ("bf16", 32, 2, 64)])
def test_copy_blocks_device_to_device(dev, dtype, bs, hkv, d):
    rng = np.random.default_rng(3)
    kc = pin.normal_tensor(rng, (40, bs, hkv, d), dtype)
    vc = pin.normal_tensor(rng, (40, bs, hkv, d), dtype)
    mapping = np.array([[0, 39], [5, 6], [12, 30], [31, 2], [7, 8], [20, 21]], dtype=np.int64)
    kd, vd = kc.to(dev), vc.to(dev)
    lib.copy_blocks(kd, vd, kd, vd, torch.from_numpy(mapping).to(dev))
    wk, wv, bad = oracle.copy_blocks(pin.bits(kc), pin.bits(vc), pin.bits(kc), pin.bits(vc),
                                     mapping)
    torch.cuda.synchronize(dev)
    assert bad == 0
    assert np.array_equal(pin.bits(kd.cpu()), wk) and np.array_equal(pin.bits(vd.cpu()), wv)
    assert lib.read_device_errors(dev) == 0
    # an id outside the pool is skipped and reported
    bad_map = torch.tensor([[1, 40], [2, 3]], dtype=torch.int64, device=dev)
    lib.copy_blocks(kd, vd, kd, vd, bad_map)
    wk2, wv2, _ = oracle.copy_blocks(wk, wv, wk, wv, np.array([[2, 3]]))
    torch.cuda.synchronize(dev)
    assert np.array_equal(pin.bits(kd.cpu()), wk2)
    assert lib.read_device_errors(dev) == lib.PA_DEVERR_BAD_SLOT


def test_copy_on_write_after_fork(dev):
    """A request forks (parallel sampling); both continue with different
    tokens.  The child's token lands in the shared, half-filled last block, so
    the allocator gives it a private copy first; the parent keeps its block."""
    bs, hkv, d, hq = 16, 2, 128, 8
    rng = np.random.default_rng(9)
    pool = pin.BlockPool(12, bs, order=rng.permutation(12))
    a = pin.PagedKVAllocator(pool)
    a.add_sequence(0)
    a.extend(0, 37)                                    # 3 blocks, last one 5/16 full
    a.fork(0, 1)
    slot_child = a.append_token(1)
    copies = a.take_copies()
    slot_parent = a.append_token(0)
    assert len(copies) == 1 and a.take_copies() == []
    kc = pin.normal_tensor(rng, (12, bs, hkv, d), "fp16")
    vc = pin.normal_tensor(rng, (12, bs, hkv, d), "fp16")
    q = pin.normal_tensor(rng, (2, hq, d), "fp16")
    k_new = pin.normal_tensor(rng, (2, hkv, d), "fp16")
    v_new = pin.normal_tensor(rng, (2, hkv, d), "fp16")
    slots = np.array([slot_parent, slot_child], dtype=np.int64)
    tables = a.table_array([0, 1])
    lens = np.array([38, 38], dtype=np.int32)
    # device: copy the shared block, write both new tokens, attend
    kd, vd = kc.to(dev), vc.to(dev)
    lib.copy_blocks(kd, vd, kd, vd, torch.tensor(copies, dtype=torch.int64, device=dev))
    lib.reshape_and_cache(k_new.to(dev), v_new.to(dev), torch.from_numpy(slots).to(dev), kd, vd)
    out = lib.decode(q.to(dev), kd, vd, torch.from_numpy(tables).to(dev),
                     torch.from_numpy(lens).to(dev), 1 / np.sqrt(d))
    # reference: the same three operations
    wk, wv, _ = oracle.copy_blocks(pin.bits(kc), pin.bits(vc), pin.bits(kc), pin.bits(vc), copies)
    wk, wv, _ = oracle.reshape_and_cache(pin.bits(k_new), pin.bits(v_new), slots, wk, wv, bs)
    want = oracle.paged_decode(pin.bits(q), wk, wv, tables, lens, 1 / np.sqrt(d), "fp16")
    torch.cuda.synchronize(dev)
    assert np.array_equal(pin.bits(kd.cpu()), wk) and np.array_equal(pin.bits(vd.cpu()), wv)
    assert_close(out.float().cpu().numpy(), want, "copy-on-write fork")
    # the two requests share their first two blocks and differ in the third
    assert tables[0, 0] == tables[1, 0] and tables[0, 2] != tables[1, 2]
    assert lib.read_device_errors(dev) == 0


def test_swap_out_to_pinned_host_and_back(dev):
    w = pin.build_workload(params=dict(dtype="bf16", num_seqs=3, lens=[20, 70, 300],
                                       num_q_heads=16, num_kv_heads=4, head_dim=128,
                                       block_size=16), seed=13)
    d = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).to(dev)
         for k, v in dict(q=w.q, kc=w.k_cache, vc=w.v_cache, bt=w.block_tables,
                          cl=w.context_lens).items()}
    before = lib.decode(d["q"], d["kc"], d["vc"], d["bt"], d["cl"], w.scale).clone()
    # rebuild the allocator state of sequence 2 and swap it out
    dev_pool = pin.BlockPool(w.num_blocks, 16)
    used = set(int(x) for b in range(3) for x in w.block_tables[b, :-(-int(w.context_lens[b]) // 16)])
    dev_pool.free_blocks = [x for x in range(w.num_blocks) if x not in used]
    for x in used:
        dev_pool.ref_count[x] = 1
    a = pin.PagedKVAllocator(dev_pool)
    n2 = -(-300 // 16)
    a.page_tables[2] = [int(x) for x in w.block_tables[2, :n2]]
    a.token_counts[2] = 300
    host_pool = pin.BlockPool(32, 16)
    hk = torch.empty((32, 16, 4, 128), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty((32, 16, 4, 128), dtype=torch.bfloat16).pin_memory()
    out_pairs = a.swap_out(2, host_pool)
    lib.copy_blocks(d["kc"], d["vc"], hk, hv, torch.tensor(out_pairs, dtype=torch.int64, device=dev))
    torch.cuda.synchronize(dev)
    assert np.array_equal(pin.bits(hk)[[h for _, h in out_pairs]],
                          pin.bits(w.k_cache)[[p for p, _ in out_pairs]])
    # the freed device blocks get overwritten by someone else
    d["kc"][[p for p, _ in out_pairs]] = 7.0
    d["vc"][[p for p, _ in out_pairs]] = -7.0
    in_pairs = a.swap_in(2)
    lib.copy_blocks(hk, hv, d["kc"], d["vc"], torch.tensor(in_pairs, dtype=torch.int64, device=dev))
    bt = d["bt"].clone()
    bt[2, :n2] = torch.tensor(a.page_tables[2], dtype=torch.int32, device=dev)
    after = lib.decode(d["q"], d["kc"], d["vc"], bt, d["cl"], w.scale)
    torch.cuda.synchronize(dev)
    assert torch.equal(after[2], before[2])
    assert lib.read_device_errors(dev) == 0
