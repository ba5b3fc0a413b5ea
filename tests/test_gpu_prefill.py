"""GPU parity of pa_prefill (chunked-prefill attention over the paged cache):
the chunk's K/V written with pa_reshape_and_cache, then causal attention of
every new token against the fp64 reference, |gpu - ref| <= 2e-3 + 1e-2 |ref|.
Both kernels are checked: the tcgen05 one (head_dim 128, groups 1/2/4/8,
what pa_prefill takes there), with its work ordered longest first
(pa_prefill_ws, "auto") or last chunk first (pa_prefill, "unscheduled"), and
the mma.sync one (pa_prefill_mma)."""
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


def _run(d, w, max_q, kernel):
    if kernel == "unscheduled":
        return lib.prefill(d["q"], d["kc"], d["vc"], d["bt"], d["cl"], d["qs"], w.scale, max_q,
                           schedule=False)
    return lib.prefill(d["q"], d["kc"], d["vc"], d["bt"], d["cl"], d["qs"], w.scale, max_q,
                       kernel=kernel)


def _check_prefill(w, dev, kernel="auto"):
    d = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).to(dev)
         for k, v in dict(q=w.q, kn=w.k_new, vn=w.v_new, kc=w.k_cache, vc=w.v_cache,
                          bt=w.block_tables, cl=w.context_lens, qs=w.query_start,
                          sm=w.slot_mapping).items()}
    lib.reshape_and_cache(d["kn"], d["vn"], d["sm"], d["kc"], d["vc"])
    max_q = int(np.diff(w.query_start).max()) if w.num_seqs else 0
    out = _run(d, w, max_q, kernel)
    kc, vc, _ = oracle.reshape_and_cache(pin.bits(w.k_new), pin.bits(w.v_new), w.slot_mapping,
                                         pin.bits(w.k_cache), pin.bits(w.v_cache), w.block_size)
    want = oracle.paged_prefill(pin.bits(w.q), kc, vc, w.block_tables, w.context_lens,
                                w.query_start, w.scale, w.dtype)
    torch.cuda.synchronize(dev)
    assert np.array_equal(pin.bits(d["kc"].cpu()), kc)
    err = assert_close(out.float().cpu().numpy(), want, f"{w.name} prefill ({kernel})")
    assert lib.read_device_errors(dev) == 0
    return err


@pytest.mark.parametrize("kernel", ["auto", "unscheduled", "mma"])
@pytest.mark.parametrize("name", ["prefill_tiny", "prefill8b"])
def test_named_prefill(dev, name, kernel):
    _check_prefill(pin.build_prefill_workload(name), dev, kernel)


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [
    ("fp16", 8, 2, 64, 16), ("bf16", 32, 8, 128, 16), ("fp16", 64, 8, 128, 32),
    ("bf16", 4, 4, 128, 16), ("fp16", 16, 8, 64, 32), ("bf16", 12, 2, 128, 16),
    ("fp16", 16, 8, 128, 16)])
@pytest.mark.parametrize("kernel", ["auto", "unscheduled", "mma"])
def test_prefill_shapes_and_ragged_chunks(dev, dtype, hq, hkv, d, bs, kernel):
    lens = [1, 15, 16, 17, 33, 100, 257, 700, 40]
    chunks = [1, 15, 1, 17, 16, 37, 257, 300, 0]
    w = pin.build_prefill_workload(params=dict(dtype=dtype, lens=lens, chunks=chunks,
                                               num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                               block_size=bs), seed=hq + d + bs)
    _check_prefill(w, dev, kernel)


def test_one_token_chunks_equal_decode(dev):
    w = pin.build_prefill_workload(params=dict(dtype="bf16", lens=[3, 90, 513, 1000],
                                               chunks=[1, 1, 1, 1], num_q_heads=32,
                                               num_kv_heads=8, head_dim=128, block_size=16),
                                   seed=2)
    d = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).to(dev)
         for k, v in dict(q=w.q, kc=w.k_cache, vc=w.v_cache, bt=w.block_tables,
                          cl=w.context_lens, qs=w.query_start).items()}
    pre = lib.prefill(d["q"], d["kc"], d["vc"], d["bt"], d["cl"], d["qs"], w.scale, 1)
    dec = lib.decode(d["q"], d["kc"], d["vc"], d["bt"], d["cl"], w.scale)
    assert_close(pre.float().cpu().numpy(), dec.float().cpu().numpy(), "prefill(1) vs decode",
                 atol=1e-3, rtol=5e-3)


def test_prefill_long_chunks_many_tiles(dev):
    """Chunks past 128 tokens and contexts of many 128-key tiles, with a
    sequence whose chunk is its whole context (plain prefill)."""
    w = pin.build_prefill_workload(params=dict(dtype="bf16", lens=[3000, 777, 1024, 129],
                                               chunks=[700, 777, 1, 129], num_q_heads=32,
                                               num_kv_heads=8, head_dim=128, block_size=32),
                                   seed=41)
    _check_prefill(w, dev)
    _check_prefill(w, dev, "mma")


@pytest.mark.parametrize("kernel", ["auto", "mma"])
@pytest.mark.parametrize("dtype,bs", [("bf16", 16), ("fp16", 32)])
def test_prefill_stale_nan_outside_the_contexts(dev, dtype, bs, kernel):
    """Slots past each context's end (inside its last block) and every block no
    table reaches hold NaN bits; neither kernel may let them into the result."""
    w = pin.build_prefill_workload(params=dict(dtype=dtype, lens=[5, 130, 300, 1000],
                                               chunks=[5, 130, 44, 300], num_q_heads=32,
                                               num_kv_heads=8, head_dim=128, block_size=bs),
                                   seed=53)
    nan = 0x7fc0 if dtype == "bf16" else 0x7e00
    kc, vc = pin.bits(w.k_cache).copy(), pin.bits(w.v_cache).copy()
    used = set()
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        nblk = -(-L // bs)
        used.update(int(x) for x in w.block_tables[b, :nblk])
        last = w.block_tables[b, nblk - 1]
        off = (L - 1) % bs + 1
        kc[last, off:] = nan
        vc[last, off:] = nan
    for blk in range(w.num_blocks):
        if blk not in used:
            kc[blk] = nan
            vc[blk] = nan
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    w.k_cache = torch.from_numpy(kc.view(np.int16)).view(tdt)
    w.v_cache = torch.from_numpy(vc.view(np.int16)).view(tdt)
    _check_prefill(w, dev, kernel)


def test_prefill_work_order_is_bitwise_irrelevant(dev):
    """Each (sequence, chunk, KV head) is computed by one CTA alone: the
    longest-first order and the last-chunk-first order give the same bits.
    The ragged batch has chunks of 1 to 900 tokens on contexts of 1 to 4100."""
    w = pin.build_prefill_workload(params=dict(dtype="bf16", lens=[4100, 1, 900, 2000, 77, 3000],
                                               chunks=[300, 1, 900, 33, 77, 1],
                                               num_q_heads=32, num_kv_heads=8, head_dim=128,
                                               block_size=16), seed=61)
    d = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).to(dev)
         for k, v in dict(q=w.q, kc=w.k_cache, vc=w.v_cache, bt=w.block_tables,
                          cl=w.context_lens, qs=w.query_start).items()}
    max_q = int(np.diff(w.query_start).max())
    a = _run(d, w, max_q, "auto")
    b = _run(d, w, max_q, "unscheduled")
    torch.cuda.synchronize(dev)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert lib.read_device_errors(dev) == 0


def test_prefill_workspace_size_and_errors(dev):
    w = pin.build_prefill_workload("prefill8b")
    d = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).to(dev)
         for k, v in dict(q=w.q, kc=w.k_cache, vc=w.v_cache, bt=w.block_tables,
                          cl=w.context_lens, qs=w.query_start).items()}
    max_q = int(np.diff(w.query_start).max())
    shp = lib.make_shape(w.num_seqs, d["q"].shape[1], d["kc"], d["bt"].shape[1])
    n = lib.prefill_workspace_size(shp, max_q)
    # 512-token chunks, 32 tokens (x 4 heads) per CTA: 16 chunks per sequence
    assert n == 256 * -(-4 * w.num_seqs * 16 // 256)
    small = torch.empty(16, dtype=torch.uint8, device=dev)
    with pytest.raises(lib.PaError, match="invalid"):
        lib.prefill(d["q"], d["kc"], d["vc"], d["bt"], d["cl"], d["qs"], w.scale, max_q,
                    workspace=small)
    # head_dim 64 takes the mma.sync kernel: no workspace needed
    q64 = torch.zeros((4, 8, 64), dtype=torch.float16, device=dev)
    kc64 = torch.zeros((4, 16, 2, 64), dtype=torch.float16, device=dev)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    assert lib.prefill_workspace_size(lib.make_shape(1, 8, kc64, 1), 4) == 0
    assert lib.read_device_errors(dev) == 0


def test_prefill_work_order_is_a_longest_first_permutation(dev):
    """The plan kernel's order (left in the workspace, int32 per item b * chunks
    + chunk) holds every (sequence, chunk) item that has query tokens exactly
    once, by non-increasing count of 128-key tiles, then -1 for the rest."""
    lens = [4100, 1, 900, 2000, 77, 3000, 129, 640]
    chunks = [300, 1, 900, 33, 77, 1, 129, 0]
    w = pin.build_prefill_workload(params=dict(dtype="bf16", lens=lens, chunks=chunks,
                                               num_q_heads=32, num_kv_heads=8, head_dim=128,
                                               block_size=16), seed=67)
    d = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).to(dev)
         for k, v in dict(q=w.q, kc=w.k_cache, vc=w.v_cache, bt=w.block_tables,
                          cl=w.context_lens, qs=w.query_start).items()}
    max_q = int(np.diff(w.query_start).max())
    shp = lib.make_shape(w.num_seqs, 32, d["kc"], d["bt"].shape[1])
    ws = torch.full((lib.prefill_workspace_size(shp, max_q),), 0x55, dtype=torch.uint8, device=dev)
    lib.prefill(d["q"], d["kc"], d["vc"], d["bt"], d["cl"], d["qs"], w.scale, max_q, workspace=ws)
    torch.cuda.synchronize(dev)
    qt = 128 // 4                                   # query tokens per item at G = 4
    n_chunks = -(-max_q // qt)
    n = w.num_seqs * n_chunks
    order = ws.view(torch.int32)[:n].cpu().numpy()
    tiles = {}
    for b in range(w.num_seqs):
        L, C = lens[b], chunks[b]
        for c in range(n_chunks):
            t0 = c * qt
            if t0 < C:
                rows = min(qt, C - t0)
                tiles[b * n_chunks + c] = (L - C + t0 + rows - 1) // 128 + 1
    valid = order[order >= 0]
    assert sorted(valid.tolist()) == sorted(tiles)
    assert (order[len(valid):] == -1).all()
    counts = [tiles[i] for i in valid]
    assert all(a >= b for a, b in zip(counts, counts[1:]))
    assert lib.read_device_errors(dev) == 0
