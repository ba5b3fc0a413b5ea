"""GPU parity: the CUDA path through the C ABI against the CPU reference on
the same seeded inputs.  Cache writes bit-exact; attention within
|gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_226_gb300 import build, lib
from paged_kv_cache_226_gb300 import inputs as pin
from parity_util import assert_close, check_workload, to_device

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


# ---------------------------------------------------------------------------
# the named workloads at full size, both decode paths
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "llama8b", "prefix", "llama70b", "long16", "long32"])
def test_named_workload(dev, name):
    w = pin.build_workload(name)
    errs = check_workload(w, dev)
    print(name, errs)


@pytest.mark.parametrize("name", ["llama8b", "prefix", "llama70b", "long16", "long32"])
def test_fused_step_at_the_benchmarked_partition(dev, name):
    """The fused step in the launch configuration the benchmark times: the
    partition size lib.choose_partition picks from the batch's lengths
    (1024, 1024, 2048, 4096 and 4096 tokens on a 152-SM part)."""
    w = pin.build_workload(name)
    P = lib.choose_partition(w.num_seqs, w.num_kv_heads, int(w.context_lens.max()),
                             w.block_size, dev, w.context_lens)
    errs = check_workload(w, dev, modes=("fused",), partition_size=P)
    print(name, P, errs)


# ---------------------------------------------------------------------------
# ragged edges: lengths around tile, block and partition boundaries
# ---------------------------------------------------------------------------

EDGE_LENS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 511, 512, 513, 1024,
             1100]


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [
    ("fp16", 8, 2, 64, 16), ("bf16", 8, 2, 64, 32), ("fp16", 32, 8, 128, 16),
    ("bf16", 64, 8, 128, 32), ("fp16", 4, 4, 128, 16), ("bf16", 2, 1, 64, 16),
    ("fp16", 16, 8, 128, 32), ("bf16", 24, 4, 128, 16)])
def test_edge_lengths(dev, dtype, hq, hkv, d, bs):
    w = pin.build_workload(params=dict(dtype=dtype, num_seqs=len(EDGE_LENS), lens=EDGE_LENS,
                                       num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                       block_size=bs), seed=hq * 7 + d + bs)
    for P in sorted({bs, 2 * bs, 64 if 64 % bs == 0 else bs, 512}):
        check_workload(w, dev, modes=("split", "fused"), partition_size=P)
    check_workload(w, dev, modes=("single", "balanced"))


def test_single_partition_split_matches_single_pass(dev):
    w = pin.build_workload(params=dict(dtype="fp16", num_seqs=6, lens=[5, 16, 100, 300, 400, 512],
                                       num_q_heads=16, num_kv_heads=4, head_dim=128,
                                       block_size=16), seed=11)
    d = to_device(w, dev)
    single = lib.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                        w.scale)
    split = lib.paged_attention(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                d["context_lens"], w.scale, 512, mode="split")
    assert_close(split.float().cpu().numpy(), single.float().cpu().numpy(),
                 "split(1 partition) vs single", atol=1e-3, rtol=5e-3)


# ---------------------------------------------------------------------------
# cache contents the kernels must not depend on / must not touch
# ---------------------------------------------------------------------------

def test_stale_nan_past_context_end_is_ignored(dev):
    """Slots past a sequence's end (inside its last block) hold NaN bits."""
    w = pin.build_workload(params=dict(dtype="bf16", num_seqs=5, lens=[1, 7, 17, 250, 513],
                                       num_q_heads=32, num_kv_heads=8, head_dim=128,
                                       block_size=32), seed=5)
    kc = pin.bits(w.k_cache).copy()
    vc = pin.bits(w.v_cache).copy()
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        last = w.block_tables[b, (L - 1) // w.block_size]
        off = (L - 1) % w.block_size + 1
        kc[last, off:] = 0x7fc0
        vc[last, off:] = 0x7fc0
    w.k_cache = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    w.v_cache = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    check_workload(w, dev, partition_size=64)


def test_padding_and_out_of_pool_slots(dev):
    w = pin.build_workload(params=dict(dtype="fp16", num_seqs=4, lens=[3, 20, 40, 70],
                                       num_q_heads=8, num_kv_heads=2, head_dim=64,
                                       block_size=16), seed=9)
    slots = w.slot_mapping.copy()
    slots[1] = -1
    w.slot_mapping = slots
    check_workload(w, dev)                     # padding: nothing written, no error
    d = to_device(w, dev)
    before = d["k_cache"].clone()
    far = torch.tensor([w.num_blocks * w.block_size + 7], dtype=torch.int64, device=dev)
    lib.reshape_and_cache(d["k_new"][:1].contiguous(), d["v_new"][:1].contiguous(), far,
                          d["k_cache"], d["v_cache"])
    assert torch.equal(before, d["k_cache"])
    assert lib.read_device_errors(dev) == lib.PA_DEVERR_BAD_SLOT
    assert lib.read_device_errors(dev) == 0


def test_context_longer_than_table_is_clamped_and_flagged(dev):
    w = pin.build_workload(params=dict(dtype="fp16", num_seqs=2, lens=[30, 64], num_q_heads=8,
                                       num_kv_heads=2, head_dim=64, block_size=16), seed=4)
    d = to_device(w, dev)
    want = lib.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], d["context_lens"],
                      w.scale).clone()
    assert lib.read_device_errors(dev) == 0
    over = d["context_lens"].clone()
    over[1] = 64 + 1000                      # table row holds 4 blocks = 64 tokens
    got = lib.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"], over, w.scale)
    assert torch.equal(got, want)
    assert lib.read_device_errors(dev) & lib.PA_DEVERR_BAD_CONTEXT


def test_repeatable_bitwise(dev):
    w = pin.build_workload("tiny")
    d = to_device(w, dev)
    outs = [lib.paged_attention(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                d["context_lens"], w.scale, 250, mode=m).clone()
            for m in ("single", "single", "split", "split")]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[2], outs[3])


def test_non_default_stream(dev):
    w = pin.build_workload("tiny")
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        d = to_device(w, dev)
        out = lib.paged_attention(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                  d["context_lens"], w.scale, 250, mode="split")
    s.synchronize()
    want = oracle.paged_decode(pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache),
                               w.block_tables, w.context_lens, w.scale, w.dtype)
    assert_close(out.float().cpu().numpy(), want, "side stream")


@pytest.mark.parametrize("mode", ["single", "split", "fused", "balanced"])
def test_step_plan_eager_and_graph_replay(dev, mode):
    """The prepared step (and its CUDA-graph replay) equals the plain calls."""
    w = pin.build_workload(params=dict(dtype="bf16", num_seqs=9, lens=[1, 16, 33, 100, 600, 1000,
                                                                      1500, 2047, 2048],
                                       num_q_heads=32, num_kv_heads=8, head_dim=128,
                                       block_size=16), seed=21)
    d = to_device(w, dev)
    plan = lib.StepPlan(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"],
                        d["v_cache"], d["block_tables"], d["context_lens"], w.scale, 2048,
                        mode=mode)
    eager = plan().clone()
    kc, vc, _ = oracle.reshape_and_cache(pin.bits(w.k_new), pin.bits(w.v_new), w.slot_mapping,
                                         pin.bits(w.k_cache), pin.bits(w.v_cache), w.block_size)
    want = oracle.paged_decode(pin.bits(w.q), kc, vc, w.block_tables, w.context_lens, w.scale,
                               w.dtype)
    assert_close(eager.float().cpu().numpy(), want, f"plan {mode}")
    plan.out.zero_()
    plan.capture_graph()
    for _ in range(3):
        got = plan.replay()
    torch.cuda.synchronize(dev)
    assert torch.equal(got, eager)
    assert lib.read_device_errors(dev) == 0


def test_step_plan_chooses_the_partition(dev):
    """Without partition_size the plan takes the partition rule: over the
    lengths when context_lens is pinned host memory, with every context at
    the maximum when it is on the device.  One 12288-token context and
    seven of 256 tokens over 8 KV heads give different sizes (1536 at the
    maximum, 512 counted); both match the reference."""
    lens = [12288] + [256] * 7
    w = pin.build_workload(params=dict(dtype="fp16", num_seqs=8, lens=lens, num_q_heads=32,
                                       num_kv_heads=8, head_dim=128, block_size=16), seed=41)
    d = to_device(w, dev)
    kc, vc, _ = oracle.reshape_and_cache(pin.bits(w.k_new), pin.bits(w.v_new), w.slot_mapping,
                                         pin.bits(w.k_cache), pin.bits(w.v_cache), w.block_size)
    want = oracle.paged_decode(pin.bits(w.q), kc, vc, w.block_tables, w.context_lens, w.scale,
                               w.dtype)
    at_max = lib.choose_partition(8, 8, 12288, 16, dev)
    counted = lib.choose_partition(8, 8, 12288, 16, dev, w.context_lens)
    assert at_max != counted
    host_lens = d["context_lens"].cpu().pin_memory()
    for lens_t, expect in ((d["context_lens"], at_max), (host_lens, counted)):
        plan = lib.StepPlan(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"],
                            d["v_cache"], d["block_tables"], lens_t, w.scale, 12288,
                            mode="fused")
        assert plan.partition_size == expect
        got = plan()
        torch.cuda.synchronize(dev)
        assert_close(got.float().cpu().numpy(), want, f"partition {expect}")
    assert lib.read_device_errors(dev) == 0


def test_fused_step_rejects_a_slot_that_is_not_the_last_position(dev):
    """A slot other than position L-1's is not written; attention runs on the
    cache as it was, and the device error word reports it."""
    w = pin.build_workload(params=dict(dtype="fp16", num_seqs=3, lens=[5, 40, 700],
                                       num_q_heads=8, num_kv_heads=2, head_dim=128,
                                       block_size=16), seed=31)
    slots = w.slot_mapping.copy()
    slots[1] = slots[1] - 1                      # points at position L-2
    d = to_device(w, dev)
    d["slot_mapping"] = torch.from_numpy(slots).to(dev)
    before_k = d["k_cache"].clone()
    lib.read_device_errors(dev)
    out = lib.decode_step(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"],
                          d["v_cache"], d["block_tables"], d["context_lens"], w.scale, 700)
    torch.cuda.synchronize(dev)
    assert lib.read_device_errors(dev) & lib.PA_DEVERR_BAD_SLOT
    # sequences 0 and 2 got their token written; sequence 1 did not
    keep = slots.copy()
    keep[1] = -1
    kc, vc, _ = oracle.reshape_and_cache(pin.bits(w.k_new), pin.bits(w.v_new), keep,
                                         pin.bits(w.k_cache), pin.bits(w.v_cache), w.block_size)
    assert np.array_equal(pin.bits(d["k_cache"].cpu()), kc)
    assert not torch.equal(before_k, d["k_cache"])
    want = oracle.paged_decode(pin.bits(w.q), kc, vc, w.block_tables, w.context_lens, w.scale,
                               w.dtype)
    assert_close(out.float().cpu().numpy(), want, "fused step with a rejected slot")


def test_fused_step_back_to_back_steps(dev):
    """Consecutive steps reuse the counters; each step appends one token."""
    w = pin.build_workload(params=dict(dtype="bf16", num_seqs=4, lens=[1, 29, 600, 1300],
                                       num_q_heads=32, num_kv_heads=8, head_dim=128,
                                       block_size=16), seed=41)
    d = to_device(w, dev)
    ws = lib.step_workspace(d["q"], w.num_kv_heads, lib.num_partitions(2048, 512))
    kc, vc = pin.bits(w.k_cache), pin.bits(w.v_cache)
    lens = w.context_lens.copy()
    for step in range(3):
        if step:
            # next token: the allocator's slot for position L (same block unless it filled)
            lens = lens + 1
            slots = np.array([w.block_tables[b, (L - 1) // 16] * 16 + (L - 1) % 16
                              for b, L in enumerate(lens)], dtype=np.int64)
            if np.any((lens - 1) // 16 >= w.block_tables.shape[1]):
                break
            d["context_lens"] = torch.from_numpy(lens.astype(np.int32)).to(dev)
            d["slot_mapping"] = torch.from_numpy(slots).to(dev)
            rng = np.random.default_rng(step)
            kn = pin.normal_tensor(rng, tuple(w.k_new.shape), "bf16")
            vn = pin.normal_tensor(rng, tuple(w.v_new.shape), "bf16")
        else:
            slots, kn, vn = w.slot_mapping, w.k_new, w.v_new
        d["k_new"], d["v_new"] = kn.to(dev), vn.to(dev)
        out = lib.decode_step(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"],
                              d["v_cache"], d["block_tables"], d["context_lens"], w.scale, 2048,
                              workspace=ws)
        kc, vc, _ = oracle.reshape_and_cache(pin.bits(kn), pin.bits(vn), slots, kc, vc,
                                             w.block_size)
        want = oracle.paged_decode(pin.bits(w.q), kc, vc, w.block_tables, lens, w.scale,
                                   w.dtype)
        assert_close(out.float().cpu().numpy(), want, f"fused step {step}")
        assert int(ws[3].abs().sum()) == 0
    assert lib.read_device_errors(dev) == 0


def test_fused_step_with_hundreds_of_partitions(dev):
    """The fused step's merge reads the partition records four at a time, so
    any partition count works: 500 16-token partitions of an 8,000-token
    context at G = 8 (with contexts of 4,001 and 17 tokens beside it), cache
    write and output against the oracle."""
    w = pin.build_workload(params=dict(dtype="bf16", num_seqs=3, lens=[8000, 4001, 17],
                                       num_q_heads=64, num_kv_heads=8, head_dim=128,
                                       block_size=16), seed=91)
    check_workload(w, dev, modes=("fused",), partition_size=16)
