"""GPU parity of the FP8 (E4M3) KV cache: the quantising cache write is
bit-exact, and decode over the codes (single pass, split + merge, fused
step) matches the fp64 reference within |gpu - ref| <= 2e-3 + 1e-2 |ref|."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_226_gb300 import build, lib
from paged_kv_cache_226_gb300 import inputs as pin
from parity_util import assert_close

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 1.0 / 64, 1.0 / 48


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib.load()
    d = torch.device("cuda:0")
    lib.read_device_errors(d)
    return d


def _fp8_case(name=None, params=None, seed=None):
    w = pin.build_workload(name, params=params, seed=seed)
    rng = np.random.default_rng(1234)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = pin.fp8_codes(rng, shape, K_SCALE)
    vc = pin.fp8_codes(rng, shape, V_SCALE)
    return w, kc, vc


@pytest.mark.parametrize("dtype,scale", [("fp16", 0.05), ("bf16", 0.004)])
def test_fp8_cache_write_bit_exact(dev, dtype, scale):
    """0.004 pushes a share of the values past 448: they must saturate."""
    w, kc, vc = _fp8_case(params=dict(dtype=dtype, num_seqs=7, lens=[1, 15, 16, 17, 100, 513, 900],
                                      num_q_heads=16, num_kv_heads=4, head_dim=128,
                                      block_size=16), seed=3)
    slots = w.slot_mapping.copy()
    slots[2] = -1
    kd, vd = kc.to(dev), vc.to(dev)
    lib.reshape_and_cache_fp8(w.k_new.to(dev), w.v_new.to(dev), torch.from_numpy(slots).to(dev),
                              kd, vd, scale, 2 * scale)
    wk, wv, bad = oracle.reshape_and_cache_fp8(pin.bits(w.k_new), pin.bits(w.v_new), slots,
                                               kc.numpy(), vc.numpy(), w.block_size, dtype,
                                               scale, 2 * scale)
    torch.cuda.synchronize(dev)
    assert bad == 0
    assert np.array_equal(kd.cpu().numpy(), wk) and np.array_equal(vd.cpu().numpy(), wv)
    if scale < 0.01:
        assert (wk == 0x7e).any() or (wk == 0xfe).any()        # saturation was exercised
    assert lib.read_device_errors(dev) == 0


def _check_fp8(w, kc, vc, dev, partition_size=512):
    d = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).to(dev)
         for k, v in dict(q=w.q, k_new=w.k_new, v_new=w.v_new, bt=w.block_tables,
                          cl=w.context_lens, sm=w.slot_mapping).items()}
    kd, vd = kc.to(dev), vc.to(dev)
    # the layer-step reference: quantised write of the new tokens, then attention
    wk, wv, _ = oracle.reshape_and_cache_fp8(pin.bits(w.k_new), pin.bits(w.v_new),
                                             w.slot_mapping, kc.numpy(), vc.numpy(),
                                             w.block_size, w.dtype, K_SCALE, V_SCALE)
    want = oracle.paged_decode_fp8(pin.bits(w.q), wk, wv, w.block_tables, w.context_lens,
                                   w.scale, K_SCALE, V_SCALE, w.dtype)
    max_len = int(w.context_lens.max())
    # fused step from the unwritten cache
    out = lib.decode_step_fp8(d["q"], d["k_new"], d["v_new"], d["sm"], kd, vd, d["bt"], d["cl"],
                              w.scale, K_SCALE, V_SCALE, max_len, partition_size=partition_size)
    torch.cuda.synchronize(dev)
    assert np.array_equal(kd.cpu().numpy(), wk) and np.array_equal(vd.cpu().numpy(), wv)
    assert_close(out.float().cpu().numpy(), want, f"{w.name} fp8 fused step")
    # the balanced step from the unwritten cache
    kb, vb = kc.to(dev), vc.to(dev)
    outb = lib.decode_step_balanced(d["q"], d["k_new"], d["v_new"], d["sm"], kb, vb, d["bt"],
                                    d["cl"], w.scale, k_scale=K_SCALE, v_scale=V_SCALE)
    torch.cuda.synchronize(dev)
    assert np.array_equal(kb.cpu().numpy(), wk) and np.array_equal(vb.cpu().numpy(), wv)
    assert_close(outb.float().cpu().numpy(), want, f"{w.name} fp8 balanced step")
    # single pass and split + merge over the written cache
    single = lib.decode_fp8(d["q"], kd, vd, d["bt"], d["cl"], w.scale, K_SCALE, V_SCALE)
    assert_close(single.float().cpu().numpy(), want, f"{w.name} fp8 single")
    S = lib.num_partitions(max_len, partition_size)
    tmp, ml, es = lib.decode_split_fp8(d["q"], kd, vd, d["bt"], d["cl"], w.scale, K_SCALE,
                                       V_SCALE, partition_size, S)
    merged = lib.reduce(tmp, ml, es, d["cl"], partition_size, kd, w.max_blocks_per_seq,
                        torch.empty_like(d["q"]))
    assert_close(merged.float().cpu().numpy(), want, f"{w.name} fp8 split")
    assert lib.read_device_errors(dev) == 0


@pytest.mark.parametrize("name", ["llama8b", "llama70b"])
def test_fp8_named_workload(dev, name):
    w, kc, vc = _fp8_case(name)
    _check_fp8(w, kc, vc, dev)


@pytest.mark.parametrize("dtype,bs", [("bf16", 16), ("fp16", 32)])
def test_fp8_edge_lengths(dev, dtype, bs):
    lens = [0, 1, 2, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1100]
    w, kc, vc = _fp8_case(params=dict(dtype=dtype, num_seqs=len(lens), lens=lens, num_q_heads=32,
                                      num_kv_heads=8, head_dim=128, block_size=bs), seed=17)
    for P in (bs, 64, 512):
        _check_fp8(w, kc, vc, dev, partition_size=P)


@pytest.mark.parametrize("log2_q", [17, -20, 0])
def test_fp8_bf16_query_magnitudes(dev, log2_q):
    """A bf16 query far above fp16's range (2^17) or far below its normal range
    (2^-20), with the softmax scale compensating, attends like any other: the
    FP8 path computes in fp16 and must bring q into range first."""
    w, kc, vc = _fp8_case(params=dict(dtype="bf16", num_seqs=5, lens=[1, 33, 300, 700, 1500],
                                      num_q_heads=32, num_kv_heads=8, head_dim=128,
                                      block_size=16), seed=23)
    w.q = (w.q.float() * 2.0 ** log2_q).to(torch.bfloat16)
    w.scale = w.scale * 2.0 ** -log2_q
    _check_fp8(w, kc, vc, dev)


def test_fp8_rejects_head_dim_64_and_bad_scales(dev):
    q = torch.zeros((1, 4, 64), dtype=torch.float16, device=dev)
    kc = torch.zeros((4, 16, 2, 64), dtype=torch.uint8, device=dev)
    bt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    cl = torch.ones((1,), dtype=torch.int32, device=dev)
    with pytest.raises(lib.PaError, match="unsupported"):
        lib.decode_fp8(q, kc, kc, bt, cl, 0.1, 1.0, 1.0)
    q2 = torch.zeros((1, 4, 128), dtype=torch.float16, device=dev)
    kc2 = torch.zeros((4, 16, 2, 128), dtype=torch.uint8, device=dev)
    with pytest.raises(lib.PaError, match="invalid"):
        lib.decode_fp8(q2, kc2, kc2, bt, cl, 0.1, 0.0, 1.0)


@pytest.mark.parametrize("mode", ["fused", "balanced"])
def test_fp8_repeated_steps(dev, mode):
    """Eight layer-steps over fresh copies of the same cache, each against the
    reference.  An FP8 tile hands its ring stage back before its P.V products;
    before the stage release ordered the warp's reads ahead of the refill
    (a proxy fence), about half of such runs had one partition of one
    (sequence, KV head) computed from a half-overwritten tile."""
    w, kc, vc = _fp8_case("llama70b")
    d = {k: (torch.from_numpy(v) if isinstance(v, np.ndarray) else v).to(dev)
         for k, v in dict(q=w.q, k_new=w.k_new, v_new=w.v_new, bt=w.block_tables,
                          cl=w.context_lens, sm=w.slot_mapping).items()}
    wk, wv, _ = oracle.reshape_and_cache_fp8(pin.bits(w.k_new), pin.bits(w.v_new),
                                             w.slot_mapping, kc.numpy(), vc.numpy(),
                                             w.block_size, w.dtype, K_SCALE, V_SCALE)
    want = oracle.paged_decode_fp8(pin.bits(w.q), wk, wv, w.block_tables, w.context_lens,
                                   w.scale, K_SCALE, V_SCALE, w.dtype)
    max_len = int(w.context_lens.max())
    for trial in range(8):
        kd, vd = kc.to(dev), vc.to(dev)
        if mode == "fused":
            out = lib.decode_step_fp8(d["q"], d["k_new"], d["v_new"], d["sm"], kd, vd, d["bt"],
                                      d["cl"], w.scale, K_SCALE, V_SCALE, max_len)
        else:
            out = lib.decode_step_balanced(d["q"], d["k_new"], d["v_new"], d["sm"], kd, vd,
                                           d["bt"], d["cl"], w.scale, k_scale=K_SCALE,
                                           v_scale=V_SCALE)
        assert_close(out.float().cpu().numpy(), want, f"{mode} fp8 step, run {trial}")
    assert lib.read_device_errors(dev) == 0
