"""lib.InputStaging: a layer-step's inputs as aligned views of one pinned host
buffer and one device buffer, uploaded by a single copy; a step planned on the
device views gives the same output as one planned on separate tensors."""
import numpy as np
import pytest
import torch

from paged_kv_cache_226_gb300 import build, lib
from paged_kv_cache_226_gb300 import inputs as pin

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


def test_staged_step_matches_separate_tensors(dev):
    w = pin.build_workload(params=dict(dtype="bf16", num_seqs=9, lens=[1, 16, 17, 40, 100, 511,
                                                                       512, 513, 900],
                                       num_q_heads=16, num_kv_heads=4, head_dim=128,
                                       block_size=16), seed=31)
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    src = {k: (torch.from_numpy(getattr(w, k)) if isinstance(getattr(w, k), np.ndarray)
               else getattr(w, k)) for k in names}
    stage = lib.InputStaging({k: (tuple(t.shape), t.dtype) for k, t in src.items()}, dev)
    for k, t in src.items():
        stage.h[k].copy_(t)
    for k in names:
        assert stage.d[k].data_ptr() % 256 == 0
    stage.upload()
    torch.cuda.synchronize(dev)
    for k, t in src.items():
        assert torch.equal(stage.d[k].cpu(), t)
    max_len = int(w.context_lens.max())
    kc1, vc1 = w.k_cache.to(dev), w.v_cache.to(dev)
    kc2, vc2 = kc1.clone(), vc1.clone()
    staged = lib.StepPlan(stage.d["q"], stage.d["k_new"], stage.d["v_new"],
                          stage.d["slot_mapping"], kc1, vc1, stage.d["block_tables"],
                          stage.d["context_lens"], w.scale, max_len)
    sep = {k: t.to(dev) for k, t in src.items()}
    plain = lib.StepPlan(sep["q"], sep["k_new"], sep["v_new"], sep["slot_mapping"], kc2, vc2,
                         sep["block_tables"], sep["context_lens"], w.scale, max_len)
    staged()
    plain()
    torch.cuda.synchronize(dev)
    assert torch.equal(staged.out, plain.out)
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    assert lib.read_device_errors(dev) == 0


def test_graph_with_upload_and_readback(dev):
    """A step captured with its upload and read-back replays to the same output
    after the host inputs change (new token rows written between replays)."""
    w = pin.build_workload(params=dict(dtype="fp16", num_seqs=6, lens=[3, 40, 77, 300, 512, 1000],
                                       num_q_heads=32, num_kv_heads=8, head_dim=128,
                                       block_size=16), seed=37)
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    src = {k: (torch.from_numpy(getattr(w, k)) if isinstance(getattr(w, k), np.ndarray)
               else getattr(w, k)) for k in names}
    stage = lib.InputStaging({k: (tuple(t.shape), t.dtype) for k, t in src.items()}, dev)
    for k, t in src.items():
        stage.h[k].copy_(t)
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    plan = lib.StepPlan(stage.d["q"], stage.d["k_new"], stage.d["v_new"], stage.d["slot_mapping"],
                        kc, vc, stage.d["block_tables"], stage.d["context_lens"], w.scale,
                        int(w.context_lens.max()))
    out_h = torch.empty(plan.out.shape, dtype=plan.out.dtype).pin_memory()
    plan.capture_graph(before=stage.upload, after=lambda: out_h.copy_(plan.out, non_blocking=True))
    for rep in range(2):
        stage.h["q"].copy_(src["q"] * (1.0 + rep))
        plan.replay()
        torch.cuda.synchronize(dev)
        got = out_h.clone()
        assert torch.equal(stage.d["q"].cpu(), stage.h["q"])      # the replay uploaded
        plan()                                   # the same step outside the graph
        torch.cuda.synchronize(dev)
        assert torch.equal(got, plan.out.cpu())
        ref = lib.decode(stage.d["q"], kc, vc, stage.d["block_tables"], stage.d["context_lens"],
                         w.scale)
        torch.cuda.synchronize(dev)
        assert torch.allclose(got.float(), ref.float().cpu(), atol=2e-3, rtol=1e-2)
    assert lib.read_device_errors(dev) == 0


def test_copy_async_between_pinned_host_and_device(dev):
    """pa_copy_async moves bytes exactly between pinned host and device memory
    in both directions and within the device; bad sizes are refused."""
    n = (1 << 20) + 4096 + 48                      # not a multiple of the grid's chunking
    src = torch.randint(-2**31, 2**31 - 1, (n // 4,), dtype=torch.int32).pin_memory()
    d1 = torch.empty(n // 4, dtype=torch.int32, device=dev)
    d2 = torch.empty_like(d1)
    back = torch.empty(n // 4, dtype=torch.int32).pin_memory()
    lib.copy_async(d1, src)
    lib.copy_async(d2, d1)
    lib.copy_async(back, d2)
    torch.cuda.synchronize(dev)
    assert torch.equal(back, src)
    with pytest.raises(lib.PaError):
        lib.copy_async(d1[1:5], src[1:5])          # 4-byte aligned, not 16
    with pytest.raises(ValueError):
        lib.copy_async(d1, torch.empty(n // 4, dtype=torch.int32))   # pageable host memory


@pytest.mark.parametrize("cache", ["fp16", "fp8"])
def test_fused_step_with_pinned_host_inputs_and_output(dev, cache):
    """The fused step reading q, the new K/V, slots, tables and lengths from
    pinned host memory and writing its output there gives the device-memory
    step's output and cache bits exactly, step after step (the host inputs
    change between steps, as a serving loop writes them)."""
    w = pin.build_workload(params=dict(dtype="fp16", num_seqs=7, lens=[1, 16, 17, 300, 1024, 1500,
                                                                       2049],
                                       num_q_heads=32, num_kv_heads=8, head_dim=128,
                                       block_size=16), seed=41)
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    src = {k: (torch.from_numpy(getattr(w, k)) if isinstance(getattr(w, k), np.ndarray)
               else getattr(w, k)) for k in names}
    host = {k: t.clone().pin_memory() for k, t in src.items()}
    devt = {k: t.to(dev) for k, t in src.items()}
    scales = {}
    if cache == "fp8":
        rng = np.random.default_rng(5)
        kc1 = pin.fp8_codes(rng, tuple(w.k_cache.shape), 1 / 64).to(dev)
        vc1 = pin.fp8_codes(rng, tuple(w.v_cache.shape), 1 / 48).to(dev)
        scales = dict(k_scale=1 / 64, v_scale=1 / 48)
    else:
        kc1, vc1 = w.k_cache.to(dev), w.v_cache.to(dev)
    kc2, vc2 = kc1.clone(), vc1.clone()
    max_len = int(w.context_lens.max())
    out_h = torch.zeros(tuple(src["q"].shape), dtype=src["q"].dtype).pin_memory()
    zero_copy = lib.StepPlan(host["q"], host["k_new"], host["v_new"], host["slot_mapping"], kc1,
                             vc1, host["block_tables"], host["context_lens"], w.scale, max_len,
                             out=out_h, mode="fused", partition_size=512, **scales)
    on_dev = lib.StepPlan(devt["q"], devt["k_new"], devt["v_new"], devt["slot_mapping"], kc2, vc2,
                          devt["block_tables"], devt["context_lens"], w.scale, max_len,
                          mode="fused", partition_size=512, **scales)
    for step in range(3):
        q = src["q"] * (1.0 + 0.5 * step)
        host["q"].copy_(q)
        devt["q"].copy_(q.to(dev))
        zero_copy()
        on_dev()
        torch.cuda.synchronize(dev)
        assert torch.equal(out_h.view(torch.int16), on_dev.out.cpu().view(torch.int16)), step
        assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    with pytest.raises(ValueError):              # pageable host memory is refused
        lib.StepPlan(src["q"], host["k_new"], host["v_new"], host["slot_mapping"], kc1, vc1,
                     host["block_tables"], host["context_lens"], w.scale, max_len, out=out_h,
                     mode="fused", **scales)
    with pytest.raises(ValueError):              # host inputs only in the fused mode
        lib.StepPlan(host["q"], host["k_new"], host["v_new"], host["slot_mapping"], kc1, vc1,
                     host["block_tables"], host["context_lens"], w.scale, max_len, out=out_h,
                     mode="split")
    assert lib.read_device_errors(dev) == 0
