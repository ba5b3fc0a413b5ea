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
    return torch.device("cuda:0")


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
