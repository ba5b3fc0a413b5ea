"""Failure detection on the device without a GPU fault: a pipeline wait that
runs out ends the kernel with PA_DEVERR_WAIT_TIMEOUT in the device error
word, the context stays usable, and after the documented recovery (zero the
fused step's counters) the next step matches the CPU reference.

The wait is made to run out in libpa_test.so, a build of the same sources
with -DPA_TEST_HOOKS (include/pa_test.h): the TMA producer of one CTA issues
no tile from a chosen tile on -- no expect_tx and no copy, so no bulk copy is
in flight when the CTA ends -- and every pipeline wait gives up after a few
milliseconds instead of a second.  The product library has no such hook."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_226_gb300 import build, lib
from paged_kv_cache_226_gb300 import inputs as pin
from parity_util import assert_close, to_device

pytestmark = pytest.mark.gpu

SHORT_LIMIT_NS = 2_000_000          # 2 ms
PRODUCT_LIMIT_NS = 1_000_000_000    # the product build's one second


@pytest.fixture(scope="module")
def test_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = lib.load(build.build(test_hooks=True))
    L.pa_test_set_wait_fault.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_ulonglong]
    L.pa_test_set_wait_fault.restype = ctypes.c_int
    return L


def test_wait_timeout_is_reported_and_the_next_step_recovers(test_lib, monkeypatch):
    monkeypatch.setattr(lib, "_lib", test_lib)       # the binding's calls go to the test build
    dev = torch.device("cuda:0")
    w = pin.build_workload(params=dict(dtype="fp16", num_seqs=4, lens=[100, 600, 1300, 2000],
                                       num_q_heads=8, num_kv_heads=2, head_dim=128,
                                       block_size=16), seed=61)
    d = to_device(w, dev)
    max_len, P = 2000, 512
    ws = lib.step_workspace(d["q"], w.num_kv_heads, lib.num_partitions(max_len, P))
    kc, vc, _ = oracle.reshape_and_cache(pin.bits(w.k_new), pin.bits(w.v_new), w.slot_mapping,
                                         pin.bits(w.k_cache), pin.bits(w.v_cache), w.block_size)
    want = oracle.paged_decode(pin.bits(w.q), kc, vc, w.block_tables, w.context_lens, w.scale,
                               w.dtype)
    lib.read_device_errors(dev)

    def step():
        return lib.decode_step(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"],
                               d["v_cache"], d["block_tables"], d["context_lens"], w.scale,
                               max_len, partition_size=P, workspace=ws)

    try:
        # CTA 0 = (sequence 0, KV head 0, partition 0): 7 tiles, the third
        # and later withheld; CTA 9 = (sequence 1, KV head 0, partition 1):
        # one partition of a sequence whose partitions merge in the kernel
        for cta, tile in ((0, 2), (9, 0)):
            assert test_lib.pa_test_set_wait_fault(cta, tile, SHORT_LIMIT_NS) == lib.PA_OK
            step()
            torch.cuda.synchronize(dev)                  # the kernel ends: no hang
            flags = lib.read_device_errors(dev)
            assert flags & lib.PA_DEVERR_WAIT_TIMEOUT, f"no timeout reported (flags {flags})"
    finally:
        assert test_lib.pa_test_set_wait_fault(-1, 0, PRODUCT_LIMIT_NS) == lib.PA_OK
    # recovery as documented: counters to zero, then a normal step (the
    # cache writes of the faulty steps put the same new tokens in the same
    # slots, so the cache is as the reference expects)
    ws[3].zero_()
    out = step()
    torch.cuda.synchronize(dev)
    assert np.array_equal(pin.bits(d["k_cache"].cpu()), kc)
    assert np.array_equal(pin.bits(d["v_cache"].cpu()), vc)
    assert_close(out.float().cpu().numpy(), want, "step after a wait timeout")
    assert int(ws[3].abs().sum()) == 0
    assert lib.read_device_errors(dev) == 0
