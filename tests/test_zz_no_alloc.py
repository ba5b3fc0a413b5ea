"""pa_decode_static_workspace: the split decode whose partition workspace is
a fixed buffer inside the library, for callers that cannot allocate device
memory (a host framework owns the pool, or cudaMalloc's synchronisation is
not acceptable).  Its output must match the caller-workspace path
(pa_decode_split + pa_reduce) within the parity tolerance, call after call,
although every call reuses the same buffer.

This file is named to run last, so that a failure here comes after every
other test has run; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

from paged_kv_cache_226_gb300 import build, lib
from paged_kv_cache_226_gb300 import inputs as pin
from parity_util import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib.load()
    return torch.device("cuda:0")


def _via_c_abi(w, d, partition):
    """Call the static-workspace entry point directly through ctypes."""
    pa = lib.load()
    out = torch.empty_like(d["q"])
    shp = lib.make_shape(w.num_seqs, w.num_q_heads, d["k_cache"], w.max_blocks_per_seq)
    S = lib.num_partitions(int(w.context_lens.max()), partition)
    st = pa.pa_decode_static_workspace(
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k_cache"].data_ptr()),
        ctypes.c_void_p(d["v_cache"].data_ptr()), ctypes.c_void_p(d["block_tables"].data_ptr()),
        ctypes.c_void_p(d["context_lens"].data_ptr()), ctypes.c_float(w.scale),
        partition, S, ctypes.c_void_p(out.data_ptr()), ctypes.byref(shp),
        ctypes.c_void_p(torch.cuda.current_stream(d["q"].device).cuda_stream))
    assert st == lib.PA_OK, lib.status_string(st)
    return out


def _via_caller_workspace(w, d, partition):
    return lib.paged_attention(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                               d["context_lens"], w.scale, int(w.context_lens.max()),
                               mode="split", partition_size=partition)


def test_static_workspace_matches_caller_workspace_twice(dev):
    # Two different workloads back to back: the second call finds the first
    # call's partitions in the shared buffer and must not be affected.
    cases = [(pin.build_workload("llama8b"), 512),
             (pin.build_workload(params=dict(dtype="bf16", num_seqs=5,
                                             lens=[1, 17, 300, 2000, 4100], num_q_heads=16,
                                             num_kv_heads=2, head_dim=64, block_size=32),
                                 seed=77), 64)]
    for w, P in cases:
        d = to_device(w, dev)
        want = _via_caller_workspace(w, d, P).float().cpu().numpy()
        got = _via_c_abi(w, d, P).float().cpu().numpy()
        assert_close(got, want, f"static workspace vs caller workspace ({w.name})")
        again = lib.decode_static_workspace(d["q"], d["k_cache"], d["v_cache"],
                                            d["block_tables"], d["context_lens"], w.scale,
                                            int(w.context_lens.max()), partition_size=P)
        assert_close(again.float().cpu().numpy(), want, f"second call ({w.name})")
    assert lib.read_device_errors(dev) == 0


def test_static_workspace_rejects_requests_over_its_limit(dev):
    w = pin.build_workload("tiny")
    d = to_device(w, dev)
    pa = lib.load()
    shp = lib.make_shape(w.num_seqs, w.num_q_heads, d["k_cache"], w.max_blocks_per_seq)
    # 4 seqs x 8 heads x S x 64 dims x 4 B > 32 MiB once S > 4096
    st = pa.pa_decode_static_workspace(
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k_cache"].data_ptr()),
        ctypes.c_void_p(d["v_cache"].data_ptr()), ctypes.c_void_p(d["block_tables"].data_ptr()),
        ctypes.c_void_p(d["context_lens"].data_ptr()), ctypes.c_float(w.scale), 16, 5000,
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.byref(shp), None)
    assert st == lib.PA_ERR_WORKSPACE
