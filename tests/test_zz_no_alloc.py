"""pa_decode_static_workspace: the split decode whose partition workspace is
a fixed buffer inside the library, for callers that cannot allocate device
memory (a host framework owns the pool, or cudaMalloc's synchronisation is
not acceptable).

It runs the same kernels on the same partitions as pa_decode_split +
pa_reduce with a caller-owned workspace, so its output must equal that path
bit for bit, call after call, although every call reuses the same buffer;
and it must match the CPU reference within the parity tolerance.

This file is named to run last, so that a failure here comes after every
other test has run; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_226_gb300 import build, lib
from paged_kv_cache_226_gb300 import inputs as pin
from parity_util import assert_close, to_device

pytestmark = pytest.mark.gpu

LIMIT = 32 << 20          # PA_STATIC_WORKSPACE_BYTES


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib.load()
    return torch.device("cuda:0")


def _static_call(w, d, partition, S, out=None, partition_arg=None):
    """The static-workspace entry point called directly through ctypes;
    returns (status, out)."""
    pa = lib.load()
    out = torch.empty_like(d["q"]) if out is None else out
    shp = lib.make_shape(w.num_seqs, w.num_q_heads, d["k_cache"], w.max_blocks_per_seq)
    st = pa.pa_decode_static_workspace(
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k_cache"].data_ptr()),
        ctypes.c_void_p(d["v_cache"].data_ptr()), ctypes.c_void_p(d["block_tables"].data_ptr()),
        ctypes.c_void_p(d["context_lens"].data_ptr()), ctypes.c_float(w.scale),
        partition if partition_arg is None else partition_arg, S,
        ctypes.c_void_p(out.data_ptr()), ctypes.byref(shp),
        ctypes.c_void_p(torch.cuda.current_stream(d["q"].device).cuda_stream))
    return st, out


def _caller_workspace(w, d, partition, S):
    """pa_decode_split + pa_reduce with a workspace the caller allocates."""
    tmp, ml, es = lib.decode_split(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                   d["context_lens"], w.scale, partition, S)
    out = torch.empty_like(d["q"])
    lib.reduce(tmp, ml, es, d["context_lens"], partition, d["k_cache"], w.max_blocks_per_seq,
               out)
    return out


def _bits(t):
    return pin.bits(t.cpu())


def _oracle(w):
    return oracle.paged_decode(pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache),
                               w.block_tables, w.context_lens, w.scale, w.dtype)


def _max_partitions_that_fit(B, hq, d):
    """Largest S whose workspace -- [tmp_out][max_logits][exp_sums], each
    part rounded up to 256 bytes -- fits in the buffer."""
    def need(S):
        rows = B * hq * S
        r256 = lambda x: (x + 255) // 256 * 256
        return r256(4 * rows * d) + 2 * r256(4 * rows)
    S = 1
    while need(S + 1) <= LIMIT:
        S += 1
    return S, need(S), need(S + 1)


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
        S = lib.num_partitions(int(w.context_lens.max()), P)
        want = _caller_workspace(w, d, P, S)
        st, got = _static_call(w, d, P, S)
        assert st == lib.PA_OK, lib.status_string(st)
        assert np.array_equal(_bits(got), _bits(want)), \
            f"static workspace differs from the caller-workspace path ({w.name})"
        # the second call through the Python binding of the same entry point
        again = lib.decode_static_workspace(d["q"], d["k_cache"], d["v_cache"],
                                            d["block_tables"], d["context_lens"], w.scale,
                                            int(w.context_lens.max()), partition_size=P)
        assert np.array_equal(_bits(again), _bits(want)), f"second call differs ({w.name})"
        assert_close(again.float().cpu().numpy(), _oracle(w), f"static workspace vs oracle "
                                                               f"({w.name})")
    assert lib.read_device_errors(dev) == 0


def test_static_workspace_limit_edge(dev):
    """A request that fills the buffer exactly as far as the rounding rule
    allows runs and matches the caller-workspace path; one more partition is
    refused with PA_ERR_WORKSPACE."""
    w = pin.build_workload(params=dict(dtype="fp16", num_seqs=1, lens=[1000], num_q_heads=8,
                                       num_kv_heads=2, head_dim=128, block_size=16), seed=31)
    S, need, need_next = _max_partitions_that_fit(1, 8, 128)
    assert need <= LIMIT < need_next
    d = to_device(w, dev)
    P = 16                                  # 63 live partitions, the rest past the end
    want = _caller_workspace(w, d, P, S)
    st, got = _static_call(w, d, P, S)
    assert st == lib.PA_OK, lib.status_string(st)
    assert np.array_equal(_bits(got), _bits(want))
    assert_close(got.float().cpu().numpy(), _oracle(w), "static workspace at its limit")
    sentinel = torch.full_like(d["q"], 7.0)
    st, after = _static_call(w, d, P, S + 1, out=sentinel)
    assert st == lib.PA_ERR_WORKSPACE
    torch.cuda.synchronize(dev)
    assert bool((after == 7.0).all()), "a refused request wrote its output"
    assert lib.read_device_errors(dev) == 0


def test_static_workspace_error_order(dev):
    """Malformed requests get the status pa_decode_split + pa_reduce give
    them, before the size limit is considered."""
    w = pin.build_workload("tiny")
    d = to_device(w, dev)
    # 4 seqs x 8 heads x 5000 partitions x 64 dims x 4 B is far over 32 MiB
    st, _ = _static_call(w, d, 16, 5000)
    assert st == lib.PA_ERR_WORKSPACE
    st, _ = _static_call(w, d, 16, 5000, partition_arg=24)      # not a multiple of the block
    assert st == lib.PA_ERR_INVALID_ARG
    st, _ = _static_call(w, d, 16, 70000)                        # over 65535 partitions
    assert st == lib.PA_ERR_UNSUPPORTED
    st, _ = _static_call(w, d, 16, 0)
    assert st == lib.PA_ERR_WORKSPACE
