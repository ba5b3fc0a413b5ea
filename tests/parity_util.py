"""Shared helpers of the GPU parity tests: run the CUDA path and the CPU
reference on the same seeded workload and compare.

Tolerance for attention outputs (fp16/bf16 caches, fp32 accumulation):
elementwise |gpu - ref| <= 2e-3 + 1e-2 * |ref|.  Cache writes: bit-exact.
"""
import numpy as np
import torch

import oracle
from paged_kv_cache_226_gb300 import inputs as pin
from paged_kv_cache_226_gb300 import lib

ATOL, RTOL = 2e-3, 1e-2


def assert_close(got, want, what, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                             f"worst at {i}: got {got[i]!r} want {want[i]!r}")
    return float(err.max()) if err.size else 0.0


def to_device(w: pin.Workload, dev):
    return dict(
        q=w.q.to(dev), k_new=w.k_new.to(dev), v_new=w.v_new.to(dev),
        k_cache=w.k_cache.to(dev), v_cache=w.v_cache.to(dev),
        block_tables=torch.from_numpy(w.block_tables).to(dev),
        context_lens=torch.from_numpy(w.context_lens).to(dev),
        slot_mapping=torch.from_numpy(w.slot_mapping).to(dev))


def gpu_bits(t: torch.Tensor) -> np.ndarray:
    return pin.bits(t.cpu())


def check_workload(w: pin.Workload, dev, modes=("single", "split", "fused", "balanced"),
                   partition_size=512,
                   check_partitions=True):
    """Cache write bit-exact, then decode through each mode against the oracle.
    Returns a dict of max errors."""
    d = to_device(w, dev)
    lib.reshape_and_cache(d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"], d["v_cache"])
    kc_ref, vc_ref, bad = oracle.reshape_and_cache(
        pin.bits(w.k_new), pin.bits(w.v_new), w.slot_mapping, pin.bits(w.k_cache),
        pin.bits(w.v_cache), w.block_size)
    torch.cuda.synchronize(dev)
    assert np.array_equal(gpu_bits(d["k_cache"]), kc_ref), "k_cache differs from the oracle"
    assert np.array_equal(gpu_bits(d["v_cache"]), vc_ref), "v_cache differs from the oracle"
    qb = pin.bits(w.q)
    want = oracle.paged_decode(qb, kc_ref, vc_ref, w.block_tables, w.context_lens, w.scale,
                               w.dtype)
    errs = {}
    max_len = int(w.context_lens.max()) if w.num_seqs else 0
    for mode in modes:
        if mode in ("fused", "balanced"):
            # one step from the unwritten caches: cache write + attention + merge
            kc = w.k_cache.to(dev)
            vc = w.v_cache.to(dev)
            if mode == "fused":
                S = lib.num_partitions(max_len, partition_size)
                ws = lib.step_workspace(d["q"], w.num_kv_heads, S)
                out = lib.decode_step(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], kc, vc,
                                      d["block_tables"], d["context_lens"], w.scale, max_len,
                                      partition_size=partition_size, workspace=ws)
                counters = ws[3]
            else:
                ws = lib.balanced_workspace(d["q"], kc, d["block_tables"])
                out = lib.decode_step_balanced(d["q"], d["k_new"], d["v_new"], d["slot_mapping"],
                                               kc, vc, d["block_tables"], d["context_lens"],
                                               w.scale, workspace=ws)
                counters = ws[:w.num_seqs * w.num_kv_heads * 4]
            torch.cuda.synchronize(dev)
            assert np.array_equal(gpu_bits(kc), kc_ref), f"{mode} step: k_cache differs"
            assert np.array_equal(gpu_bits(vc), vc_ref), f"{mode} step: v_cache differs"
            assert int(counters.abs().sum()) == 0, f"{mode} step left counters non-zero"
            errs[mode] = assert_close(out.float().cpu().numpy(), want, f"{w.name} {mode} out")
            continue
        if mode == "single":
            out = lib.decode(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                             d["context_lens"], w.scale)
        else:
            S = lib.num_partitions(max_len, partition_size)
            tmp, ml, es = lib.decode_split(d["q"], d["k_cache"], d["v_cache"],
                                           d["block_tables"], d["context_lens"], w.scale,
                                           partition_size, S)
            out = torch.empty_like(d["q"])
            lib.reduce(tmp, ml, es, d["context_lens"], partition_size, d["k_cache"],
                       w.max_blocks_per_seq, out)
            if check_partitions:
                po, pm, ps = oracle.paged_decode_partitions(
                    qb, kc_ref, vc_ref, w.block_tables, w.context_lens, w.scale, w.dtype,
                    partition_size, S)
                live = ~np.isnan(pm)
                errs["tmp_out"] = assert_close(tmp.cpu().numpy()[live], po[live],
                                               f"{w.name} split tmp_out")
                errs["max_logits"] = assert_close(ml.cpu().numpy()[live], pm[live],
                                                  f"{w.name} split max_logits")
                errs["exp_sums"] = assert_close(es.cpu().numpy()[live], ps[live],
                                                f"{w.name} split exp_sums")
        got = out.float().cpu().numpy()
        errs[mode] = assert_close(got, want, f"{w.name} {mode} out")
    assert lib.read_device_errors(dev) == 0
    return errs
