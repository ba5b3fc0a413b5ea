"""Plain CPU reference ("oracle") for paged decode attention.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg are the only code allowed to import this package.
The product path (the CUDA library and its Python binding) never imports it and
shares no code with it.

The arithmetic lives in ``oracle.c`` (fp64, exact widening of the 16-bit
inputs); this module only loads it with ctypes and marshals numpy arrays.
``alloc_model`` holds the allocator / waste accounting from the pages.

Arrays of 16-bit floats are passed as their raw bit patterns (``uint16``);
``dtype`` is ``"fp16"`` or ``"bf16"``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_DTYPES = {"fp16": 0, "bf16": 1}
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fopenmp", "-shared",
           "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_f16_to_f64.restype = f64
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = f64
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_widen.restype = None
            lib.oracle_widen.argtypes = [P, P, i64, i32]
            lib.oracle_reshape_and_cache.restype = i64
            lib.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64]
            lib.oracle_paged_decode.restype = i32
            lib.oracle_paged_decode.argtypes = [P, P, P, P, P, f64, i32, i32, i32, i32,
                                                i32, i32, i32, P]
            lib.oracle_paged_decode_partitions.restype = i32
            lib.oracle_paged_decode_partitions.argtypes = [P, P, P, P, P, f64, i32, i32, i32,
                                                           i32, i32, i32, i32, i32, i32, P, P, P]
            lib.oracle_lse_merge.restype = i32
            lib.oracle_lse_merge.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P]
            lib.oracle_contiguous_decode.restype = i32
            lib.oracle_contiguous_decode.argtypes = [P, P, P, P, P, f64, i32, i32, i32, i32,
                                                     i32, P]
            lib.oracle_e4m3_to_f64.restype = f64
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_f32_to_e4m3.restype = ctypes.c_uint8
            lib.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
            lib.oracle_reshape_and_cache_fp8.restype = i64
            lib.oracle_reshape_and_cache_fp8.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64,
                                                         i32, ctypes.c_float, ctypes.c_float]
            lib.oracle_paged_decode_fp8.restype = i32
            lib.oracle_paged_decode_fp8.argtypes = [P, P, P, P, P, f64, f64, f64, i32, i32, i32,
                                                    i32, i32, i32, i32, P]
            lib.oracle_paged_prefill.restype = i32
            lib.oracle_paged_prefill.argtypes = [P, P, P, P, P, P, f64, i32, i32, i32, i32, i32,
                                                 i32, i32, P]
            lib.oracle_copy_blocks.restype = i64
            lib.oracle_copy_blocks.argtypes = [P, P, i64, P, P, i64, P, i64, i32, i32, i32]
            lib.oracle_max_threads.restype = i32
            lib.oracle_max_threads.argtypes = []
            lib.oracle_set_threads.restype = None
            lib.oracle_set_threads.argtypes = [i32]
            _lib = lib
    return _lib


class use_library:
    """Test helper: route the wrappers below to another build of oracle.c
    (used to check that the pins fail on a deliberately broken copy)."""

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        _load()
        lib = ctypes.CDLL(self.path)
        for name in dir(_lib):
            if name.startswith("oracle_"):
                fn, ref = getattr(lib, name), getattr(_lib, name)
                fn.restype, fn.argtypes = ref.restype, ref.argtypes
        with _lock:
            self.saved, _lib = _lib, lib
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile a modified copy of oracle.c (test helper)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O1", "-std=c99", "-ffp-contract=off", "-shared", "-fPIC", src,
                    "-o", out_path, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        if a.dtype.itemsize != 2:
            raise TypeError(f"expected 16-bit bit patterns, got {a.dtype}")
        a = a.view(np.uint16)
    return a


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def f16_to_f64(bits: int) -> float:
    return float(_load().oracle_f16_to_f64(int(bits)))


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(bits)))


def widen(bits, dtype: str) -> np.ndarray:
    """Exact value of each 16-bit pattern as float64."""
    src = _u16(bits)
    dst = np.empty(src.shape, dtype=np.float64)
    _load().oracle_widen(_ptr(src), _ptr(dst), src.size, _DTYPES[dtype])
    return dst


def reshape_and_cache(k, v, slot_mapping, k_cache, v_cache, block_size: int):
    """Return (k_cache', v_cache', n_out_of_pool) after writing the new tokens.

    k, v: [T][Hkv][D] bits; caches: [NB][bs][Hkv][D] bits (copied, not
    modified); slot_mapping: int64 [T], negative = padding.
    """
    k, v = _u16(k), _u16(v)
    kc, vc = _u16(k_cache).copy(), _u16(v_cache).copy()
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = sm.shape[0]
    nb, bs, hkv, d = kc.shape
    assert bs == block_size and k.shape == (T, hkv, d) and v.shape == (T, hkv, d)
    bad = _load().oracle_reshape_and_cache(_ptr(k), _ptr(v), _ptr(sm), _ptr(kc), _ptr(vc),
                                           T, hkv, d, bs, nb)
    return kc, vc, int(bad)


def e4m3_to_f64(code: int) -> float:
    return float(_load().oracle_e4m3_to_f64(int(code)))


def f32_to_e4m3(y: float) -> int:
    """Nearest E4M3 code (ties to even, saturating at 448) of float32(y)."""
    return int(_load().oracle_f32_to_e4m3(float(np.float32(y))))


def reshape_and_cache_fp8(k, v, slot_mapping, k_cache, v_cache, block_size: int, dtype: str,
                          k_scale: float, v_scale: float):
    """FP8 cache write: returns (k_cache', v_cache', n_out_of_pool); caches
    are uint8 [NB][bs][Hkv][D] (copied, not modified)."""
    k, v = _u16(k), _u16(v)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8).copy()
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8).copy()
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = sm.shape[0]
    nb, bs, hkv, d = kc.shape
    assert bs == block_size and k.shape == (T, hkv, d) and v.shape == (T, hkv, d)
    bad = _load().oracle_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(sm), _ptr(kc), _ptr(vc),
                                               T, hkv, d, bs, nb, _DTYPES[dtype],
                                               float(k_scale), float(v_scale))
    return kc, vc, int(bad)


def paged_decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                     k_scale: float, v_scale: float, dtype: str) -> np.ndarray:
    """fp64 attention over an E4M3 cache (uint8 [NB][bs][Hkv][D])."""
    q = _u16(q)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, hq, d = q.shape
    nb, bs, hkv, d2 = kc.shape
    assert d2 == d and vc.shape == kc.shape and cl.shape == (B,) and bt.shape[0] == B
    out = np.zeros((B, hq, d), dtype=np.float64)
    rc = _load().oracle_paged_decode_fp8(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl),
                                         float(scale), float(k_scale), float(v_scale), B, hq,
                                         hkv, d, bs, bt.shape[1], _DTYPES[dtype], _ptr(out))
    if rc != 0:
        raise ValueError("oracle_paged_decode_fp8: bad shape")
    return out


def copy_blocks(k_src, v_src, k_dst, v_dst, mapping):
    """Return (k_dst', v_dst', n_skipped): copies of the destination pools with
    the mapped blocks copied in.  Pools [NB][bs][Hkv][D] bits; mapping int64
    [P][2] of (src, dst)."""
    ks, vs = _u16(k_src), _u16(v_src)
    kd, vd = _u16(k_dst).copy(), _u16(v_dst).copy()
    mp = np.ascontiguousarray(mapping, dtype=np.int64).reshape(-1, 2)
    _, bs, hkv, d = ks.shape
    assert kd.shape[1:] == ks.shape[1:] and vs.shape == ks.shape and vd.shape == kd.shape
    bad = _load().oracle_copy_blocks(_ptr(ks), _ptr(vs), ks.shape[0], _ptr(kd), _ptr(vd),
                                     kd.shape[0], _ptr(mp), mp.shape[0], bs, hkv, d)
    return kd, vd, int(bad)


def _decode_args(q, k_cache, v_cache, block_tables, context_lens):
    q = _u16(q)
    kc, vc = _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, hq, d = q.shape
    nb, bs, hkv, d2 = kc.shape
    assert d2 == d and vc.shape == kc.shape and cl.shape == (B,)
    assert bt.ndim == 2 and bt.shape[0] == B
    if B:
        need = -(-int(cl.max()) // bs) if cl.size else 0
        assert need <= bt.shape[1], "context longer than the block table row"
        assert int(cl.min()) >= 0
    return q, kc, vc, bt, cl, B, hq, hkv, d, bs


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 dtype: str) -> np.ndarray:
    """fp64 [B][Hq][D] attention output through the block table."""
    q, kc, vc, bt, cl, B, hq, hkv, d, bs = _decode_args(q, k_cache, v_cache, block_tables,
                                                       context_lens)
    out = np.zeros((B, hq, d), dtype=np.float64)
    rc = _load().oracle_paged_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl),
                                     float(scale), B, hq, hkv, d, bs, bt.shape[1],
                                     _DTYPES[dtype], _ptr(out))
    if rc != 0:
        raise ValueError("oracle_paged_decode: bad shape")
    return out


def paged_decode_partitions(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                            dtype: str, partition_size: int, max_parts: int):
    """Per-partition (out [B][Hq][S][D], max [B][Hq][S], sum [B][Hq][S]) in fp64.

    Entries of partitions at or past the context end stay NaN.
    """
    q, kc, vc, bt, cl, B, hq, hkv, d, bs = _decode_args(q, k_cache, v_cache, block_tables,
                                                       context_lens)
    po = np.full((B, hq, max_parts, d), np.nan)
    pm = np.full((B, hq, max_parts), np.nan)
    ps = np.full((B, hq, max_parts), np.nan)
    rc = _load().oracle_paged_decode_partitions(
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), float(scale), B, hq, hkv, d, bs,
        bt.shape[1], _DTYPES[dtype], int(partition_size), int(max_parts), _ptr(po),
        _ptr(pm), _ptr(ps))
    if rc != 0:
        raise ValueError("oracle_paged_decode_partitions: bad arguments")
    return po, pm, ps


def paged_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale: float,
                  dtype: str) -> np.ndarray:
    """fp64 causal attention of every new token of every sequence
    ([total_tokens][Hq][D]); new tokens are the last C_b of each context."""
    q = _u16(q)
    kc, vc = _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    B = cl.shape[0]
    total, hq, d = q.shape
    nb, bs, hkv, d2 = kc.shape
    assert d2 == d and qs.shape == (B + 1,) and int(qs[-1]) == total and bt.shape[0] == B
    assert np.all(np.diff(qs) <= cl) and np.all(np.diff(qs) >= 0)
    out = np.zeros((total, hq, d), dtype=np.float64)
    rc = _load().oracle_paged_prefill(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), _ptr(qs),
                                      float(scale), B, hq, hkv, d, bs, bt.shape[1],
                                      _DTYPES[dtype], _ptr(out))
    if rc != 0:
        raise ValueError("oracle_paged_prefill: bad shape")
    return out


def lse_merge(part_out, part_max, part_sum, context_lens, partition_size: int) -> np.ndarray:
    po = np.ascontiguousarray(part_out, dtype=np.float64)
    pm = np.ascontiguousarray(part_max, dtype=np.float64)
    ps = np.ascontiguousarray(part_sum, dtype=np.float64)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, hq, S, d = po.shape
    out = np.zeros((B, hq, d), dtype=np.float64)
    rc = _load().oracle_lse_merge(_ptr(po), _ptr(pm), _ptr(ps), _ptr(cl), B, hq, d,
                                  int(partition_size), S, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_lse_merge: bad arguments")
    return out


def contiguous_decode(q, k_seq, v_seq, seq_start, context_lens, scale: float,
                      dtype: str) -> np.ndarray:
    """fp64 attention over contiguous per-sequence K/V ([sum L][Hkv][D] bits)."""
    q = _u16(q)
    ks, vs = _u16(k_seq), _u16(v_seq)
    st = np.ascontiguousarray(seq_start, dtype=np.int64)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, hq, d = q.shape
    hkv = ks.shape[1]
    out = np.zeros((B, hq, d), dtype=np.float64)
    rc = _load().oracle_contiguous_decode(_ptr(q), _ptr(ks), _ptr(vs), _ptr(st), _ptr(cl),
                                          float(scale), B, hq, hkv, d, _DTYPES[dtype],
                                          _ptr(out))
    if rc != 0:
        raise ValueError("oracle_contiguous_decode: bad shape")
    return out
