"""Python binding of libpa.so (the C ABI declared in include/pa.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  torch provides device memory and the current
stream.  There is no fallback: if libpa.so is missing or cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional, Tuple

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "pa.h")

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(5)
PA_FP16, PA_BF16 = 0, 1
PA_DEVERR_WAIT_TIMEOUT, PA_DEVERR_BAD_CONTEXT, PA_DEVERR_BAD_SLOT = 1, 2, 4
DEFAULT_PARTITION = 512

_DTYPE_CODES = {torch.float16: PA_FP16, torch.bfloat16: PA_BF16}


class PaShape(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class PaError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status}){detail}")


_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libpa.so (raises if it is absent: build it with
    ``python -m paged_kv_cache_226_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libpa.so not found at {p}; build it with "
                              "`python -m paged_kv_cache_226_gb300.build`")
        lib = ctypes.CDLL(p)
        V, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        S = ctypes.POINTER(PaShape)
        lib.pa_reshape_and_cache.argtypes = [V, V, V, V, V, I64, S, V]
        lib.pa_decode.argtypes = [V, V, V, V, V, F, V, S, V]
        lib.pa_split_workspace_size.argtypes = [S, I32, I32]
        lib.pa_split_workspace_size.restype = ctypes.c_size_t
        lib.pa_decode_split.argtypes = [V, V, V, V, V, F, I32, I32, V, V, V, S, V]
        lib.pa_reduce.argtypes = [V, V, V, V, I32, I32, V, S, V]
        lib.pa_reshape_and_cache_fp8.argtypes = [V, V, V, V, V, I64, F, F, S, V]
        lib.pa_decode_fp8.argtypes = [V, V, V, V, V, F, F, F, V, S, V]
        lib.pa_decode_split_fp8.argtypes = [V, V, V, V, V, F, F, F, I32, I32, V, V, V, S, V]
        lib.pa_decode_step_fp8.argtypes = [V, V, V, V, V, V, V, V, F, F, F, I32, I32, V, V, V, V,
                                           V, S, V]
        for fn in ("pa_reshape_and_cache_fp8", "pa_decode_fp8", "pa_decode_split_fp8",
                   "pa_decode_step_fp8"):
            getattr(lib, fn).restype = ctypes.c_int
        lib.pa_balanced_workspace_size.argtypes = [S]
        lib.pa_balanced_workspace_size.restype = ctypes.c_size_t
        lib.pa_decode_step_balanced.argtypes = [V, V, V, V, V, V, V, V, F, V, ctypes.c_size_t, V,
                                                S, V]
        lib.pa_decode_step_balanced_fp8.argtypes = [V, V, V, V, V, V, V, V, F, F, F, V,
                                                    ctypes.c_size_t, V, S, V]
        lib.pa_decode_step_balanced.restype = ctypes.c_int
        lib.pa_decode_step_balanced_fp8.restype = ctypes.c_int
        lib.pa_copy_async.argtypes = [V, V, ctypes.c_size_t, V]
        lib.pa_copy_async.restype = ctypes.c_int
        for fn in (lib.pa_prefill, lib.pa_prefill_mma):
            fn.argtypes = [V, V, V, V, V, V, F, I32, V, S, V]
            fn.restype = ctypes.c_int
        lib.pa_prefill_workspace_size.argtypes = [S, I32]
        lib.pa_prefill_workspace_size.restype = ctypes.c_size_t
        lib.pa_prefill_ws.argtypes = [V, V, V, V, V, V, F, I32, V, ctypes.c_size_t, V, S, V]
        lib.pa_prefill_ws.restype = ctypes.c_int
        lib.pa_copy_blocks.argtypes = [V, V, I64, V, V, I64, V, I64, S, V]
        lib.pa_copy_blocks.restype = ctypes.c_int
        lib.pa_decode_step.argtypes = [V, V, V, V, V, V, V, V, F, I32, I32, V, V, V, V, V, S, V]
        lib.pa_decode_step.restype = ctypes.c_int
        lib.pa_decode_static_workspace.argtypes = [V, V, V, V, V, F, I32, I32, V, S, V]
        lib.pa_decode_static_workspace.restype = ctypes.c_int
        lib.pa_status_string.argtypes = [ctypes.c_int]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_last_cuda_error.argtypes = []
        lib.pa_read_device_errors.argtypes = [ctypes.POINTER(I32), V]
        for fn in ("pa_reshape_and_cache", "pa_decode", "pa_decode_split", "pa_reduce",
                   "pa_last_cuda_error", "pa_read_device_errors"):
            getattr(lib, fn).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def header_symbols(header: str = HEADER_PATH):
    """Names of the functions include/pa.h declares."""
    with open(header) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != PA_OK:
        detail = ""
        if status == PA_ERR_CUDA:
            detail = f", cudaError {load().pa_last_cuda_error()}"
        raise PaError(fn, status, detail)


def _stream_handle(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype=None, device=None, host_ok: bool = False):
    """Checks a tensor argument; with ``host_ok`` a pinned host tensor is
    accepted too (the kernel reaches it through unified addressing)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    pinned_host = host_ok and not t.is_cuda and t.is_pinned()
    if not t.is_cuda and not pinned_host:
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.is_cuda and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def make_shape(num_seqs: int, num_q_heads: int, k_cache: torch.Tensor,
               max_blocks_per_seq: int) -> PaShape:
    nb, bs, hkv, d = k_cache.shape
    if k_cache.dtype not in _DTYPE_CODES:
        raise TypeError(f"cache dtype must be float16 or bfloat16, got {k_cache.dtype}")
    return PaShape(num_seqs=num_seqs, num_q_heads=num_q_heads, num_kv_heads=hkv, head_dim=d,
                   block_size=bs, max_blocks_per_seq=max_blocks_per_seq, num_blocks=nb,
                   dtype=_DTYPE_CODES[k_cache.dtype], reserved=0)


def reshape_and_cache(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                      k_cache: torch.Tensor, v_cache: torch.Tensor) -> None:
    """Write each new token's K/V ([T][Hkv][D]) into slot_mapping's cache slots."""
    lib = load()
    dev = k_cache.device
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, k_cache.dtype, dev)
    for t, n in ((k, "k"), (v, "v")):
        _need(t, n, k_cache.dtype, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    T = slot_mapping.shape[0]
    if k.shape != (T, k_cache.shape[2], k_cache.shape[3]) or v.shape != k.shape:
        raise ValueError("k and v must be [num_tokens][num_kv_heads][head_dim]")
    shp = make_shape(0, k_cache.shape[2], k_cache, 1)
    _check("pa_reshape_and_cache",
           lib.pa_reshape_and_cache(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_cache),
                                    _ptr(v_cache), T, ctypes.byref(shp), _stream_handle(dev)))


def _decode_common(q, k_cache, v_cache, block_tables, context_lens, host_ok: bool = False):
    dev = k_cache.device
    _need(q, "q", k_cache.dtype, dev, host_ok)
    _need(k_cache, "k_cache", None, dev)
    _need(v_cache, "v_cache", k_cache.dtype, dev)
    _need(block_tables, "block_tables", torch.int32, dev, host_ok)
    _need(context_lens, "context_lens", torch.int32, dev, host_ok)
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [num_blocks][block_size][num_kv_heads][head_dim]")
    B, hq, d = q.shape
    if d != k_cache.shape[3] or block_tables.dim() != 2 or block_tables.shape[0] != B \
            or context_lens.shape != (B,):
        raise ValueError("inconsistent q / block_tables / context_lens shapes")
    return make_shape(B, hq, k_cache, block_tables.shape[1]), dev


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
           out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Single-pass paged decode attention (one CTA per sequence and KV head)."""
    lib = load()
    shp, dev = _decode_common(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, dev)
    _check("pa_decode", lib.pa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                      _ptr(context_lens), float(scale), _ptr(out),
                                      ctypes.byref(shp), _stream_handle(dev)))
    return out


def num_partitions(max_context_len: int, partition_size: int = DEFAULT_PARTITION) -> int:
    return max(1, -(-int(max_context_len) // int(partition_size)))


def split_workspace(q: torch.Tensor, max_num_partitions: int, device=None
                    ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Allocate (tmp_out, max_logits, exp_sums) for the split path (on
    ``device``, default q's)."""
    B, hq, d = q.shape
    device = q.device if device is None else device
    tmp = torch.empty((B, hq, max_num_partitions, d), dtype=torch.float32, device=device)
    ml = torch.empty((B, hq, max_num_partitions), dtype=torch.float32, device=device)
    es = torch.empty((B, hq, max_num_partitions), dtype=torch.float32, device=device)
    return tmp, ml, es


def workspace_size(num_seqs, num_q_heads, k_cache, max_blocks_per_seq, max_context_len,
                   partition_size=DEFAULT_PARTITION) -> int:
    shp = make_shape(num_seqs, num_q_heads, k_cache, max_blocks_per_seq)
    return int(load().pa_split_workspace_size(ctypes.byref(shp), int(max_context_len),
                                              int(partition_size)))


def decode_split(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 partition_size: int, max_num_partitions: int, tmp_out=None, max_logits=None,
                 exp_sums=None):
    """Per-partition outputs (tmp_out, max_logits, exp_sums) of the context split."""
    lib = load()
    shp, dev = _decode_common(q, k_cache, v_cache, block_tables, context_lens)
    if tmp_out is None:
        tmp_out, max_logits, exp_sums = split_workspace(q, max_num_partitions)
    for t, n in ((tmp_out, "tmp_out"), (max_logits, "max_logits"), (exp_sums, "exp_sums")):
        _need(t, n, torch.float32, dev)
    B, hq, d = q.shape
    if tmp_out.numel() < B * hq * max_num_partitions * d or \
            max_logits.numel() < B * hq * max_num_partitions or \
            exp_sums.numel() < B * hq * max_num_partitions:
        raise PaError("pa_decode_split", PA_ERR_WORKSPACE)
    _check("pa_decode_split",
           lib.pa_decode_split(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               _ptr(context_lens), float(scale), int(partition_size),
                               int(max_num_partitions), _ptr(tmp_out), _ptr(max_logits),
                               _ptr(exp_sums), ctypes.byref(shp), _stream_handle(dev)))
    return tmp_out, max_logits, exp_sums


def reduce(tmp_out, max_logits, exp_sums, context_lens, partition_size: int,
           k_cache: torch.Tensor, max_blocks_per_seq: int, out: torch.Tensor) -> torch.Tensor:
    """Log-sum-exp merge of decode_split's partitions into out [B][Hq][D]."""
    lib = load()
    dev = out.device
    _need(out, "out", out.dtype, dev)
    for t, n in ((tmp_out, "tmp_out"), (max_logits, "max_logits"), (exp_sums, "exp_sums")):
        _need(t, n, torch.float32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    B, hq, d = out.shape
    S = tmp_out.shape[2]
    if k_cache.dtype == torch.uint8:                     # FP8 cache: out keeps its own type
        shp = _fp8_shape(B, hq, k_cache, max_blocks_per_seq, out.dtype)
    else:
        if out.dtype != k_cache.dtype:
            raise TypeError("out must have the cache's dtype")
        shp = make_shape(B, hq, k_cache, max_blocks_per_seq)
    _check("pa_reduce", lib.pa_reduce(_ptr(tmp_out), _ptr(max_logits), _ptr(exp_sums),
                                      _ptr(context_lens), int(partition_size), int(S), _ptr(out),
                                      ctypes.byref(shp), _stream_handle(dev)))
    return out


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                    max_context_len: int, out: Optional[torch.Tensor] = None,
                    mode: str = "auto", partition_size: int = DEFAULT_PARTITION,
                    workspace=None) -> torch.Tensor:
    """Decode attention through the single-pass or the split + merge path.

    ``mode="auto"`` splits when there are too few (sequence, KV head) pairs to
    fill the GPU evenly or when contexts are long; ``max_context_len`` is the
    host-known bound on ``context_lens`` (it sizes the split grid).
    """
    if out is None:
        out = torch.empty_like(q)
    if mode == "auto":
        mode = choose_mode(q.shape[0], k_cache.shape[2], max_context_len, partition_size,
                           q.device)
    if mode == "single":
        return decode(q, k_cache, v_cache, block_tables, context_lens, scale, out)
    if mode != "split":
        raise ValueError(f"unknown mode {mode!r}")
    S = num_partitions(max_context_len, partition_size)
    if workspace is None:
        workspace = split_workspace(q, S)
    tmp, ml, es = workspace
    decode_split(q, k_cache, v_cache, block_tables, context_lens, scale, partition_size, S,
                 tmp, ml, es)
    return reduce(tmp, ml, es, context_lens, partition_size, k_cache, block_tables.shape[1], out)


def copy_blocks(k_src: torch.Tensor, v_src: torch.Tensor, k_dst: torch.Tensor,
                v_dst: torch.Tensor, block_mapping: torch.Tensor,
                device: Optional[torch.device] = None) -> None:
    """Copy whole blocks ``(src, dst)`` of ``block_mapping`` (int64 [P][2], on
    the device) from the src pools to the dst pools (pa_copy_blocks): the same
    pool for copy-on-write, a pinned host pool on one side for swapping."""
    lib = load()
    dev = device or block_mapping.device
    _need(block_mapping, "block_mapping", torch.int64, dev)
    for t, n in ((k_src, "k_src"), (v_src, "v_src"), (k_dst, "k_dst"), (v_dst, "v_dst")):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{n} must be a CUDA tensor or pinned host memory")
        if not t.is_contiguous() or t.dtype != k_src.dtype or t.dim() != 4:
            raise ValueError(f"{n} must be a contiguous 4-D pool of {k_src.dtype}")
        if t.shape[1:] != k_src.shape[1:]:
            raise ValueError("pools differ in block shape")
    if v_src.shape != k_src.shape or v_dst.shape != k_dst.shape:
        raise ValueError("K and V pools differ in shape")
    mp = block_mapping.reshape(-1, 2)
    shp = make_shape(0, k_src.shape[2], k_src, 1)
    with torch.cuda.device(dev):
        _check("pa_copy_blocks",
               lib.pa_copy_blocks(_ptr(k_src), _ptr(v_src), k_src.shape[0], _ptr(k_dst),
                                  _ptr(v_dst), k_dst.shape[0], _ptr(mp), mp.shape[0],
                                  ctypes.byref(shp), _stream_handle(dev)))


# ---- FP8 (E4M3) KV cache ---------------------------------------------------
#
# The cache tensors are torch.uint8 [num_blocks][block_size][Hkv][D] holding
# E4M3 codes; element value = e4m3(code) * scale, one scale for K and one for V.
# q, the new tokens and the output keep their fp16 / bf16 type.

def _fp8_shape(num_seqs, num_q_heads, k_cache: torch.Tensor, max_blocks_per_seq, dtype):
    nb, bs, hkv, d = k_cache.shape
    if k_cache.dtype != torch.uint8:
        raise TypeError("an FP8 cache is a torch.uint8 tensor of E4M3 codes")
    return PaShape(num_seqs=num_seqs, num_q_heads=num_q_heads, num_kv_heads=hkv, head_dim=d,
                   block_size=bs, max_blocks_per_seq=max_blocks_per_seq, num_blocks=nb,
                   dtype=_DTYPE_CODES[dtype], reserved=0)


def reshape_and_cache_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale: float,
                          v_scale: float) -> None:
    """Quantise each new token's K/V to E4M3 (x / scale) into its cache slot."""
    lib = load()
    dev = k_cache.device
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, torch.uint8, dev)
    for t, n in ((k, "k"), (v, "v")):
        _need(t, n, k.dtype, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    T = slot_mapping.shape[0]
    if k.shape != (T, k_cache.shape[2], k_cache.shape[3]) or v.shape != k.shape:
        raise ValueError("k and v must be [num_tokens][num_kv_heads][head_dim]")
    shp = _fp8_shape(0, k_cache.shape[2], k_cache, 1, k.dtype)
    _check("pa_reshape_and_cache_fp8",
           lib.pa_reshape_and_cache_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_cache),
                                        _ptr(v_cache), T, float(k_scale), float(v_scale),
                                        ctypes.byref(shp), _stream_handle(dev)))


def _fp8_common(q, k_cache, v_cache, block_tables, context_lens, host_ok: bool = False):
    dev = k_cache.device
    _need(q, "q", q.dtype, dev, host_ok)
    _need(k_cache, "k_cache", torch.uint8, dev)
    _need(v_cache, "v_cache", torch.uint8, dev)
    _need(block_tables, "block_tables", torch.int32, dev, host_ok)
    _need(context_lens, "context_lens", torch.int32, dev, host_ok)
    if q.dtype not in _DTYPE_CODES:
        raise TypeError("q must be float16 or bfloat16")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [num_blocks][block_size][num_kv_heads][head_dim]")
    B, hq, d = q.shape
    if d != k_cache.shape[3] or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("inconsistent q / block_tables / context_lens shapes")
    return _fp8_shape(B, hq, k_cache, block_tables.shape[1], q.dtype), dev


def decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale: float, k_scale: float,
               v_scale: float, out=None) -> torch.Tensor:
    """Single-pass paged decode over an E4M3 cache."""
    lib = load()
    shp, dev = _fp8_common(q, k_cache, v_cache, block_tables, context_lens)
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", q.dtype, dev)
    _check("pa_decode_fp8",
           lib.pa_decode_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                             _ptr(context_lens), float(scale), float(k_scale), float(v_scale),
                             _ptr(out), ctypes.byref(shp), _stream_handle(dev)))
    return out


def decode_split_fp8(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                     k_scale: float, v_scale: float, partition_size: int,
                     max_num_partitions: int, workspace=None):
    """Per-partition outputs over an E4M3 cache (merge them with ``reduce``)."""
    lib = load()
    shp, dev = _fp8_common(q, k_cache, v_cache, block_tables, context_lens)
    tmp, ml, es = workspace if workspace is not None else split_workspace(q, max_num_partitions)
    _check("pa_decode_split_fp8",
           lib.pa_decode_split_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                   _ptr(context_lens), float(scale), float(k_scale),
                                   float(v_scale), int(partition_size), int(max_num_partitions),
                                   _ptr(tmp), _ptr(ml), _ptr(es), ctypes.byref(shp),
                                   _stream_handle(dev)))
    return tmp, ml, es


def decode_step_fp8(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                    context_lens, scale: float, k_scale: float, v_scale: float,
                    max_context_len: int, out=None, partition_size: int = DEFAULT_PARTITION,
                    workspace=None) -> torch.Tensor:
    """Fused decode layer-step over an E4M3 cache (pa_decode_step_fp8)."""
    lib = load()
    shp, dev = _fp8_common(q, k_cache, v_cache, block_tables, context_lens)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, q.dtype, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    out = torch.empty_like(q) if out is None else out
    S = num_partitions(max_context_len, partition_size)
    if workspace is None:
        workspace = step_workspace(q, k_cache.shape[2], S)
    tmp, ml, es, counters = workspace
    _check("pa_decode_step_fp8",
           lib.pa_decode_step_fp8(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                  _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                  _ptr(context_lens), float(scale), float(k_scale),
                                  float(v_scale), int(partition_size), int(S), _ptr(tmp),
                                  _ptr(ml), _ptr(es), _ptr(counters), _ptr(out),
                                  ctypes.byref(shp), _stream_handle(dev)))
    return out


def step_workspace(q: torch.Tensor, num_kv_heads: int, max_num_partitions: int, device=None):
    """(tmp_out, max_logits, exp_sums, counters) for ``decode_step`` (on
    ``device``, default q's); the counters start at zero and every step leaves
    them at zero."""
    device = q.device if device is None else device
    tmp, ml, es = split_workspace(q, max_num_partitions, device)
    counters = torch.zeros((q.shape[0], num_kv_heads), dtype=torch.int32, device=device)
    return tmp, ml, es, counters


def decode_step(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables, context_lens,
                scale: float, max_context_len: int, out: Optional[torch.Tensor] = None,
                partition_size: int = DEFAULT_PARTITION, workspace=None) -> torch.Tensor:
    """One fused decode layer-step (pa_decode_step): write each sequence's new
    token into the cache and attend, merging partitions in the same launch."""
    lib = load()
    shp, dev = _decode_common(q, k_cache, v_cache, block_tables, context_lens)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, k_cache.dtype, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    if k_new.shape != (q.shape[0], k_cache.shape[2], k_cache.shape[3]) or \
            v_new.shape != k_new.shape or slot_mapping.shape != (q.shape[0],):
        raise ValueError("k_new / v_new must be [num_seqs][num_kv_heads][head_dim], "
                         "slot_mapping [num_seqs]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, dev)
    S = num_partitions(max_context_len, partition_size)
    if workspace is None:
        workspace = step_workspace(q, k_cache.shape[2], S)
    tmp, ml, es, counters = workspace
    _need(counters, "counters", torch.int32, dev)
    _check("pa_decode_step",
           lib.pa_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                              _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                              _ptr(context_lens), float(scale), int(partition_size), int(S),
                              _ptr(tmp), _ptr(ml), _ptr(es), _ptr(counters), _ptr(out),
                              ctypes.byref(shp), _stream_handle(dev)))
    return out


def balanced_workspace(q: torch.Tensor, k_cache: torch.Tensor,
                       block_tables: torch.Tensor) -> torch.Tensor:
    """Zeroed workspace for ``decode_step_balanced`` (reusable across steps)."""
    if k_cache.dtype == torch.uint8:
        shp = _fp8_shape(q.shape[0], q.shape[1], k_cache, block_tables.shape[1], q.dtype)
    else:
        shp = make_shape(q.shape[0], q.shape[1], k_cache, block_tables.shape[1])
    with torch.cuda.device(q.device):
        n = int(load().pa_balanced_workspace_size(ctypes.byref(shp)))
    if n == 0:
        raise PaError("pa_balanced_workspace_size", PA_ERR_INVALID_ARG)
    return torch.zeros(n, dtype=torch.uint8, device=q.device)


def decode_step_balanced(q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                         context_lens, scale: float, out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, k_scale: float = None,
                         v_scale: float = None) -> torch.Tensor:
    """Fused decode layer-step with the work balanced over one wave of CTAs
    (pa_decode_step_balanced; pa_decode_step_balanced_fp8 for a uint8 E4M3
    cache with k_scale / v_scale)."""
    lib = load()
    fp8 = k_cache.dtype == torch.uint8
    if fp8:
        shp, dev = _fp8_common(q, k_cache, v_cache, block_tables, context_lens)
    else:
        shp, dev = _decode_common(q, k_cache, v_cache, block_tables, context_lens)
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, n, q.dtype, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    if k_new.shape != (q.shape[0], k_cache.shape[2], k_cache.shape[3]) or \
            v_new.shape != k_new.shape or slot_mapping.shape != (q.shape[0],):
        raise ValueError("k_new / v_new must be [num_seqs][num_kv_heads][head_dim], "
                         "slot_mapping [num_seqs]")
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", q.dtype, dev)
    if workspace is None:
        workspace = balanced_workspace(q, k_cache, block_tables)
    _need(workspace, "workspace", torch.uint8, dev)
    args = [_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
            _ptr(block_tables), _ptr(context_lens), ctypes.c_float(scale)]
    if fp8:
        args += [ctypes.c_float(k_scale), ctypes.c_float(v_scale)]
    args += [_ptr(workspace), ctypes.c_size_t(workspace.numel()), _ptr(out), ctypes.byref(shp),
             _stream_handle(dev)]
    fn = lib.pa_decode_step_balanced_fp8 if fp8 else lib.pa_decode_step_balanced
    _check("pa_decode_step_balanced" + ("_fp8" if fp8 else ""), fn(*args))
    return out


def prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale: float,
            max_query_len: int, out: Optional[torch.Tensor] = None,
            kernel: str = "auto", schedule: bool = True,
            workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Chunked-prefill attention (pa_prefill): the last C_b tokens of each
    sequence attend causally over its cache; q, out [total_tokens][Hq][D].
    kernel "mma" forces the mma.sync kernel (pa_prefill_mma).  schedule: order
    the tcgen05 kernel's work longest first (pa_prefill_ws, with ``workspace``
    or a fresh one of pa_prefill_workspace_size bytes); False: pa_prefill."""
    lib = load()
    dev = k_cache.device
    _need(q, "q", k_cache.dtype, dev)
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n, k_cache.dtype, dev)
    _need(block_tables, "block_tables", torch.int32, dev)
    _need(context_lens, "context_lens", torch.int32, dev)
    _need(query_start, "query_start", torch.int32, dev)
    B = context_lens.shape[0]
    if query_start.shape != (B + 1,) or block_tables.shape[0] != B or q.dim() != 3:
        raise ValueError("query_start must be [num_seqs + 1], q [total_tokens][Hq][D]")
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", q.dtype, dev)
    shp = make_shape(B, q.shape[1], k_cache, block_tables.shape[1])
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
            _ptr(query_start), float(scale), int(max_query_len))
    if kernel == "mma" or not schedule:
        fn = lib.pa_prefill_mma if kernel == "mma" else lib.pa_prefill
        _check("pa_prefill", fn(*args, _ptr(out), ctypes.byref(shp), _stream_handle(dev)))
        return out
    if workspace is None:
        n = prefill_workspace_size(shp, max_query_len)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    _check("pa_prefill_ws", lib.pa_prefill_ws(*args, _ptr(workspace), workspace.numel(), _ptr(out),
                                              ctypes.byref(shp), _stream_handle(dev)))
    return out


def prefill_workspace_size(shp, max_query_len: int) -> int:
    """Bytes of the work-ordering workspace pa_prefill_ws needs (0: none)."""
    return int(load().pa_prefill_workspace_size(ctypes.byref(shp), int(max_query_len)))


STATIC_WORKSPACE_BYTES = 32 << 20


def decode_static_workspace(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                            max_context_len: int, out: Optional[torch.Tensor] = None,
                            partition_size: int = DEFAULT_PARTITION) -> torch.Tensor:
    """Split decode + merge using the library's own fixed device buffer for
    the partition workspace (pa_decode_static_workspace): for callers that
    must not allocate device memory, e.g. inside a framework that owns the
    device memory pool.  ``out`` must be given by such callers (allocating it
    here is a convenience for tests).  Calls that overlap on the GPU share
    the buffer and race; keep them ordered."""
    lib = load()
    shp, dev = _decode_common(q, k_cache, v_cache, block_tables, context_lens)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, dev)
    S = num_partitions(max_context_len, partition_size)
    _check("pa_decode_static_workspace",
           lib.pa_decode_static_workspace(_ptr(q), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(block_tables), _ptr(context_lens), float(scale),
                                          int(partition_size), int(S), _ptr(out),
                                          ctypes.byref(shp), _stream_handle(dev)))
    return out


CTAS_PER_SM = 6          # resident decode CTAs per SM in the shipped build


def choose_partition(num_seqs: int, num_kv_heads: int, max_context_len: int,
                     block_size: int = 16, device=None, context_lens=None) -> int:
    """Partition size for the split / fused paths.

    With at least half as many (sequence, KV head) pairs as resident CTA
    slots, the pairs alone give every slot work: 1024-token partitions then
    leave most contexts of a ragged batch in one partition (no merge) and
    the rest in few (measured on the fused step: shared-prefix batch 119 us
    against 133 us at 512 tokens, Llama-3-8B-shaped batch 60 us against 62).

    Fewer pairs (long contexts, small batches): the smallest multiple of 512
    that cuts the batch into at most 4.8 CTAs per SM, counting every
    context's ragged last piece (``context_lens``, host values; without them
    every context is taken at ``max_context_len``).  Fewer CTAs pay the
    per-partition start and merge fewer times, but below ~3 per SM too few
    stages are in flight to keep HBM busy; more than one wave of CTAs
    leaves a tail of late, long partitions.  Measured on the fused step
    (µs per layer-step, best partition, this rule's choice): 256 pairs of
    4096 tokens 91.8 at 2048 (2048; 1536 gives 94.3); 64 pairs of
    U[32768, 50000] 217.2 at 4352 (4096: 220.1; 3584 gives 230.3);
    32 x U[128, 4096] x 8 heads 54.9 at 1024 (1024; 2048 gives 67.4);
    40 x 4096 x 8 heads 108.3 at 2048 (2048; 1536 gives 115.5)."""
    if device is None and torch.cuda.is_available():
        device = torch.cuda.current_device()
    sms = torch.cuda.get_device_properties(device).multi_processor_count if device is not None \
        else 152
    slots = sms * CTAS_PER_SM
    pairs = max(1, num_seqs * num_kv_heads)
    if max_context_len <= 512:
        p = 512
    elif 2 * pairs >= slots:
        p = 1024
    else:
        if context_lens is None:
            lens = np.full(max(1, num_seqs), max_context_len, dtype=np.int64)
        else:
            if isinstance(context_lens, torch.Tensor):
                context_lens = context_lens.detach().cpu().numpy()
            lens = np.asarray(context_lens, dtype=np.int64).reshape(-1)
        limit = (24 * sms) // 5                        # 4.8 CTAs per SM

        def ctas(units: int) -> int:                   # CTAs at 512 * units tokens
            return num_kv_heads * int(np.sum(-(-lens // (512 * units))))

        # The count falls as the partition grows; one partition per context
        # (pairs < slots / 2 <= limit CTAs) always fits.
        lo, hi = 1, max(1, -(-max_context_len // 512))
        while lo < hi:
            mid = (lo + hi) // 2
            if ctas(mid) <= limit:
                hi = mid
            else:
                lo = mid + 1
        p = 512 * lo
    return max(block_size, p - p % block_size)


def choose_mode(num_seqs: int, num_kv_heads: int, max_context_len: int, partition_size: int,
                device=None) -> str:
    """Single pass when every (sequence, KV head) CTA is short, else split."""
    if max_context_len <= partition_size:
        return "single"
    return "split"


def read_device_errors(device: Optional[torch.device] = None) -> int:
    """Return and clear the library's device error word (PA_DEVERR_* bits)."""
    lib = load()
    dev = device or torch.device("cuda", torch.cuda.current_device())
    flags = ctypes.c_int32(0)
    with torch.cuda.device(dev):
        _check("pa_read_device_errors",
               lib.pa_read_device_errors(ctypes.byref(flags), _stream_handle(dev)))
    return int(flags.value)


def copy_async(dst: torch.Tensor, src: torch.Tensor) -> torch.Tensor:
    """dst <- src by a short kernel (pa_copy_async) on the current stream of
    whichever side is on the device; either may be pinned host memory."""
    if dst.numel() * dst.element_size() != src.numel() * src.element_size():
        raise ValueError("copy_async needs equal byte sizes")
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy_async needs contiguous tensors")
    for t in (dst, src):
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("copy_async: host tensors must be pinned")
    dev = dst.device if dst.is_cuda else src.device
    if not dev.type == "cuda":
        raise ValueError("copy_async: one side must be on a CUDA device")
    _check("pa_copy_async", load().pa_copy_async(_ptr(dst), _ptr(src),
                                                 ctypes.c_size_t(dst.numel() * dst.element_size()),
                                                 _stream_handle(dev)))
    return dst


class InputStaging:
    """A layer-step's host inputs (q, new K/V, slots, tables, lengths) as views
    into one pinned host buffer and one device buffer, each view 256-byte
    aligned, so a step uploads all of them with a single host-to-device copy.

    ``specs`` maps names to (shape, dtype); ``h[name]`` / ``d[name]`` are the
    host and device views.  Fill the host views, call ``upload()`` (on the
    current stream), and hand the device views to the kernels.
    """

    def __init__(self, specs: dict, device: torch.device):
        offsets, total = {}, 0
        for name, (shape, dtype) in specs.items():
            nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            offsets[name] = (total, nbytes, tuple(shape), dtype)
            total += (nbytes + 255) // 256 * 256
        self.nbytes = total
        self.host = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(total, dtype=torch.uint8, device=device)
        self.h, self.d = {}, {}
        for name, (off, nbytes, shape, dtype) in offsets.items():
            self.h[name] = self.host[off:off + nbytes].view(dtype).view(shape)
            self.d[name] = self.dev[off:off + nbytes].view(dtype).view(shape)

    def upload(self, engine: str = "kernel") -> None:
        """All inputs host -> device in one asynchronous copy on the current
        stream: by a short kernel reading the pinned buffer (``"kernel"``,
        pa_copy_async) or by the copy engine (``"dma"``)."""
        if engine == "kernel":
            copy_async(self.dev, self.host)
        else:
            self.dev.copy_(self.host, non_blocking=True)


class StepPlan:
    """One decode layer-step with its arguments marshalled once.

    Holds the C-ABI argument lists of the step for fixed tensors, so that
    each launch costs one ctypes call.  Modes: ``"fused"`` (the default: one
    pa_decode_step launch), ``"split"`` (reshape_and_cache, decode_split,
    reduce) and ``"single"`` (reshape_and_cache, decode).  The work goes to the caller's current stream at
    call time, which also makes a step capturable into a CUDA graph
    (``capture_graph``).  The tensors must stay alive and keep their shapes;
    their contents (new tokens, tables, lengths) may change between steps as
    long as ``context_lens`` stays within ``max_context_len``.

    In the fused mode q, k_new, v_new, slot_mapping, block_tables,
    context_lens and out may be pinned host tensors: the kernel reads the
    inputs and writes the output over the host link through unified
    addressing, with no copy launch (on a Grace-Blackwell node the fastest
    way to move a step's inputs in and its output out).  The caches and the
    workspace stay in device memory.

    ``partition_size=None`` takes ``choose_partition`` for the batch: with
    the lengths counted when ``context_lens`` is in host memory, else every
    context taken at ``max_context_len`` (no device read).  Any multiple of
    the block size gives the same result; the size only sets the speed.
    """

    def __init__(self, q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                 context_lens, scale: float, max_context_len: int, out=None,
                 mode: str = "auto", partition_size: Optional[int] = None, workspace=None,
                 k_scale: Optional[float] = None, v_scale: Optional[float] = None):
        self._lib = load()
        self.fp8 = k_cache.dtype == torch.uint8
        if mode == "auto":
            mode = "fused"
        if mode not in ("single", "split", "fused", "balanced"):
            raise ValueError(f"unknown mode {mode!r}")
        host_ok = mode == "fused"            # pinned host inputs / output allowed
        if self.fp8:
            if k_scale is None or v_scale is None:
                raise ValueError("an FP8 cache needs k_scale and v_scale")
            if mode not in ("fused", "balanced"):
                raise ValueError("StepPlan runs an FP8 cache through the fused steps only")
            shp, dev = _fp8_common(q, k_cache, v_cache, block_tables, context_lens, host_ok)
        else:
            shp, dev = _decode_common(q, k_cache, v_cache, block_tables, context_lens, host_ok)
        for t, n in ((k_new, "k_new"), (v_new, "v_new")):
            _need(t, n, q.dtype, dev, host_ok)
        _need(slot_mapping, "slot_mapping", torch.int64, dev, host_ok)
        T = slot_mapping.shape[0]
        if k_new.shape != (T, k_cache.shape[2], k_cache.shape[3]) or v_new.shape != k_new.shape:
            raise ValueError("k_new and v_new must be [num_tokens][num_kv_heads][head_dim]")
        self.device = dev
        self.out = torch.empty(q.shape, dtype=q.dtype, device=dev) if out is None else out
        _need(self.out, "out", q.dtype, dev, host_ok)
        if mode in ("fused", "balanced") and T != q.shape[0]:
            raise ValueError("the fused step takes exactly one new token per sequence")
        self.mode = mode
        if partition_size is None:
            partition_size = choose_partition(
                q.shape[0], k_cache.shape[2], max_context_len, k_cache.shape[1], dev,
                context_lens if context_lens.device.type == "cpu" else None)
        self.partition_size = int(partition_size)
        self.num_partitions = num_partitions(max_context_len, partition_size)
        self._shape = shp
        self._keep = [q, k_new, v_new, slot_mapping, k_cache, v_cache, block_tables,
                      context_lens, self.out]
        sref = ctypes.byref(self._shape)
        self._reshape_args = (_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache),
                              _ptr(v_cache), ctypes.c_int64(T), sref)
        if mode == "single":
            self._decode_args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                 _ptr(context_lens), ctypes.c_float(scale), _ptr(self.out), sref)
        elif mode == "balanced":
            if workspace is None:
                workspace = balanced_workspace(q, k_cache, block_tables)
            self.workspace = workspace
            self._keep.append(workspace)
            scales = (ctypes.c_float(k_scale), ctypes.c_float(v_scale)) if self.fp8 else ()
            self._step_args = (_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                               _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               _ptr(context_lens), ctypes.c_float(scale), *scales,
                               _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                               _ptr(self.out), sref)
        elif mode == "fused":
            if workspace is None:
                workspace = step_workspace(q, k_cache.shape[2], self.num_partitions, dev)
            tmp, ml, es, counters = workspace
            self.workspace = workspace
            self._keep += list(workspace)
            scales = (ctypes.c_float(k_scale), ctypes.c_float(v_scale)) if self.fp8 else ()
            self._step_args = (_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                               _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               _ptr(context_lens), ctypes.c_float(scale), *scales,
                               ctypes.c_int32(self.partition_size),
                               ctypes.c_int32(self.num_partitions), _ptr(tmp), _ptr(ml),
                               _ptr(es), _ptr(counters), _ptr(self.out), sref)
        else:
            if workspace is None:
                workspace = split_workspace(q, self.num_partitions)
            tmp, ml, es = workspace
            B, hq, d = q.shape
            if tmp.numel() < B * hq * self.num_partitions * d or \
                    ml.numel() < B * hq * self.num_partitions or \
                    es.numel() < B * hq * self.num_partitions:
                raise PaError("pa_decode_split", PA_ERR_WORKSPACE)
            self.workspace = workspace
            self._keep += list(workspace)
            S = ctypes.c_int32(self.num_partitions)
            P = ctypes.c_int32(self.partition_size)
            self._decode_args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                 _ptr(context_lens), ctypes.c_float(scale), P, S, _ptr(tmp),
                                 _ptr(ml), _ptr(es), sref)
            self._reduce_args = (_ptr(tmp), _ptr(ml), _ptr(es), _ptr(context_lens), P, S,
                                 _ptr(self.out), sref)
        self._graph = None

    def _stream(self):
        return ctypes.c_void_p(torch.cuda.current_stream(self.device).cuda_stream)

    def reshape_and_cache(self):
        if self.mode in ("fused", "balanced"):
            return                          # part of the fused step
        _check("pa_reshape_and_cache",
               self._lib.pa_reshape_and_cache(*self._reshape_args, self._stream()))

    def decode(self):
        if self.mode == "balanced":
            fn = self._lib.pa_decode_step_balanced_fp8 if self.fp8 else \
                self._lib.pa_decode_step_balanced
            _check("pa_decode_step_balanced", fn(*self._step_args, self._stream()))
        elif self.mode == "fused" and self.fp8:
            _check("pa_decode_step_fp8",
                   self._lib.pa_decode_step_fp8(*self._step_args, self._stream()))
        elif self.mode == "fused":
            _check("pa_decode_step", self._lib.pa_decode_step(*self._step_args, self._stream()))
        elif self.mode == "single":
            _check("pa_decode", self._lib.pa_decode(*self._decode_args, self._stream()))
        else:
            _check("pa_decode_split",
                   self._lib.pa_decode_split(*self._decode_args, self._stream()))

    def reduce(self):
        if self.mode == "split":
            _check("pa_reduce", self._lib.pa_reduce(*self._reduce_args, self._stream()))

    def __call__(self) -> torch.Tensor:
        self.reshape_and_cache()
        self.decode()
        self.reduce()
        return self.out

    def capture_graph(self, before=None, after=None) -> "torch.cuda.CUDAGraph":
        """Capture one step into a CUDA graph (replayed by ``replay``).

        ``before`` / ``after`` are called inside the capture around the step,
        e.g. ``InputStaging.upload`` and the copy of ``out`` to pinned host
        memory, so that a replay uploads, computes and reads back in one
        graph launch."""
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):                   # warm the lazy set-up outside capture,
            if before is not None:                   # with the same inputs the graph sees
                before()
            self()
            if after is not None:
                after()
        torch.cuda.current_stream(self.device).wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            if before is not None:
                before()
            self()
            if after is not None:
                after()
        self._graph = g
        return g

    def replay(self) -> torch.Tensor:
        if self._graph is None:
            self.capture_graph()
        self._graph.replay()
        return self.out
