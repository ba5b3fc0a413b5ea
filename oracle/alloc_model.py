"""KV-cache memory accounting from the pages (oracle side, test infrastructure).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Plain arithmetic, each function citing the passage it restates:

* ``kv_cache_bytes`` -- youngju.dev "vLLM inference optimization" post,
  section "KV Cache問題の理解" (why the KV cache is a problem): total bytes =
  2 (K and V) x layers x heads x head_dim x sequence length x batch x bytes
  per element.  The same post prints 5.2 GB / 166 GB for its 70B example;
  those figures do not follow from its own formula (with 64 heads it gives
  10 GiB, with 8 KV heads 1.25 GiB), so only the formula is modelled.
* ``kv_bytes_per_token`` -- ta-paperlens "LLM serving from scratch",
  section "なぜ「まとめる」とタダで得をするのか": 2 x 32 layers x 8 KV heads x
  128 dims x 2 bytes = 131,072 bytes per token.
* ``contiguous_reservation`` -- youngju.dev post, section "従来方式の無駄"
  (waste of the conventional scheme): every request reserves max_len slots
  up front; waste = 1 - used / reserved.
* ``paged_usage`` -- same post, section "PagedAttention": blocks are taken on
  demand, so a request of n tokens holds ceil(n / block_size) blocks and
  wastes only the unfilled tail of its last block (ta-paperlens page: the only
  waste left is the remainder inside a block).
* ``pool_occupancy`` -- same post's page-table diagram: physical blocks named
  in any table are in use, the rest are free.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Sequence


def kv_cache_bytes(num_layers: int, num_heads: int, head_dim: int, seq_len: int,
                   batch_size: int, dtype_bytes: int = 2) -> int:
    return 2 * num_layers * num_heads * head_dim * seq_len * batch_size * dtype_bytes


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int,
                       dtype_bytes: int = 2) -> int:
    return kv_cache_bytes(num_layers, num_kv_heads, head_dim, 1, 1, dtype_bytes)


def contiguous_reservation(used_lens: Sequence[int], max_len: int) -> Dict[str, float]:
    reserved = len(used_lens) * max_len
    used = sum(int(n) for n in used_lens)
    if any(n > max_len for n in used_lens):
        raise ValueError("a request is longer than its reservation")
    return {"reserved": reserved, "used": used,
            "waste": (1.0 - used / reserved) if reserved else 0.0}


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def paged_usage(used_lens: Sequence[int], block_size: int) -> Dict[str, object]:
    blocks = [_ceil_div(int(n), block_size) for n in used_lens]
    slots = sum(blocks) * block_size
    used = sum(int(n) for n in used_lens)
    tail_waste = [b * block_size - int(n) for b, n in zip(blocks, used_lens)]
    return {"blocks": sum(blocks), "blocks_per_request": blocks, "slots": slots,
            "used": used, "waste": (1.0 - used / slots) if slots else 0.0,
            "tail_waste": tail_waste}


def pool_occupancy(num_blocks: int, tables: Iterable[Sequence[int]]) -> Dict[str, List[int]]:
    used = sorted({int(p) for t in tables for p in t})
    if any(p < 0 or p >= num_blocks for p in used):
        raise ValueError("table names a block outside the pool")
    free = [p for p in range(num_blocks) if p not in set(used)]
    return {"used": used, "free": free}
