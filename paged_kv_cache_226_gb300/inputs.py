"""Host-side block allocator and seeded synthetic workloads.

This module builds inputs only: it holds no attention arithmetic and no cache
write.  Tests feed the same tensors to the CUDA library and to the CPU
reference; the benchmark uses it to build its workload.

Allocator (youngju.dev "vLLM inference optimization" post, section
"PagedAttention", PagedAttentionManager):

* the pool's free list starts as a list of block ids and ``allocate`` pops
  from its end, failing with ``MemoryError("No free blocks")`` when empty;
  ``free`` puts a block back;
* ``append_token`` computes ``slot_in_block = count % block_size`` and takes a
  new block only when that is 0 and the request already holds tokens; the
  token goes to (last block, slot_in_block);
* blocks may be shared: a shared system-prompt block carries a reference
  count (same post, "Copy-on-Writeによるプレフィックス共有") and returns to the
  free list only when the count reaches zero.

Random physical placement: the initial free list is a seeded permutation of
the pool, so consecutive logical blocks land anywhere in the pool (the
techfeed summary of ngrok's "Serving models at scale with vLLM": blocks may be
scattered anywhere in GPU memory, the block table records where).  The
parameter ``placement="sequential"`` hands blocks out in pool order instead.

A slot number is ``physical_block * block_size + offset``.  The token written
in a decode step is the last one of its sequence: ``context_lens[b]`` counts
it, and ``slot_mapping[b]`` is the slot of position ``context_lens[b] - 1``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

# ----------------------------------------------------------------------------
# allocator
# ----------------------------------------------------------------------------


class BlockPool:
    """Free list of physical block ids with reference counts."""

    def __init__(self, num_blocks: int, block_size: int,
                 order: Optional[Sequence[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        ids = list(range(num_blocks)) if order is None else [int(i) for i in order]
        if sorted(ids) != list(range(num_blocks)):
            raise ValueError("order must be a permutation of the pool's block ids")
        self.free_blocks: List[int] = ids
        self.ref_count: List[int] = [0] * num_blocks

    @property
    def num_free(self) -> int:
        return len(self.free_blocks)

    def allocate(self) -> int:
        if not self.free_blocks:
            raise MemoryError("No free blocks")
        p = self.free_blocks.pop()
        self.ref_count[p] = 1
        return p

    def share(self, block: int) -> None:
        if self.ref_count[block] <= 0:
            raise ValueError(f"block {block} is not allocated")
        self.ref_count[block] += 1

    def free(self, block: int) -> None:
        if self.ref_count[block] <= 0:
            raise ValueError(f"block {block} is already free")
        self.ref_count[block] -= 1
        if self.ref_count[block] == 0:
            self.free_blocks.append(block)


class PagedKVAllocator:
    """Per-request block tables over a ``BlockPool``."""

    def __init__(self, pool: BlockPool):
        self.pool = pool
        self.block_size = pool.block_size
        self.page_tables: Dict[int, List[int]] = {}
        self.token_counts: Dict[int, int] = {}
        self.pending_copies: List[tuple] = []
        self.swapped: Dict[int, BlockPool] = {}

    def add_sequence(self, seq_id: int, shared_prefix: Sequence[int] = (),
                     prefix_tokens: int = 0) -> None:
        """Admit a request.  With ``shared_prefix`` it starts on those blocks
        (reference counts raised) holding ``prefix_tokens`` tokens; otherwise it
        gets one fresh block and zero tokens."""
        if seq_id in self.page_tables:
            raise ValueError(f"sequence {seq_id} exists")
        if shared_prefix:
            if not (len(shared_prefix) - 1) * self.block_size < prefix_tokens \
                    <= len(shared_prefix) * self.block_size:
                raise ValueError("prefix_tokens does not match the shared blocks")
            for p in shared_prefix:
                self.pool.share(p)
            self.page_tables[seq_id] = list(shared_prefix)
            self.token_counts[seq_id] = int(prefix_tokens)
        else:
            self.page_tables[seq_id] = [self.pool.allocate()]
            self.token_counts[seq_id] = 0

    def append_token(self, seq_id: int) -> int:
        """Reserve the slot of the request's next token and return it.

        If the token lands in a block that other requests still share, the
        request first gets a private copy of that block (copy-on-write); the
        (source, destination) pair is queued in ``pending_copies`` and must be
        copied on the device before the token is written."""
        table = self.page_tables[seq_id]
        count = self.token_counts[seq_id]
        slot_in_block = count % self.block_size
        if slot_in_block == 0 and count > 0:
            table.append(self.pool.allocate())
        elif self.pool.ref_count[table[-1]] > 1:
            shared = table[-1]
            private = self.pool.allocate()
            self.pending_copies.append((shared, private))
            self.pool.free(shared)
            table[-1] = private
        last_block = table[-1]
        self.token_counts[seq_id] = count + 1
        return last_block * self.block_size + slot_in_block

    def fork(self, parent_id: int, child_id: int) -> None:
        """The child shares every block of the parent (parallel sampling,
        beam search): reference counts rise, nothing is copied yet."""
        if child_id in self.page_tables:
            raise ValueError(f"sequence {child_id} exists")
        for p in self.page_tables[parent_id]:
            self.pool.share(p)
        self.page_tables[child_id] = list(self.page_tables[parent_id])
        self.token_counts[child_id] = self.token_counts[parent_id]

    def take_copies(self) -> List[tuple]:
        """Copy-on-write pairs queued since the last call."""
        out, self.pending_copies = self.pending_copies, []
        return out

    def swap_out(self, seq_id: int, host_pool: "BlockPool") -> List[tuple]:
        """Move a request's blocks to ``host_pool``: returns (device block,
        host block) pairs to copy; the device blocks return to the free list.
        Blocks still shared with other requests cannot be swapped out."""
        table = self.page_tables[seq_id]
        if any(self.pool.ref_count[p] > 1 for p in table):
            raise ValueError("cannot swap out shared blocks")
        pairs = []
        for i, p in enumerate(table):
            h = host_pool.allocate()
            pairs.append((p, h))
            self.pool.free(p)
            table[i] = h
        self.swapped[seq_id] = host_pool
        return pairs

    def swap_in(self, seq_id: int) -> List[tuple]:
        """Bring a swapped-out request back: returns (host block, device
        block) pairs to copy; the host blocks return to their free list."""
        host_pool = self.swapped.pop(seq_id)
        table = self.page_tables[seq_id]
        pairs = []
        for i, h in enumerate(table):
            p = self.pool.allocate()
            pairs.append((h, p))
            host_pool.free(h)
            table[i] = p
        return pairs

    def extend(self, seq_id: int, n: int) -> None:
        """Same effect as ``n`` calls of ``append_token`` (slots not returned)."""
        if n < 0:
            raise ValueError("n must be >= 0")
        count = self.token_counts[seq_id]
        table = self.page_tables[seq_id]
        held = len(table) * self.block_size
        need = max(count + n, 1)
        while held < need:
            table.append(self.pool.allocate())
            held += self.block_size
        self.token_counts[seq_id] = count + n

    def free_sequence(self, seq_id: int) -> None:
        for p in self.page_tables.pop(seq_id):
            self.pool.free(p)
        del self.token_counts[seq_id]

    def table_array(self, seq_ids: Sequence[int], max_blocks: Optional[int] = None,
                    pad: int = 0) -> np.ndarray:
        rows = [self.page_tables[s] for s in seq_ids]
        mb = max((len(r) for r in rows), default=0) if max_blocks is None else max_blocks
        out = np.full((len(rows), max(mb, 1)), pad, dtype=np.int32)
        for i, r in enumerate(rows):
            if len(r) > out.shape[1]:
                raise ValueError("max_blocks is smaller than a table")
            out[i, :len(r)] = r
        return out


# ----------------------------------------------------------------------------
# seeded values
# ----------------------------------------------------------------------------

_TORCH_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


def normal_tensor(rng: np.random.Generator, shape, dtype: str,
                  chunk_elems: int = 1 << 24) -> torch.Tensor:
    """N(0,1) float32 draws rounded to nearest-even 16-bit, drawn in chunks."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=_TORCH_DTYPES[dtype])
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if dtype == "fp16":
            out[s:e] = torch.from_numpy(x.astype(np.float16))
        else:
            out[s:e] = torch.from_numpy(x).to(torch.bfloat16)
    return out.view(*shape)


def normal_tensor_device(gen: torch.Generator, shape, dtype: str, device,
                         chunk_elems: int = 1 << 26) -> torch.Tensor:
    """N(0,1) float32 draws of a seeded device generator rounded to
    nearest-even 16-bit, made on the device (large pools for timing runs,
    where the host draw would take tens of seconds)."""
    out = torch.empty(tuple(shape), dtype=_TORCH_DTYPES[dtype], device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device,
                                dtype=torch.float32).to(out.dtype)
    return out


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------


@dataclass
class Workload:
    name: str
    dtype: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    context_lens: np.ndarray          # int32 [B]
    block_tables: np.ndarray          # int32 [B][MB]
    slot_mapping: np.ndarray          # int64 [T] (T = B, one new token each)
    q: torch.Tensor                   # [B][Hq][D]
    k_new: torch.Tensor               # [T][Hkv][D]
    v_new: torch.Tensor               # [T][Hkv][D]
    k_cache: torch.Tensor             # [NB][bs][Hkv][D], before the write
    v_cache: torch.Tensor
    shared_prefix_blocks: int = 0
    meta: Dict[str, object] = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_tokens(self) -> int:
        return int(self.slot_mapping.shape[0])

    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def kv_bytes_logical(self) -> int:
        """K and V bytes of every context token, as each sequence reads them."""
        e = 2
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_dim * e * 2

    def kv_bytes_unique(self) -> int:
        """K and V bytes of distinct cache slots (shared prefix counted once)."""
        e = 2
        per_tok = self.num_kv_heads * self.head_dim * e * 2
        shared_tok = self.shared_prefix_blocks * self.block_size
        total = int(self.context_lens.astype(np.int64).sum())
        if shared_tok:
            total -= shared_tok * (self.num_seqs - 1)
        return total * per_tok

    def qo_bytes(self) -> int:
        return 2 * self.num_seqs * self.num_q_heads * self.head_dim * 2


CONFIGS = {
    # name: (seed, dict of parameters)
    "tiny": (20260, dict(dtype="fp16", num_seqs=4, lens=[1, 17, 100, 250], num_q_heads=8,
                         num_kv_heads=2, head_dim=64, block_size=16, num_blocks=64)),
    "llama8b": (20261, dict(dtype="fp16", num_seqs=64, len_uniform=(128, 2048),
                            num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16)),
    "prefix": (20262, dict(dtype="bf16", num_seqs=256, prefix_tokens=512,
                           suffix_lognormal=(300.0, 1.0, 1, 4096), num_q_heads=32,
                           num_kv_heads=8, head_dim=128, block_size=16)),
    "llama70b": (20263, dict(dtype="fp16", num_seqs=32, lens=[4096] * 32, num_q_heads=64,
                             num_kv_heads=8, head_dim=128, block_size=16)),
    "long16": (20264, dict(dtype="bf16", num_seqs=8, len_uniform=(32768, 50000),
                           num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16)),
    "long32": (20264, dict(dtype="bf16", num_seqs=8, len_uniform=(32768, 50000),
                           num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32)),
}

DESCRIPTIONS = {
    "tiny": "batch 4, context {1,17,100,250}, 8 q / 2 KV heads, head_dim 64, block 16, fp16, "
            "pool 64 blocks",
    "llama8b": "Llama-3-8B-shaped decode layer: batch 64, context U[128,2048], 32 q / 8 KV heads, "
               "head_dim 128, block 16, fp16, pool +10% free, scattered",
    "prefix": "shared-prefix batch: 256 requests on one 512-token prefix (32 blocks, ref 256) + "
              "lognormal suffix (median 300, cap 4096), 32 q / 8 KV heads, head_dim 128, bf16",
    "llama70b": "Llama-3-70B-shaped decode layer: batch 32, context 4096, 64 q / 8 KV heads, "
                "head_dim 128, block 16, fp16",
    "long16": "long context: batch 8, context U[32768,50000], 32 q / 8 KV heads, head_dim 128, "
              "bf16, block 16",
    "long32": "long context: batch 8, context U[32768,50000], 32 q / 8 KV heads, head_dim 128, "
              "bf16, block 32",
}


def _draw_lengths(rng: np.random.Generator, p: dict) -> (np.ndarray, int):
    B = p["num_seqs"]
    if "lens" in p:
        return np.asarray(p["lens"], dtype=np.int64), 0
    if "len_uniform" in p:
        lo, hi = p["len_uniform"]
        return rng.integers(lo, hi, size=B, endpoint=True).astype(np.int64), 0
    med, sigma, lo, hi = p["suffix_lognormal"]
    suf = np.rint(rng.lognormal(math.log(med), sigma, size=B)).astype(np.int64)
    suf = np.clip(suf, lo, hi)
    return p["prefix_tokens"] + suf, p["prefix_tokens"]


def build_workload(name: Optional[str] = None, seed: Optional[int] = None,
                   params: Optional[dict] = None, pool_slack: float = 0.10,
                   pool_device=None) -> Workload:
    """Build one named configuration (or ``params`` for a custom one).

    Recipe (seeded numpy PCG64): context lengths, then the pool permutation,
    then q, the new tokens' K and V, then the whole K pool and V pool, all
    N(0,1) float32 rounded to nearest-even fp16/bf16.  Every sequence holds
    its first ``L_b - 1`` tokens; its last token is appended with
    ``append_token`` and its slot goes to ``slot_mapping``.  Table rows are
    padded with block id 0 past their end.

    With ``pool_device`` the two pools are drawn instead on that device by a
    torch generator seeded with ``seed`` (same distribution, other values;
    everything else is unchanged) and returned there: timing runs of the
    large workloads use it.
    """
    if params is None:
        base_seed, params = CONFIGS[name]
        seed = base_seed if seed is None else seed
    else:
        params = dict(params)
        seed = 0 if seed is None else seed
        name = name or "custom"
    p = params
    rng = np.random.default_rng(seed)
    B, bs = p["num_seqs"], p["block_size"]
    hq, hkv, d, dt = p["num_q_heads"], p["num_kv_heads"], p["head_dim"], p["dtype"]
    lens, prefix = _draw_lengths(rng, p)
    if np.any(lens < 0):
        raise ValueError("negative context length")
    prefix_blocks = -(-prefix // bs)
    need = prefix_blocks + sum(max(1, -(-(int(n) - prefix) // bs)) for n in lens)
    nb = int(p.get("num_blocks") or math.ceil(need * (1.0 + pool_slack)))
    if nb < need:
        raise ValueError(f"pool of {nb} blocks cannot hold {need}")
    perm = rng.permutation(nb)
    if p.get("placement", "random") == "sequential":
        perm = np.arange(nb)[::-1]          # pops 0, 1, 2, ...: blocks in pool order
    pool = BlockPool(nb, bs, order=perm)
    alloc = PagedKVAllocator(pool)
    shared = [pool.allocate() for _ in range(prefix_blocks)]
    slots = np.full(B, -1, dtype=np.int64)
    for b in range(B):
        L = int(lens[b])
        if shared:
            alloc.add_sequence(b, shared, prefix)
        else:
            alloc.add_sequence(b)
        if L == 0:
            continue
        alloc.extend(b, L - 1 - (prefix if shared else 0))
        slots[b] = alloc.append_token(b)
    for p_ in shared:          # the builder's own hold on the prefix
        pool.free(p_)
    tables = alloc.table_array(range(B))
    q = normal_tensor(rng, (B, hq, d), dt)
    k_new = normal_tensor(rng, (B, hkv, d), dt)
    v_new = normal_tensor(rng, (B, hkv, d), dt)
    if pool_device is None:
        k_cache = normal_tensor(rng, (nb, bs, hkv, d), dt)
        v_cache = normal_tensor(rng, (nb, bs, hkv, d), dt)
    else:
        gen = torch.Generator(device=pool_device)
        gen.manual_seed(seed)
        k_cache = normal_tensor_device(gen, (nb, bs, hkv, d), dt, pool_device)
        v_cache = normal_tensor_device(gen, (nb, bs, hkv, d), dt, pool_device)
    return Workload(name=name, dtype=dt, num_seqs=B, num_q_heads=hq, num_kv_heads=hkv,
                    head_dim=d, block_size=bs, num_blocks=nb, scale=1.0 / math.sqrt(d),
                    context_lens=lens.astype(np.int32), block_tables=tables,
                    slot_mapping=slots, q=q, k_new=k_new, v_new=v_new, k_cache=k_cache,
                    v_cache=v_cache, shared_prefix_blocks=prefix_blocks,
                    meta={"seed": seed, "params": p, "ref_count_prefix":
                          (pool.ref_count[shared[0]] if shared else 0)})


def fp8_codes(rng: np.random.Generator, shape, scale: float) -> torch.Tensor:
    """uint8 E4M3 codes of N(0,1) / scale (clipped to +-448), for a synthetic
    FP8 cache whose elements are code values times ``scale``."""
    x = normal_tensor(rng, shape, "bf16").float() / scale
    return x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def fp8_codes_device(gen: torch.Generator, shape, scale: float, device,
                     chunk_elems: int = 1 << 26) -> torch.Tensor:
    """The same as ``fp8_codes`` from a seeded device generator, made on the
    device."""
    out = torch.empty(tuple(shape), dtype=torch.uint8, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        x = x.to(torch.bfloat16).float() / scale
        flat[s:e] = x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return out


@dataclass
class PrefillWorkload:
    """A chunked-prefill batch: sequence b holds L_b tokens, the last C_b of
    them new in this step (their slots from append_token, their K/V in
    k_new / v_new, their queries in q)."""
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    context_lens: np.ndarray          # int32 [B]
    query_start: np.ndarray           # int32 [B + 1]
    block_tables: np.ndarray          # int32 [B][MB]
    slot_mapping: np.ndarray          # int64 [T], T = sum C_b
    q: torch.Tensor                   # [T][Hq][D]
    k_new: torch.Tensor               # [T][Hkv][D]
    v_new: torch.Tensor
    k_cache: torch.Tensor             # [NB][bs][Hkv][D], before the write
    v_cache: torch.Tensor

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def num_tokens(self) -> int:
        return int(self.query_start[-1])

    def flops(self) -> int:
        """Score and value products of the causal attention: 4*D per
        (query row, visible key)."""
        hq, d = self.num_q_heads, self.head_dim
        total = 0
        for b in range(self.num_seqs):
            L, C = int(self.context_lens[b]), int(self.query_start[b + 1] - self.query_start[b])
            total += sum(L - C + i + 1 for i in range(C))
        return 4 * d * hq * total

    def kv_bytes(self) -> int:
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * self.head_dim * 4


PREFILL_CONFIGS = {
    # chunked prefill of Llama-3-8B-shaped layers: 4 sequences, 512-token
    # chunks appended to contexts of 0..3584 earlier tokens
    "prefill8b": (20270, dict(dtype="bf16", lens=[512, 1536, 2560, 4096], chunks=[512] * 4,
                              num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16)),
    "prefill_tiny": (20271, dict(dtype="fp16", lens=[1, 20, 64, 100], chunks=[1, 20, 17, 33],
                                 num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16)),
}


PREFILL_DESCRIPTIONS = {
    "prefill8b": "chunked prefill, Llama-3-8B-shaped layer: 4 sequences, 512 new tokens each "
                 "on contexts of 512/1536/2560/4096, 32 q / 8 KV heads, head_dim 128, bf16, "
                 "block 16",
    "prefill_tiny": "small chunked prefill: 4 sequences, chunks 1/20/17/33 on contexts "
                    "1/20/64/100, 8 q / 2 KV heads, head_dim 64, fp16, block 16",
}


def build_prefill_workload(name: Optional[str] = None, seed: Optional[int] = None,
                           params: Optional[dict] = None, pool_slack: float = 0.10):
    """Seeded chunked-prefill batch (same recipe as ``build_workload``: the
    pool permutation, then q, new K, new V, K pool, V pool)."""
    if params is None:
        base_seed, params = PREFILL_CONFIGS[name]
        seed = base_seed if seed is None else seed
    else:
        seed = 0 if seed is None else seed
        name = name or "custom"
    p = params
    rng = np.random.default_rng(seed)
    lens = np.asarray(p["lens"], dtype=np.int64)
    chunks = np.asarray(p["chunks"], dtype=np.int64)
    if np.any(chunks > lens) or np.any(chunks < 0):
        raise ValueError("a chunk is longer than its context")
    B, bs = len(lens), p["block_size"]
    hq, hkv, d, dt = p["num_q_heads"], p["num_kv_heads"], p["head_dim"], p["dtype"]
    need = sum(max(1, -(-int(n) // bs)) for n in lens)
    nb = int(p.get("num_blocks") or math.ceil(need * (1.0 + pool_slack)))
    pool = BlockPool(nb, bs, order=rng.permutation(nb))
    alloc = PagedKVAllocator(pool)
    slots = []
    for b in range(B):
        alloc.add_sequence(b)
        alloc.extend(b, int(lens[b] - chunks[b]))
        slots += [alloc.append_token(b) for _ in range(int(chunks[b]))]
    T = int(chunks.sum())
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return PrefillWorkload(
        name=name, dtype=dt, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
        num_blocks=nb, scale=1.0 / math.sqrt(d), context_lens=lens.astype(np.int32),
        query_start=qs, block_tables=alloc.table_array(range(B)),
        slot_mapping=np.asarray(slots, dtype=np.int64),
        q=normal_tensor(rng, (T, hq, d), dt), k_new=normal_tensor(rng, (T, hkv, d), dt),
        v_new=normal_tensor(rng, (T, hkv, d), dt),
        k_cache=normal_tensor(rng, (nb, bs, hkv, d), dt),
        v_cache=normal_tensor(rng, (nb, bs, hkv, d), dt))


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a CPU fp16/bf16 tensor (no copy)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
