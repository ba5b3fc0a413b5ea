"""Pins for the CPU reference: checks against facts fixed by the pages, by
library routines and by mathematics -- never against the oracle itself.

CPU only.  Each test names what pins it.
"""
import json
import math
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
from oracle import alloc_model
from paged_kv_cache_226_gb300 import inputs as pin

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _to_bits(x, dtype):
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(pin.torch_dtype(dtype))
    return pin.bits(t)


# --------------------------------------------------------------------------
# widening of the storage formats: pinned to numpy / torch conversions
# --------------------------------------------------------------------------

def test_widen_fp16_every_pattern_matches_numpy():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(pats, "fp16")
    want = pats.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_widen_bf16_every_pattern_matches_torch():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(pats, "bf16")
    want = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


# --------------------------------------------------------------------------
# hand-worked decode cases (tests/golden/hand_worked_decode.json)
# --------------------------------------------------------------------------

def _place_hand_case(c, dtype):
    hkv, d, bs, nb = c["num_kv_heads"], c["head_dim"], c["block_size"], c["num_blocks"]
    kc = np.tile(np.asarray(c["junk_k"], np.float32), (nb, bs, hkv, 1))
    vc = np.tile(np.asarray(c["junk_v"], np.float32), (nb, bs, hkv, 1))
    lk = np.asarray(c["logical_k"], np.float32)
    lv = np.asarray(c["logical_v"], np.float32)
    table = c["block_tables"][0]
    for i in range(c["context_lens"][0]):
        p, o = table[i // bs], i % bs
        kc[p, o] = lk[i]
        vc[p, o] = lv[i]
    return _to_bits(kc, dtype), _to_bits(vc, dtype)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_hand_worked_cases(dtype):
    for c in _golden("hand_worked_decode.json")["cases"]:
        kc, vc = _place_hand_case(c, dtype)
        q = _to_bits(c["q"], dtype)
        scale = math.log(2.0) if c["scale"] == "ln2" else float(c["scale"])
        out = oracle.paged_decode(q, kc, vc, np.asarray(c["block_tables"], np.int32),
                                  np.asarray(c["context_lens"], np.int32), scale, dtype)
        np.testing.assert_allclose(out, np.asarray(c["expected_out"], np.float64),
                                   rtol=0, atol=1e-12, err_msg=c["name"])


# --------------------------------------------------------------------------
# agreement with torch's scaled_dot_product_attention (fp64) on the
# logical (gathered) K/V: pins the table walk, the GQA mapping and the math
# --------------------------------------------------------------------------

def _small_workload(dtype, hq=8, hkv=2, d=64, bs=16, lens=(1, 5, 16, 17, 33, 70), seed=7):
    return pin.build_workload(params=dict(dtype=dtype, num_seqs=len(lens), lens=list(lens),
                                          num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                          block_size=bs), seed=seed)


def _logical_kv(w, kc_bits, vc_bits):
    """numpy gather of each sequence's tokens, in logical order (test code)."""
    kc = oracle.widen(kc_bits, w.dtype)
    vc = oracle.widen(vc_bits, w.dtype)
    ks, vs = [], []
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        idx = np.arange(L)
        phys = w.block_tables[b][idx // w.block_size]
        ks.append(kc[phys, idx % w.block_size])     # [L][Hkv][D]
        vs.append(vc[phys, idx % w.block_size])
    return ks, vs


def _sdpa_reference(w, q_bits, ks, vs):
    q = oracle.widen(q_bits, w.dtype)
    G = w.num_q_heads // w.num_kv_heads
    out = np.zeros((w.num_seqs, w.num_q_heads, w.head_dim))
    for b in range(w.num_seqs):
        if ks[b].shape[0] == 0:
            continue
        K = torch.from_numpy(ks[b]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        V = torch.from_numpy(vs[b]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        Q = torch.from_numpy(q[b]).unsqueeze(1)                     # [Hq][1][D]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=w.scale)
        out[b] = o[:, 0, :].numpy()
    return out


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [("fp16", 8, 2, 64, 16), ("bf16", 32, 8, 128, 16),
                                               ("fp16", 4, 4, 64, 32), ("bf16", 8, 1, 128, 32)])
def test_paged_decode_matches_sdpa(dtype, hq, hkv, d, bs):
    w = _small_workload(dtype, hq, hkv, d, bs)
    qb, kcb, vcb = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    got = oracle.paged_decode(qb, kcb, vcb, w.block_tables, w.context_lens, w.scale, dtype)
    ks, vs = _logical_kv(w, kcb, vcb)
    want = _sdpa_reference(w, qb, ks, vs)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_contiguous_decode_matches_paged():
    w = _small_workload("fp16")
    qb, kcb, vcb = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    ks_f, vs_f = [], []
    kc, vc = kcb, vcb
    starts, pos = [], 0
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        idx = np.arange(L)
        phys = w.block_tables[b][idx // w.block_size]
        ks_f.append(kc[phys, idx % w.block_size])
        vs_f.append(vc[phys, idx % w.block_size])
        starts.append(pos)
        pos += L
    kseq = np.concatenate(ks_f)
    vseq = np.concatenate(vs_f)
    got = oracle.contiguous_decode(qb, kseq, vseq, np.asarray(starts), w.context_lens, w.scale,
                                   "fp16")
    want = oracle.paged_decode(qb, kcb, vcb, w.block_tables, w.context_lens, w.scale, "fp16")
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def test_permutation_invariance():
    """The same logical tokens placed in three different physical layouts
    give the same answer: the table changes where K/V live, not the result."""
    base = _small_workload("bf16", lens=(3, 40, 64, 65, 100))
    qb, kcb, vcb = pin.bits(base.q), pin.bits(base.k_cache), pin.bits(base.v_cache)
    ks, vs = _logical_kv(base, kcb, vcb)
    ref = None
    for seed in (1, 2, 3):
        rng = np.random.default_rng(seed)
        perm = rng.permutation(base.num_blocks)
        kc = np.zeros_like(kcb) + np.uint16(0x3c00)
        vc = np.zeros_like(vcb) + np.uint16(0xbc00)
        tables = np.zeros_like(base.block_tables)
        nxt = 0
        for b in range(base.num_seqs):
            L = int(base.context_lens[b])
            for j in range(-(-L // base.block_size)):
                p = perm[nxt]
                nxt += 1
                tables[b, j] = p
                lo, hi = j * base.block_size, min(L, (j + 1) * base.block_size)
                kc[p, :hi - lo] = pin.bits(torch.from_numpy(ks[b][lo:hi]).to(torch.bfloat16))
                vc[p, :hi - lo] = pin.bits(torch.from_numpy(vs[b][lo:hi]).to(torch.bfloat16))
        out = oracle.paged_decode(qb, kc, vc, tables, base.context_lens, base.scale, "bf16")
        if ref is None:
            ref = out
        else:
            assert np.array_equal(out, ref)


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

def test_context_one_returns_that_value_row():
    w = _small_workload("fp16", lens=(1, 1, 1))
    qb, kcb, vcb = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    out = oracle.paged_decode(qb, kcb, vcb, w.block_tables, w.context_lens, w.scale, "fp16")
    vc = oracle.widen(vcb, "fp16")
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.num_seqs):
        p = w.block_tables[b, 0]
        for h in range(w.num_q_heads):
            assert np.array_equal(out[b, h], vc[p, 0, h // G])


@pytest.mark.parametrize("mode", ["identical_keys", "zero_query"])
def test_uniform_weights_give_mean_of_values(mode):
    w = _small_workload("bf16", lens=(7, 16, 50))
    qb, kcb, vcb = pin.bits(w.q).copy(), pin.bits(w.k_cache).copy(), pin.bits(w.v_cache)
    if mode == "identical_keys":
        kcb[:] = kcb[0, 0, 0]           # every key row equal
    else:
        qb[:] = 0
    out = oracle.paged_decode(qb, kcb, vcb, w.block_tables, w.context_lens, w.scale, "bf16")
    _, vs = _logical_kv(w, kcb, vcb)
    G = w.num_q_heads // w.num_kv_heads
    for b in range(w.num_seqs):
        mean = vs[b].mean(axis=0)                          # [Hkv][D]
        np.testing.assert_allclose(out[b], np.repeat(mean, G, axis=0), rtol=1e-13,
                                   atol=1e-13)


def test_empty_context_gives_zeros():
    w = _small_workload("fp16", lens=(0, 5))
    out = oracle.paged_decode(pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache),
                              w.block_tables, w.context_lens, w.scale, "fp16")
    assert np.all(out[0] == 0)
    assert np.all(np.isfinite(out[1]))


def test_gqa_equals_mha_with_duplicated_kv_heads():
    w = _small_workload("fp16", hq=8, hkv=2, lens=(9, 31, 48))
    G = 4
    qb, kcb, vcb = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    gqa = oracle.paged_decode(qb, kcb, vcb, w.block_tables, w.context_lens, w.scale, "fp16")
    kdup = np.ascontiguousarray(np.repeat(kcb, G, axis=2))
    vdup = np.ascontiguousarray(np.repeat(vcb, G, axis=2))
    mha = oracle.paged_decode(qb, kdup, vdup, w.block_tables, w.context_lens, w.scale, "fp16")
    assert np.array_equal(gqa, mha)


# --------------------------------------------------------------------------
# context split + log-sum-exp merge
# --------------------------------------------------------------------------

@pytest.mark.parametrize("P", [16, 32, 48, 512])
def test_partition_merge_equals_unsplit(P):
    w = _small_workload("bf16", lens=(1, 16, 17, 47, 48, 49, 130))
    qb, kcb, vcb = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    S = -(-int(w.context_lens.max()) // P)
    po, pm, ps = oracle.paged_decode_partitions(qb, kcb, vcb, w.block_tables, w.context_lens,
                                                w.scale, "bf16", P, S)
    merged = oracle.lse_merge(po, pm, ps, w.context_lens, P)
    full = oracle.paged_decode(qb, kcb, vcb, w.block_tables, w.context_lens, w.scale, "bf16")
    np.testing.assert_allclose(merged, full, rtol=1e-12, atol=1e-13)
    for b in range(w.num_seqs):
        nb = -(-int(w.context_lens[b]) // P)
        assert np.all(np.isfinite(pm[b, :, :nb])) and np.all(np.isnan(pm[b, :, nb:]))


def test_partition_statistics_against_numpy_scores():
    """m_s and l_s against scores formed with numpy's dot (library) in fp64."""
    w = _small_workload("fp16", hq=4, hkv=2, lens=(20, 33))
    P = 16
    qb, kcb, vcb = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    po, pm, ps = oracle.paged_decode_partitions(qb, kcb, vcb, w.block_tables, w.context_lens,
                                                w.scale, "fp16", P, 3)
    ks, vs = _logical_kv(w, kcb, vcb)
    q = oracle.widen(qb, "fp16")
    for b in range(w.num_seqs):
        for h in range(w.num_q_heads):
            s_all = w.scale * (ks[b][:, h // 2, :] @ q[b, h])
            for s in range(-(-len(s_all) // P)):
                seg = s_all[s * P:(s + 1) * P]
                assert pm[b, h, s] == pytest.approx(seg.max(), abs=1e-13)
                assert ps[b, h, s] == pytest.approx(np.exp(seg - seg.max()).sum(), rel=1e-13)
                wts = np.exp(seg - seg.max())
                o = (wts[:, None] * vs[b][s * P:s * P + len(seg), h // 2, :]).sum(0) / wts.sum()
                np.testing.assert_allclose(po[b, h, s], o, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# reshape_and_cache: bit-exact against numpy indexed assignment
# --------------------------------------------------------------------------

def test_reshape_and_cache_matches_numpy_assignment():
    w = _small_workload("fp16", lens=(1, 16, 17, 32, 90))
    slots = w.slot_mapping.copy()
    slots[2] = -1                                     # padding token
    kb, vb = pin.bits(w.k_new), pin.bits(w.v_new)
    kc, vc, bad = oracle.reshape_and_cache(kb, vb, slots, pin.bits(w.k_cache),
                                           pin.bits(w.v_cache), w.block_size)
    assert bad == 0
    for src, new, cache in ((kb, kc, pin.bits(w.k_cache)), (vb, vc, pin.bits(w.v_cache))):
        want = cache.copy().reshape(w.num_blocks * w.block_size, -1)
        keep = slots >= 0
        want[slots[keep]] = src.reshape(len(slots), -1)[keep]
        assert np.array_equal(new.reshape(want.shape), want)
    # out-of-pool slots are reported and not written
    far = np.array([w.num_blocks * w.block_size + 3], dtype=np.int64)
    kc2, _, bad2 = oracle.reshape_and_cache(kb[:1], vb[:1], far, pin.bits(w.k_cache),
                                            pin.bits(w.v_cache), w.block_size)
    assert bad2 == 1 and np.array_equal(kc2, pin.bits(w.k_cache))


def test_append_token_slot_semantics():
    """Slots from append_token: count % block_size inside the last block, a
    new block when that is 0 and the request already holds tokens
    (youngju.dev post, PagedAttentionManager.append_token)."""
    pool = pin.BlockPool(4, 4, order=[3, 2, 1, 0])       # pops 0, 1, 2, 3
    a = pin.PagedKVAllocator(pool)
    a.add_sequence(0)
    slots = [a.append_token(0) for _ in range(9)]
    assert slots == [0, 1, 2, 3, 4, 5, 6, 7, 8]
    assert a.page_tables[0] == [0, 1, 2]
    b = pin.PagedKVAllocator(pin.BlockPool(4, 4, order=[0, 2, 1, 3]))
    b.add_sequence(0)
    assert [b.append_token(0) for _ in range(6)] == [12, 13, 14, 15, 4, 5]
    c = pin.PagedKVAllocator(pin.BlockPool(4, 4, order=[0, 2, 1, 3]))
    c.add_sequence(0)
    c.extend(0, 5)
    assert c.append_token(0) == 5 and c.page_tables[0] == b.page_tables[0]


def test_allocator_exhaustion_and_ref_counts():
    pool = pin.BlockPool(3, 16)
    ids = [pool.allocate() for _ in range(3)]
    assert ids == [2, 1, 0]
    with pytest.raises(MemoryError, match="No free blocks"):
        pool.allocate()
    pool.share(ids[0])
    pool.share(ids[0])
    pool.free(ids[0])
    pool.free(ids[0])
    assert pool.num_free == 0 and pool.ref_count[ids[0]] == 1
    pool.free(ids[0])
    assert pool.num_free == 1
    with pytest.raises(ValueError):
        pool.free(ids[0])


def test_shared_prefix_workload_ref_counts():
    w = pin.build_workload(params=dict(dtype="bf16", num_seqs=5, prefix_tokens=64,
                                       suffix_lognormal=(20.0, 1.0, 1, 100), num_q_heads=4,
                                       num_kv_heads=2, head_dim=64, block_size=16), seed=3)
    assert w.shared_prefix_blocks == 4 and w.meta["ref_count_prefix"] == 5
    first = w.block_tables[:, :4]
    assert np.all(first == first[0])
    private = [set(w.block_tables[b, 4:-(-int(w.context_lens[b]) // 16)]) for b in range(5)]
    for i in range(5):
        for j in range(i + 1, 5):
            assert not private[i] & private[j]


# --------------------------------------------------------------------------
# the pages' printed numbers
# --------------------------------------------------------------------------

def test_contiguous_reservation_waste_example():
    g = _golden("waste_example.json")
    r = alloc_model.contiguous_reservation(g["used_lens"], g["max_len"])
    assert r["reserved"] == g["printed_reserved_slots"]
    assert r["used"] == g["printed_used_slots"]
    assert r["waste"] * 100 == pytest.approx(g["printed_waste_percent"], abs=1e-12)
    paged = alloc_model.paged_usage(g["used_lens"], 16)
    assert paged["slots"] == 4608 and paged["waste"] == 0.0
    assert all(0 <= t < 16 for t in alloc_model.paged_usage([1, 17, 100, 250], 16)["tail_waste"])


def test_page_table_example():
    g = _golden("page_table_example.json")
    occ = alloc_model.pool_occupancy(g["num_blocks"], g["tables"].values())
    assert occ["free"] == g["printed_free"]
    assert len(occ["used"]) == 7


def test_kv_byte_formulas():
    g = _golden("kv_bytes.json")
    p = g["per_token"]
    assert alloc_model.kv_bytes_per_token(p["num_layers"], p["num_kv_heads"], p["head_dim"],
                                          p["dtype_bytes"]) == p["printed_bytes"]
    f = g["formula_case"]
    gib = 1024 ** 3
    assert alloc_model.kv_cache_bytes(f["num_layers"], f["num_heads"], f["head_dim"],
                                      f["seq_len"], f["batch_size"], f["dtype_bytes"]) / gib \
        == f["gib_with_64_heads"]
    assert alloc_model.kv_cache_bytes(f["num_layers"], f["num_kv_heads"], f["head_dim"],
                                      f["seq_len"], f["batch_size"], f["dtype_bytes"]) / gib \
        == f["gib_with_8_kv_heads"]


# --------------------------------------------------------------------------
# the pins catch plausible mistakes: each planted into a copy of the oracle
# --------------------------------------------------------------------------

MUTATIONS = {
    "gqa_mapping": ("h / G, num_kv_heads, head_dim, block_size,\n                    dtype",
                    "h % num_kv_heads, num_kv_heads, head_dim, block_size,\n                    dtype"),
    "dropped_scale": ("s[i] = scale * dot;\n        if (s[i] > m) m = s[i];\n    }\n    double l",
                      "s[i] = dot;\n        if (s[i] > m) m = s[i];\n    }\n    double l"),
    "offset_index": ("int64_t o = i % block_size;\n    return",
                     "int64_t o = (i + 1) % block_size;\n    return"),
    "no_normalise": ("for (int d = 0; d < head_dim; ++d) o[d] /= l;\n    }\n    free(s);",
                     "for (int d = 0; d < head_dim; ++d) o[d] /= 1.0;\n    }\n    free(s);"),
    "table_stride": ("block_tables + (int64_t)b * max_blocks_per_seq, 0,\n"
                     "                    context_lens[b]",
                     "block_tables + (int64_t)b, 0,\n                    context_lens[b]"),
    "k_for_v": ("const uint16_t* vr = paged_row(v_cache, table_row",
                "const uint16_t* vr = paged_row(k_cache, table_row"),
    "exp_sign": ("double w = exp(s[i] - m);\n        l += w;\n        const uint16_t* vr = paged_row",
                 "double w = exp(m - s[i]);\n        l += w;\n        const uint16_t* vr = paged_row"),
}


def _pins_pass() -> bool:
    try:
        test_hand_worked_cases("fp16")
        test_paged_decode_matches_sdpa("bf16", 32, 8, 128, 16)
    except AssertionError:
        return False
    return True


# mistakes in the chunked-prefill oracle, caught by the prefill pins below
PREFILL_MUTATIONS = {
    "prefill_origin": ("int64_t p = context_lens[b] - C + (tok - query_start[b]);",
                       "int64_t p = tok - query_start[b];"),
    "prefill_not_causal": ("p + 1, h / G, num_kv_heads", "context_lens[b], h / G, num_kv_heads"),
    "prefill_gqa": ("p + 1, h / G, num_kv_heads", "p + 1, h % num_kv_heads, num_kv_heads"),
    "prefill_includes_next": ("p + 1, h / G, num_kv_heads",
                              "(p + 2 < context_lens[b] ? p + 2 : p + 1), h / G, num_kv_heads"),
}


def _prefill_pins_pass() -> bool:
    try:
        test_prefill_matches_causal_sdpa("bf16", 16, 4, 128)
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("name", sorted(PREFILL_MUTATIONS))
def test_prefill_pins_fail_on_planted_mistake(name):
    old, new = PREFILL_MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as tmp:
        path = oracle.compile_variant(src.replace(old, new), os.path.join(tmp, "lib_mut.so"))
        with oracle.use_library(path):
            assert not _prefill_pins_pass(), f"prefill pins did not catch {name}"
    assert _prefill_pins_pass()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_fail_on_planted_mistake(name):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    with tempfile.TemporaryDirectory() as tmp:
        path = oracle.compile_variant(src.replace(old, new), os.path.join(tmp, "lib_mut.so"))
        with oracle.use_library(path):
            assert not _pins_pass(), f"pins did not catch planted mistake {name}"
    assert _pins_pass()


# --------------------------------------------------------------------------
# FP8 (E4M3) KV cache: decoding, quantisation, and attention over it
# --------------------------------------------------------------------------

def _torch_e4m3_values(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_e4m3_every_code_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = np.array([oracle.e4m3_to_f64(c) for c in codes])
    want = _torch_e4m3_values(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert oracle.e4m3_to_f64(0x7e) == 448.0 and np.isnan(oracle.e4m3_to_f64(0x7f))


def test_e4m3_rounding_matches_torch_in_range():
    rng = np.random.default_rng(5)
    ys = np.concatenate([rng.standard_normal(2000).astype(np.float32) * s
                         for s in (0.01, 1.0, 30.0, 200.0)])
    # exact midpoints between neighbouring codes exercise ties-to-even
    vals = _torch_e4m3_values(np.arange(0, 0x7e, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    ys = np.concatenate([ys, mids, -mids])
    ys = ys[np.abs(ys) < 448]
    got = np.array([oracle.f32_to_e4m3(y) for y in ys], dtype=np.uint8)
    want = torch.from_numpy(ys).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


def test_e4m3_saturates_and_keeps_nan():
    assert oracle.f32_to_e4m3(448.0) == 0x7e and oracle.f32_to_e4m3(1e30) == 0x7e
    assert oracle.f32_to_e4m3(-500.0) == 0xfe and oracle.f32_to_e4m3(float("-inf")) == 0xfe
    assert oracle.f32_to_e4m3(float("nan")) == 0x7f
    assert oracle.f32_to_e4m3(-0.0) == 0x80 and oracle.f32_to_e4m3(0.0) == 0x00


def test_fp8_cache_write_quantises_x_over_scale():
    w = _small_workload("bf16", hq=8, hkv=2, d=64, lens=(3, 20, 33))
    kc0 = np.zeros((w.num_blocks, w.block_size, 2, 64), np.uint8)
    vc0 = np.full_like(kc0, 0x38)
    ks, vs = 0.05, 0.11
    kc, vc, bad = oracle.reshape_and_cache_fp8(pin.bits(w.k_new), pin.bits(w.v_new),
                                               w.slot_mapping, kc0, vc0, w.block_size, "bf16",
                                               ks, vs)
    assert bad == 0
    for src, cache, base, sc in ((w.k_new, kc, kc0, ks), (w.v_new, vc, vc0, vs)):
        y = (src.float() / torch.tensor(sc, dtype=torch.float32)).numpy()   # fp32 quotient
        y = np.clip(y, -448, 448)
        codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        want = base.copy().reshape(w.num_blocks * w.block_size, -1)
        want[w.slot_mapping] = codes.reshape(len(w.slot_mapping), -1)
        assert np.array_equal(cache.reshape(want.shape), want)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_fp8_decode_matches_sdpa_on_dequantised_cache(dtype):
    w = _small_workload(dtype, hq=16, hkv=4, d=128, lens=(1, 17, 48, 90))
    rng = np.random.default_rng(11)
    kc = rng.integers(0, 256, size=(w.num_blocks, w.block_size, 4, 128), dtype=np.uint8)
    vc = rng.integers(0, 256, size=kc.shape, dtype=np.uint8)
    kc[(kc & 0x7f) == 0x7f] = 0x10                   # no NaN codes
    vc[(vc & 0x7f) == 0x7f] = 0x21
    ks, vs = 0.02, 0.3
    got = oracle.paged_decode_fp8(pin.bits(w.q), kc, vc, w.block_tables, w.context_lens,
                                  w.scale, ks, vs, dtype)
    kf = _torch_e4m3_values(kc) * ks
    vf = _torch_e4m3_values(vc) * vs
    q = oracle.widen(pin.bits(w.q), dtype)
    G = 4
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        idx = np.arange(L)
        phys = w.block_tables[b][idx // w.block_size]
        K = torch.from_numpy(kf[phys, idx % w.block_size]).permute(1, 0, 2).repeat_interleave(G, 0)
        V = torch.from_numpy(vf[phys, idx % w.block_size]).permute(1, 0, 2).repeat_interleave(G, 0)
        o = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[b]).unsqueeze(1), K, V, scale=w.scale)[:, 0].numpy()
        np.testing.assert_allclose(got[b], o, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# paged prefill (chunked prefill): causal attention of the new tokens
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,hq,hkv,d", [("fp16", 8, 2, 64), ("bf16", 16, 4, 128)])
def test_prefill_matches_causal_sdpa(dtype, hq, hkv, d):
    w = pin.build_prefill_workload(params=dict(dtype=dtype, lens=[1, 17, 40, 96],
                                               chunks=[1, 17, 9, 33], num_q_heads=hq,
                                               num_kv_heads=hkv, head_dim=d, block_size=16),
                                   seed=5)
    qb, kcb, vcb = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    got = oracle.paged_prefill(qb, kcb, vcb, w.block_tables, w.context_lens, w.query_start,
                               w.scale, dtype)
    kc, vc = oracle.widen(kcb, dtype), oracle.widen(vcb, dtype)
    q = oracle.widen(qb, dtype)
    G = hq // hkv
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        s0, s1 = int(w.query_start[b]), int(w.query_start[b + 1])
        C = s1 - s0
        idx = np.arange(L)
        phys = w.block_tables[b][idx // 16]
        K = torch.from_numpy(kc[phys, idx % 16]).permute(1, 0, 2).repeat_interleave(G, 0)
        V = torch.from_numpy(vc[phys, idx % 16]).permute(1, 0, 2).repeat_interleave(G, 0)
        Q = torch.from_numpy(q[s0:s1]).permute(1, 0, 2)               # [Hq][C][D]
        pos = L - C + torch.arange(C)
        mask = torch.arange(L)[None, :] <= pos[:, None]               # [C][L]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                             scale=w.scale)
        np.testing.assert_allclose(got[s0:s1], o.permute(1, 0, 2).numpy(), rtol=1e-12,
                                   atol=1e-12)


def test_prefill_of_one_token_is_decode():
    w = pin.build_prefill_workload(params=dict(dtype="bf16", lens=[5, 64, 200],
                                               chunks=[1, 1, 1], num_q_heads=8,
                                               num_kv_heads=2, head_dim=64, block_size=16),
                                   seed=8)
    qb, kcb, vcb = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    pre = oracle.paged_prefill(qb, kcb, vcb, w.block_tables, w.context_lens, w.query_start,
                               w.scale, "bf16")
    dec = oracle.paged_decode(qb, kcb, vcb, w.block_tables, w.context_lens, w.scale, "bf16")
    assert np.array_equal(pre, dec)
