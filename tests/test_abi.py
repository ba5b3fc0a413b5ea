"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks reject bad calls before anything touches a GPU.  CPU only."""
import ctypes

import pytest

from paged_kv_cache_226_gb300 import build, lib


@pytest.fixture(scope="module")
def pa():
    build.build()
    return lib.load()


def test_exports_every_header_symbol(pa):
    names = lib.header_symbols()
    assert {"pa_reshape_and_cache", "pa_decode", "pa_decode_split", "pa_reduce"} <= set(names)
    for n in names:
        assert hasattr(pa, n), f"libpa.so does not export {n}"


def test_product_library_has_no_test_hook(pa):
    """The failure-detection hook (include/pa_test.h) exists only in the test
    build, libpa_test.so."""
    assert not hasattr(pa, "pa_test_set_wait_fault")


def test_status_strings(pa):
    assert lib.status_string(lib.PA_OK) == "ok"
    assert "unsupported" in lib.status_string(lib.PA_ERR_UNSUPPORTED)
    assert lib.status_string(99) == "unknown status"


def _shape(**kw):
    base = dict(num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                max_blocks_per_seq=4, num_blocks=16, dtype=lib.PA_FP16, reserved=0)
    base.update(kw)
    return lib.PaShape(**base)


FAKE = ctypes.c_void_p(1 << 20)      # 16-byte aligned, never dereferenced


def _decode(pa, shp, **ptrs):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, cl=FAKE, out=FAKE)
    a.update(ptrs)
    return pa.pa_decode(a["q"], a["kc"], a["vc"], a["bt"], a["cl"], 0.1, a["out"],
                        ctypes.byref(shp), None)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), lib.PA_ERR_UNSUPPORTED),
    (dict(head_dim=0), lib.PA_ERR_INVALID_ARG),
    (dict(block_size=8), lib.PA_ERR_UNSUPPORTED),
    (dict(num_q_heads=7), lib.PA_ERR_INVALID_ARG),
    (dict(num_q_heads=32, num_kv_heads=2), lib.PA_ERR_UNSUPPORTED),
    (dict(dtype=5), lib.PA_ERR_INVALID_ARG),
    (dict(reserved=1), lib.PA_ERR_INVALID_ARG),
    (dict(max_blocks_per_seq=0), lib.PA_ERR_INVALID_ARG),
    (dict(num_seqs=70000), lib.PA_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_shapes(pa, kw, status):
    assert _decode(pa, _shape(**kw)) == status


def test_decode_rejects_null_and_misaligned(pa):
    assert _decode(pa, _shape(), q=None) == lib.PA_ERR_INVALID_ARG
    assert _decode(pa, _shape(), out=None) == lib.PA_ERR_INVALID_ARG
    assert _decode(pa, _shape(), kc=ctypes.c_void_p((1 << 20) + 8)) == lib.PA_ERR_INVALID_ARG
    assert pa.pa_decode(FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, FAKE, None, None) == \
        lib.PA_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(pa):
    assert _decode(pa, _shape(num_seqs=0), q=None, out=None) == lib.PA_OK
    shp = _shape()
    assert pa.pa_reshape_and_cache(None, None, None, None, None, 0, ctypes.byref(shp),
                                   None) == lib.PA_OK


def test_split_argument_checks(pa):
    shp = _shape()
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 0.1]
    assert pa.pa_decode_split(*args, 500, 4, FAKE, FAKE, FAKE, ctypes.byref(shp), None) == \
        lib.PA_ERR_INVALID_ARG                      # partition not a multiple of block_size
    assert pa.pa_decode_split(*args, 512, 0, FAKE, FAKE, FAKE, ctypes.byref(shp), None) == \
        lib.PA_ERR_WORKSPACE
    assert pa.pa_decode_split(*args, 512, 4, None, FAKE, FAKE, ctypes.byref(shp), None) == \
        lib.PA_ERR_WORKSPACE
    assert pa.pa_reduce(FAKE, FAKE, FAKE, FAKE, 512, 0, FAKE, ctypes.byref(shp), None) == \
        lib.PA_ERR_WORKSPACE


def test_reshape_argument_checks(pa):
    shp = _shape()
    assert pa.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, -1, ctypes.byref(shp),
                                   None) == lib.PA_ERR_INVALID_ARG
    assert pa.pa_reshape_and_cache(FAKE, None, FAKE, FAKE, FAKE, 3, ctypes.byref(shp),
                                   None) == lib.PA_ERR_INVALID_ARG
    bad = _shape(head_dim=80)
    assert pa.pa_reshape_and_cache(FAKE, FAKE, FAKE, FAKE, FAKE, 3, ctypes.byref(bad),
                                   None) == lib.PA_ERR_UNSUPPORTED


def test_workspace_size(pa):
    shp = _shape(num_seqs=8, num_q_heads=32, num_kv_heads=8, max_blocks_per_seq=3125)
    sz = pa.pa_split_workspace_size(ctypes.byref(shp), 50000, 512)
    parts = -(-50000 // 512)
    rows = 8 * 32 * parts
    assert sz == -(-rows * 128 * 4 // 256) * 256 + 2 * (-(-rows * 4 // 256) * 256)
    assert pa.pa_split_workspace_size(ctypes.byref(shp), 50000, 500) == 0


@pytest.mark.parametrize("hq,hkv,d,max_q,want_chunks", [
    (32, 8, 128, 512, 16),      # G = 4: 32 tokens per tcgen05 CTA
    (64, 8, 128, 700, 44),      # G = 8: 16 tokens, a ragged last chunk
    (8, 8, 128, 129, 2),        # G = 1: 128 tokens
    (32, 8, 128, 31, 0),        # a chunk that cannot fill 128 rows: mma.sync kernel
    (8, 2, 64, 512, 0),         # head_dim 64: mma.sync kernel
    (12, 2, 128, 512, 0),       # G = 6: mma.sync kernel
])
def test_prefill_workspace_size(pa, hq, hkv, d, max_q, want_chunks):
    """One int32 per (sequence, chunk) item of the tcgen05 kernel, rounded up to
    256 bytes; 0 where pa_prefill takes the mma.sync kernel."""
    shp = _shape(num_seqs=5, num_q_heads=hq, num_kv_heads=hkv, head_dim=d)
    want = -(-5 * want_chunks * 4 // 256) * 256
    assert pa.pa_prefill_workspace_size(ctypes.byref(shp), max_q) == want
    assert pa.pa_prefill_workspace_size(ctypes.byref(shp), 0) == 0
    assert pa.pa_prefill_workspace_size(None, max_q) == 0


def test_prefill_ws_argument_checks(pa):
    shp = _shape(num_seqs=2, num_q_heads=32, num_kv_heads=8)
    # a workspace smaller than the size query asks for, or misaligned
    for ws, n in ((FAKE, 16), (ctypes.c_void_p((1 << 20) + 4), 4096)):
        st = pa.pa_prefill_ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.1, 512, ws, n, FAKE,
                              ctypes.byref(shp), None)
        assert st == lib.PA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        lib.load(str(tmp_path / "missing.so"))
