"""The C-ABI library on the CPU: it loads, exports every symbol include/pkv.h
declares, and its host-only parts (page pool, block-table helpers, host
validation, sizing, argument checks that return before any CUDA call) behave
as documented.  No compute call is made here."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import paged_kv_decode_append_gb300 as pkv
from paged_kv_decode_append_gb300 import _lib
from paged_kv_decode_append_gb300.api import CacheDesc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = open(os.path.join(ROOT, "include", "pkv.h")).read()
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "printed_values.json")))


def declared_functions():
    return re.findall(r"PKV_API\s+[\w\s\*]*?\b(pkv_\w+)\s*\(", HEADER)


def test_every_declared_symbol_is_exported_and_bound():
    lib = _lib.load()
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"{n} has no ctypes signature"
    assert set(_lib.SIGNATURES) == set(names)


def test_status_strings():
    lib = _lib.load()
    for code in range(7):
        assert lib.pkv_status_str(code) not in (None, b"", b"unknown status")
    assert lib.pkv_status_str(99) == b"unknown status"


def test_pool_hands_out_ascending_and_never_page_zero():
    pool = pkv.PagePool(8)
    assert pool.num_free == 7
    assert list(pool.alloc(3)) == [1, 2, 3]
    with pytest.raises(pkv.PkvError) as e:
        pool.alloc(5)  # only 4 left: nothing taken
    assert e.value.status == pkv.api.ENOPAGES
    assert pool.num_free == 4
    assert list(pool.alloc(4)) == [4, 5, 6, 7]
    assert pool.num_free == 0


def test_pool_free_validates_everything_first():
    pool = pkv.PagePool(6)
    got = pool.alloc(3)
    for bad in ([0], [6], [4], [1, 1], [2, -1]):
        with pytest.raises(pkv.PkvError):
            pool.free(bad)
        assert pool.num_free == 2  # nothing returned
    pool.free([3, 1])
    assert pool.num_free == 4
    assert list(pool.alloc(2)) == [3, 1]  # returned pages are reused first
    assert set(got) == {1, 2, 3}


def test_shuffle_is_a_seeded_permutation():
    a, b, c = pkv.PagePool(1000), pkv.PagePool(1000), pkv.PagePool(1000)
    a.shuffle(7)
    b.shuffle(7)
    c.shuffle(8)
    pa, pb, pc = a.alloc(999), b.alloc(999), c.alloc(999)
    assert np.array_equal(pa, pb) and not np.array_equal(pa, pc)
    assert sorted(pa.tolist()) == list(range(1, 1000))
    assert not np.array_equal(pa, np.arange(1, 1000))


def test_table_reserve_and_release():
    pool = pkv.PagePool(20)
    row = np.zeros(6, np.int32)
    pool.reserve(row, 16, 0, 17)          # 2 blocks
    assert list(row[:2]) == [1, 2] and row[2] == 0
    pool.reserve(row, 16, 17, 32)         # still 2 blocks
    assert pool.num_free == 17
    pool.reserve(row, 16, 32, 33)         # third block
    assert list(row[:3]) == [1, 2, 3]
    with pytest.raises(pkv.PkvError):
        pool.reserve(row, 16, 33, 7 * 16)  # beyond max_blocks
    with pytest.raises(pkv.PkvError):
        pool.reserve(row, 16, 33, 20)      # shrinking
    pool.release(row, 16, 33)
    assert pool.num_free == 19 and not row.any()
    small = pkv.PagePool(3)
    row2 = np.zeros(4, np.int32)
    with pytest.raises(pkv.PkvError) as e:
        small.reserve(row2, 4, 0, 13)     # needs 4 pages, 2 free
    assert e.value.status == pkv.api.ENOPAGES and not row2.any() and small.num_free == 2


def test_validate_host():
    d = CacheDesc(10, 4, 2, 64, 0)
    bt = np.array([[1, 2, 0], [3, 0, 0], [9, 0, 0]], np.int32)
    assert pkv.pkv_validate_host(d, bt, np.array([5, 3, -1], np.int32), 1) == (0, -1)
    assert pkv.pkv_validate_host(d, bt, np.array([5, 4, -1], np.int32), 1) == (pkv.api.EINVAL, 1)
    assert pkv.pkv_validate_host(d, bt, np.array([5, 3, 12], np.int32), 0) == (pkv.api.EINVAL, 2)
    bt[2, 0] = 10  # == num_pages: out of range
    assert pkv.pkv_validate_host(d, bt, np.array([5, 3, 1], np.int32), 0) == (pkv.api.EINVAL, 2)


def test_pool_bytes_matches_printed_example():
    g = GOLDEN["pool_bytes"]
    per_layer_kv = 2 * pkv.pkv_pool_bytes(CacheDesc(g["num_pages"], g["page_size"], g["num_kv_heads"],
                                                    g["head_dim"], 0))
    assert per_layer_kv * g["layers"] == g["total_bytes"]


def test_workspace_size():
    d = CacheDesc(65536, 16, 8, 128, 0)
    n = pkv.pkv_decode_workspace_size(32, 65, 32, d)
    assert n > 0 and n % 256 == 0
    assert pkv.pkv_decode_workspace_size(64, 2049, 32, d) > n
    assert pkv.pkv_decode_workspace_size(1025, 65, 32, d) == 0
    assert pkv.pkv_decode_workspace_size(32, 65, 30, d) == 0          # Hq % Hkv
    assert pkv.pkv_decode_workspace_size(32, 65, 32, CacheDesc(100, 16, 8, 96, 0)) == 0   # D
    assert pkv.pkv_decode_workspace_size(32, 65, 32, CacheDesc(100, 12, 8, 128, 0)) == 0  # P


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced on the host paths below


def _decode(lib, desc, batch=4, hq=8, ws=FAKE, ws_bytes=1 << 30, q=FAKE, k_new=None, v_new=None, scale=0.1):
    return lib.pkv_decode_attn(ctypes.byref(desc), FAKE, FAKE, q, k_new, v_new, FAKE, 4, FAKE, batch, hq, scale,
                               FAKE, None, ws, ws_bytes, None, None)


def test_decode_argument_errors_return_before_any_launch():
    lib = _lib.load()
    d = CacheDesc(64, 16, 2, 128, 0)
    assert _decode(lib, CacheDesc(1, 16, 2, 128, 0)) == pkv.api.EINVAL        # no page beside the null page
    assert _decode(lib, CacheDesc(64, 16, 2, 128, 3)) == pkv.api.EINVAL       # layout
    assert _decode(lib, CacheDesc(64, 24, 2, 128, 0)) == pkv.api.EUNSUPPORTED  # page size
    assert _decode(lib, CacheDesc(64, 16, 2, 80, 0)) == pkv.api.EUNSUPPORTED   # head dim
    assert _decode(lib, d, hq=7) == pkv.api.EINVAL                             # Hq % Hkv
    assert _decode(lib, d, hq=6) == pkv.api.EUNSUPPORTED                       # group 3
    assert _decode(lib, d, q=None) == pkv.api.EINVAL
    assert _decode(lib, d, q=ctypes.c_void_p(0x10008)) == pkv.api.EINVAL       # misaligned
    assert _decode(lib, d, k_new=FAKE) == pkv.api.EINVAL                       # k_new without v_new
    assert _decode(lib, d, scale=float("nan")) == pkv.api.EINVAL
    assert _decode(lib, d, ws=None) == pkv.api.EWORKSPACE
    assert _decode(lib, d, ws_bytes=16) == pkv.api.EWORKSPACE
    assert _decode(lib, d, batch=0) == pkv.api.OK                              # nothing to do
    assert _decode(lib, d, batch=2000) == pkv.api.EUNSUPPORTED


def test_decode_flags():
    lib = _lib.load()
    d = CacheDesc(64, 16, 2, 128, 0)
    args = (ctypes.byref(d), FAKE, FAKE, FAKE, None, None, FAKE, 4, FAKE, 0, 8, 0.1, FAKE, None, FAKE, 1 << 30,
            None, None)
    assert lib.pkv_decode_attn_ex(*args, pkv.api.DECODE_OVERLAP_PROLOGUE) == pkv.api.OK
    assert lib.pkv_decode_attn_ex(*args, pkv.api.DECODE_OVERLAP_PROLOGUE | pkv.api.DECODE_EARLY_KV) == pkv.api.OK
    assert lib.pkv_decode_attn_ex(*args, pkv.api.DECODE_EARLY_KV) == pkv.api.EINVAL  # needs the overlap launch
    assert lib.pkv_decode_attn_ex(*args, 16) == pkv.api.EINVAL                       # unknown flag
    for f in (pkv.api.DECODE_MAKE_PLAN, pkv.api.DECODE_USE_PLAN,
              pkv.api.DECODE_USE_PLAN | pkv.api.DECODE_OVERLAP_PROLOGUE | pkv.api.DECODE_EARLY_KV):
        assert lib.pkv_decode_attn_ex(*args, f) == pkv.api.OK
    assert lib.pkv_decode_attn_ex(*args, pkv.api.DECODE_MAKE_PLAN | pkv.api.DECODE_USE_PLAN) == pkv.api.EINVAL


def test_decode_workspace_holds_a_step_plan():
    """The decode workspace ends with room for one step plan: a 256-byte
    header, the per-row arrays and a 256-byte record per persistent CTA (at
    most 2048), whatever the sizes."""
    d = CacheDesc(64, 128, 8, 128, 0)
    for batch in (1, 64, 1024):
        plan = 256 + 256 * ((4 * batch + 255) // 256) + 256 * ((4 * (batch + 1) + 255) // 256) + \
            256 * ((8 * (batch + 1) + 255) // 256) + 2048 * 256
        # before it: a ticket per (row, kv head), then (m, l) and o partials of 4 heads
        # for two slots of each of 2048 persistent CTAs
        al = lambda x: 256 * ((x + 255) // 256)  # noqa: E731
        base = al(4 * batch * 8) + al(8 * 4096 * 4) + al(4 * 4096 * 4 * 128)
        assert pkv.pkv_decode_workspace_size(batch, 9, 32, d) == base + plan


def test_append_argument_errors():
    lib = _lib.load()
    d = CacheDesc(64, 16, 2, 128, 0)

    def app(desc=d, k_new=FAKE, ntok=4, indptr=None, batch=4):
        return lib.pkv_append(ctypes.byref(desc), FAKE, FAKE, k_new, FAKE, ntok, indptr, FAKE, 4, FAKE, batch,
                              None, None)

    assert app(ntok=3) == pkv.api.EINVAL            # one token per row without indptr
    assert app(k_new=None) == pkv.api.EINVAL
    assert app(k_new=ctypes.c_void_p(0x10004)) == pkv.api.EINVAL
    assert app(desc=CacheDesc(64, 16, 2, 100, 0)) == pkv.api.EUNSUPPORTED
    assert app(batch=0, ntok=0) == pkv.api.OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    big = CacheDesc(64, 16, 8, 256, 0)  # head_dim 256, 8 query heads per kv head: > 16 MiB of scratch
    assert pkv.pkv_decode_workspace_size(4, 4, 64, big) > (16 << 20)
    st = lib.pkv_decode_attn_noalloc(ctypes.byref(big), FAKE, FAKE, FAKE, None, None, FAKE, 4, FAKE, 4, 64, 0.1,
                                     FAKE, None, None, None)
    assert st == pkv.api.ETOOBIG
    small = CacheDesc(64, 16, 8, 128, 0)
    assert pkv.pkv_decode_workspace_size(1024, 65, 32, small) <= (16 << 20)
    st = lib.pkv_decode_attn_noalloc(ctypes.byref(small), FAKE, FAKE, FAKE, None, None, FAKE, 4, FAKE, 4, 6 * 8, 0.1,
                                     FAKE, None, None, None)
    assert st == pkv.api.EUNSUPPORTED  # argument errors are those of pkv_decode_attn
    # an invalid call that is also too big gets the argument error, not ETOOBIG
    for args in ((None, FAKE), (FAKE, ctypes.c_void_p(0x10004))):  # null q; misaligned out
        q, out = args
        st = lib.pkv_decode_attn_noalloc(ctypes.byref(big), FAKE, FAKE, q, None, None, FAKE, 4, FAKE, 4, 64, 0.1,
                                         out, None, None, None)
        assert st == pkv.api.EINVAL
    st = lib.pkv_decode_attn_noalloc(ctypes.byref(big), FAKE, FAKE, FAKE, None, None, FAKE, 4, FAKE, 4, 64,
                                     float("nan"), FAKE, None, None, None)
    assert st == pkv.api.EINVAL
    st = lib.pkv_decode_attn_noalloc(ctypes.byref(big), FAKE, FAKE, FAKE, None, None, FAKE, 4, FAKE, 0, 64, 0.1,
                                     FAKE, None, None, None)
    assert st == pkv.api.OK  # an empty batch is valid and launches nothing


def _prefill(lib, desc, batch=2, hq=8, total_q=40, ws=FAKE, ws_bytes=1 << 30, q=FAKE, scale=0.1, max_blocks=4):
    return lib.pkv_prefill_attn(ctypes.byref(desc), FAKE, FAKE, q, FAKE, FAKE, FAKE, max_blocks, batch, hq, total_q,
                                scale, FAKE, None, ws, ws_bytes, None, None)


def test_prefill_workspace_size():
    d = CacheDesc(4096, 16, 6, 256, 1)
    n = pkv.pkv_prefill_workspace_size(8, 4352, 48, d)
    # plan header + one 32-byte record per (request, query tile): 4352/16 + 8 tiles at most
    assert n == 256 + ((4352 // 16 + 8) * 32 + 255) // 256 * 256
    assert pkv.pkv_prefill_workspace_size(8, 4352, 6 * 6, d) == 0         # group 6: not a power of two
    assert pkv.pkv_prefill_workspace_size(8, 4352, 6 * 256, d) == 0       # group above 128
    assert pkv.pkv_prefill_workspace_size(1025, 4352, 48, d) == 0
    assert pkv.pkv_prefill_workspace_size(8, 4352, 48, CacheDesc(4096, 4, 6, 256, 1)) == 0  # page 4


def test_prefill_argument_errors_return_before_any_launch():
    lib = _lib.load()
    d = CacheDesc(64, 16, 2, 128, 1)
    assert _prefill(lib, CacheDesc(64, 16, 2, 96, 1)) == pkv.api.EUNSUPPORTED   # head dim
    assert _prefill(lib, CacheDesc(64, 4, 2, 128, 1)) == pkv.api.EUNSUPPORTED   # page below 8
    assert _prefill(lib, d, hq=7) == pkv.api.EINVAL                             # Hq % Hkv
    assert _prefill(lib, d, hq=6) == pkv.api.EUNSUPPORTED                       # group 3
    assert _prefill(lib, d, q=None) == pkv.api.EINVAL
    assert _prefill(lib, d, q=ctypes.c_void_p(0x10008)) == pkv.api.EINVAL        # misaligned
    assert _prefill(lib, d, scale=float("inf")) == pkv.api.EINVAL
    assert _prefill(lib, d, ws=None) == pkv.api.EWORKSPACE
    assert _prefill(lib, d, ws_bytes=16) == pkv.api.EWORKSPACE
    assert _prefill(lib, d, batch=0) == pkv.api.OK
    assert _prefill(lib, d, total_q=0) == pkv.api.OK
    assert _prefill(lib, d, batch=1025) == pkv.api.EUNSUPPORTED
    assert _prefill(lib, d, total_q=-1) == pkv.api.EINVAL


def test_decode_bucket():
    lib = _lib.load()
    assert [lib.pkv_decode_bucket(b) for b in (1, 8, 9, 16, 17, 64, 65, 1000, 1024)] == \
        [8, 8, 16, 16, 32, 64, 128, 1024, 1024]
    assert lib.pkv_decode_bucket(0) == 0 and lib.pkv_decode_bucket(1025) == 0


def test_decode_step_argument_errors_before_any_cuda_call():
    lib = _lib.load()
    d = CacheDesc(64, 16, 2, 128, 0)
    arr = ctypes.c_void_p * 2
    two = arr(0x10000, 0x10000)
    out = ctypes.c_void_p()

    def create(desc=d, layers=2, k=two, q=two, o=two, ws=FAKE, ws_bytes=1 << 30, batch=4, hq=8, flags=0, handle=True):
        return lib.pkv_decode_step_create(ctypes.byref(desc), layers, k, k, q, None, None, FAKE, 4, FAKE, batch, hq,
                                          0.1, o, None, ws, ws_bytes, None, flags,
                                          ctypes.byref(out) if handle else None)

    assert create(handle=False) == pkv.api.EINVAL
    assert create(layers=0) == pkv.api.EINVAL
    assert create(k=None) == pkv.api.EINVAL
    assert create(q=arr(0x10000, 0)) == pkv.api.EINVAL                    # a missing layer pointer
    assert create(q=arr(0x10000, 0x10008)) == pkv.api.EINVAL              # misaligned
    assert create(desc=CacheDesc(64, 16, 2, 96, 0)) == pkv.api.EUNSUPPORTED
    assert create(hq=6) == pkv.api.EUNSUPPORTED
    assert create(ws=None) == pkv.api.EWORKSPACE
    assert create(ws_bytes=64) == pkv.api.EWORKSPACE
    assert create(flags=pkv.api.DECODE_EARLY_KV) == pkv.api.EINVAL
    assert create(flags=pkv.api.DECODE_MAKE_PLAN) == pkv.api.EINVAL       # the step makes its own plan
    assert out.value is None
    lib.pkv_decode_step_destroy(None)


def _mixed(lib, desc, batch=2, hq=8, total_q=40, max_qlen=32, dq=4, ws=FAKE, ws_bytes=1 << 30, q=FAKE,
           k_new=FAKE, v_new=FAKE, scale=0.1, max_blocks=4, qo=FAKE):
    return lib.pkv_mixed_attn(ctypes.byref(desc), FAKE, FAKE, q, k_new, v_new, qo, FAKE, max_blocks, FAKE, batch, hq,
                              total_q, max_qlen, dq, scale, FAKE, None, ws, ws_bytes, None, None)


def test_mixed_workspace_size():
    d = CacheDesc(65536, 16, 8, 128, 0)
    decode_only = pkv.pkv_mixed_workspace_size(64, 256, 65, 32, 4, 4, d)
    with_prefill = pkv.pkv_mixed_workspace_size(64, 256, 65, 32, 512, 4, d)
    assert 0 < decode_only < with_prefill
    # the decode part: 16 (query, head) columns per unit once G * q > 8
    # (partials 16 columns wide, two combine tickets per unit)
    assert decode_only >= pkv.pkv_decode_workspace_size(64, 65, 32, d)
    eight_cols = pkv.pkv_mixed_workspace_size(64, 256, 65, 32, 2, 2, d)
    assert 0 < eight_cols < decode_only
    # every head_dim has 16-column multi-query kernels: shapes of 9..32 columns per kv head are accepted
    for D in (64, 128, 256):
        dd = CacheDesc(65536, 16, 8, D, 0)
        for hq, dq in ((32, 3), (32, 4), (64, 2), (128, 1), (16, 8), (32, 8)):
            assert pkv.pkv_mixed_workspace_size(64, 256, 65, hq, dq, dq, dd) > 0, (D, hq, dq)
    assert pkv.pkv_mixed_workspace_size(64, 256, 65, 32, 0, 4, d) == 0        # max_qlen < 1
    assert pkv.pkv_mixed_workspace_size(64, 256, 65, 32, 4, 0, d) == 0        # decode_max_qlen < 1
    assert pkv.pkv_mixed_workspace_size(1025, 256, 65, 32, 4, 4, d) == 0
    assert pkv.pkv_mixed_workspace_size(64, 1 << 26, 65, 32, 4, 4, d) == 0    # total_q * Hq >= 2^31
    d4 = CacheDesc(65536, 4, 8, 128, 0)
    assert pkv.pkv_mixed_workspace_size(64, 256, 65, 32, 4, 4, d4) > 0        # decode only: any page size
    assert pkv.pkv_mixed_workspace_size(64, 256, 65, 32, 8, 4, d4) == 0       # prefill needs page >= 8


def test_mixed_argument_errors_return_before_any_launch():
    lib = _lib.load()
    d = CacheDesc(64, 16, 2, 128, 1)
    assert _mixed(lib, CacheDesc(64, 16, 2, 96, 1)) == pkv.api.EUNSUPPORTED   # head dim
    assert _mixed(lib, CacheDesc(64, 4, 2, 128, 1)) == pkv.api.EUNSUPPORTED   # prefill rows, page 4
    assert _mixed(lib, d, hq=7) == pkv.api.EINVAL                             # Hq % Hkv
    assert _mixed(lib, d, hq=6) == pkv.api.EUNSUPPORTED                       # group 3
    assert _mixed(lib, d, max_qlen=0) == pkv.api.EINVAL
    assert _mixed(lib, d, dq=0) == pkv.api.EINVAL
    assert _mixed(lib, d, q=None) == pkv.api.EINVAL
    assert _mixed(lib, d, qo=None) == pkv.api.EINVAL
    assert _mixed(lib, d, k_new=None) == pkv.api.EINVAL                       # one of the pair
    assert _mixed(lib, d, q=ctypes.c_void_p(0x10008)) == pkv.api.EINVAL        # misaligned
    assert _mixed(lib, d, scale=float("nan")) == pkv.api.EINVAL
    assert _mixed(lib, d, ws=None) == pkv.api.EWORKSPACE
    assert _mixed(lib, d, ws_bytes=16) == pkv.api.EWORKSPACE
    assert _mixed(lib, d, batch=0) == pkv.api.OK
    assert _mixed(lib, d, batch=1025) == pkv.api.EUNSUPPORTED
    assert _mixed(lib, d, total_q=-1) == pkv.api.EINVAL


def test_default_decode_max_qlen():
    assert pkv.default_decode_max_qlen(32, 8) == 4   # Qwen3: 4 queries x 4 heads = 16 columns
    assert pkv.default_decode_max_qlen(48, 6) == 2
    assert pkv.default_decode_max_qlen(8, 8) == 16
    assert pkv.default_decode_max_qlen(128, 1) == 1
