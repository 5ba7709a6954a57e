"""GPU parity of the standalone append (pkv_append) with the fp64 oracle's
append: the whole pools must be bit-identical afterwards (sha256), and the
error flag must match the oracle's error bits."""
import hashlib
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_append_gb300 as pkv
from paged_kv_decode_append_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _sha(a) -> str:
    if isinstance(a, torch.Tensor):
        a = wl.bits(a)
    return hashlib.sha256(a.tobytes()).hexdigest()


def _case(seed, B, Hkv, D, P, lens, n_new, layout, spare=6):
    g = torch.Generator().manual_seed(seed)
    lens = np.asarray(lens, np.int32)
    n_new = np.asarray(n_new, np.int32)
    needed = (np.maximum(lens, 0) + n_new + P - 1) // P
    NP = int(needed.sum()) + 1 + spare
    max_blocks = int(needed.max()) + 1
    order = (torch.randperm(NP - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = wl.assign_pages(needed, NP, max_blocks, order)
    case = wl.PagedCase("append", B, Hkv, Hkv, D, P, NP, layout, max_blocks, bt, lens, 1.0 / math.sqrt(D),
                        q=torch.empty(0))
    wl._fill_cache(case, g, DEV, "cpu")
    indptr = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    T = int(indptr[-1])
    kn = wl._randn_bf16((T, Hkv, D), g, "cpu").to(DEV)
    vn = wl._randn_bf16((T, Hkv, D), g, "cpu").to(DEV)
    return case, indptr, kn, vn


def _check(case, indptr, kn, vn, use_indptr=True):
    k_ref, v_ref = wl.bits(case.k_cache).copy(), wl.bits(case.v_cache).copy()
    d = oracle.CacheDesc(case.num_pages, case.page_size, case.num_kv_heads, case.head_dim, case.layout)
    ref_err, _ = oracle.append(d, k_ref, v_ref, wl.bits(kn), wl.bits(vn), indptr if use_indptr else None,
                               case.block_table, case.cache_seqlens)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.pkv_append(case.k_cache, case.v_cache, kn, vn, torch.as_tensor(case.block_table, device=DEV),
                   torch.as_tensor(case.cache_seqlens, device=DEV),
                   append_indptr=torch.as_tensor(indptr, device=DEV) if use_indptr else None, err_flag=err,
                   layout=case.layout)
    torch.cuda.synchronize()
    assert int(err.item()) == ref_err
    assert _sha(case.k_cache) == _sha(k_ref)
    assert _sha(case.v_cache) == _sha(v_ref)
    return ref_err


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
@pytest.mark.parametrize("Hkv,D,P", [(8, 128, 16), (8, 128, 128), (2, 64, 1), (6, 256, 16), (1, 64, 32)])
def test_one_token_per_row(layout, Hkv, D, P):
    lens = [0, 1, 15, 16, 17, 100, -1, 255]
    case, indptr, kn, vn = _case(7 + D + P, len(lens), Hkv, D, P, lens, [1] * len(lens), layout)
    assert _check(case, indptr, kn, vn, use_indptr=False) == 0


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
def test_ragged_multi_token(layout):
    lens = [0, 5, 31, 64, -1, 1000]
    n_new = [40, 1, 33, 0, 7, 1023]  # a prefill-sized append crosses many pages
    case, indptr, kn, vn = _case(11, len(lens), 6, 256, 16, lens, n_new, layout)
    assert _check(case, indptr, kn, vn) == 0


def test_bad_destination_pages_drop_the_row():
    lens = [3, 20, 40]
    case, indptr, kn, vn = _case(13, 3, 2, 64, 16, lens, [2, 20, 1], wl.NHD)
    case.block_table = case.block_table.copy()
    case.block_table[1, 2] = 0                 # a page row 1 writes into
    case.block_table[2, 0] = case.num_pages    # a page row 2 reads but an append at 40 does not touch
    assert _check(case, indptr, kn, vn) == oracle.ERR_PAGE


def test_overflow_drops_the_row():
    case, indptr, kn, vn = _case(17, 2, 2, 64, 16, [10, 20], [3, 4], wl.NHD)
    case.cache_seqlens = case.cache_seqlens.copy()
    case.cache_seqlens[0] = case.max_blocks * case.page_size - 2  # 3 new tokens do not fit
    assert _check(case, indptr, kn, vn) == oracle.ERR_OVERFLOW


def test_pool_helpers_feed_the_append():
    """Pages from the host pool (reserve / release) route the append."""
    P, Hkv, D = 16, 2, 64
    pool = pkv.PagePool(64)
    pool.shuffle(3)
    bt = np.zeros((3, 8), np.int32)
    lens = np.array([0, 17, 40], np.int32)
    n_new = np.array([5, 20, 1], np.int32)
    for b in range(3):
        pool.reserve(bt[b], P, 0, int(lens[b] + n_new[b]))
    g = torch.Generator().manual_seed(5)
    case = wl.PagedCase("pool", 3, Hkv, Hkv, D, P, 64, wl.NHD, 8, bt, lens, 0.125, q=torch.empty(0))
    wl._fill_cache(case, g, DEV, "cpu")
    indptr = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    kn = wl._randn_bf16((int(indptr[-1]), Hkv, D), g, "cpu").to(DEV)
    vn = wl._randn_bf16((int(indptr[-1]), Hkv, D), g, "cpu").to(DEV)
    assert pkv.pkv_validate_host(pkv.api.CacheDesc(64, P, Hkv, D, 0), bt, lens, 0)[0] == 0
    assert _check(case, indptr, kn, vn) == 0
    for b in range(3):
        pool.release(bt[b], P, int(lens[b] + n_new[b]))
    assert pool.num_free == 63
