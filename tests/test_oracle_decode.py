"""Pins for the fp64 oracle's append + decode attention (CPU only).

Each test ties the oracle to something other than itself:
* torch's fp64 scaled_dot_product_attention on a dense gather (a library
  routine that the paged problem reduces to once tokens are laid out in
  logical order), and torch.logsumexp for lse;
* closed forms: scale 0 gives the mean of V; constant V rows give that row;
  a single key gives V exactly;
* invariances: renumbering physical pages changes no output bit;
* the append definition: the only bytes that change are the new token's
  slot, which then holds k_new / v_new bit for bit.
"""
import hashlib
import math

import numpy as np
import pytest
import torch

from paged_kv_decode_append_gb300 import workloads as wl


def _desc(oracle, case):
    return oracle.CacheDesc(case.num_pages, case.page_size, case.num_kv_heads, case.head_dim, case.layout)


def _pool_tokens(pool_bits, layout, page, slot):
    """[Hkv, D] bits of one token (numpy indexing, independent of the oracle)."""
    if layout == wl.NHD:
        return pool_bits[page, slot]
    return pool_bits[page, :, slot]


def _dense(case, k_bits, v_bits, b, n):
    ks = [_pool_tokens(k_bits, case.layout, case.block_table[b, t // case.page_size], t % case.page_size)
          for t in range(n)]
    vs = [_pool_tokens(v_bits, case.layout, case.block_table[b, t // case.page_size], t % case.page_size)
          for t in range(n)]
    shape = (0, case.num_kv_heads, case.head_dim)
    if n == 0:
        return np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    return np.stack(ks), np.stack(vs)  # [n, Hkv, D] bits


def _sdpa(q_bits, k_bits, v_bits, group, scale):
    """q [Hq, D], k/v [n, Hkv, D] bits -> out [Hq, D], lse [Hq] in fp64 via torch."""
    q = torch.from_numpy(wl_f64(q_bits))[None, :, None, :]  # [1, Hq, 1, D]
    k = torch.from_numpy(wl_f64(k_bits)).permute(1, 0, 2).repeat_interleave(group, 0)[None]
    v = torch.from_numpy(wl_f64(v_bits)).permute(1, 0, 2).repeat_interleave(group, 0)[None]
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)[0, :, 0]
    s = (q[0, :, 0, None, :] * k[0]).sum(-1) * scale  # [Hq, n]
    return out.numpy(), torch.logsumexp(s, dim=-1).numpy()


def wl_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _run_decode(oracle, case, with_new=True, scale=None, sel=None):
    k = wl.bits(case.k_cache).copy()
    v = wl.bits(case.v_cache).copy()
    out, lse, err, err_rows = oracle.decode(
        _desc(oracle, case), k, v, wl.bits(case.q),
        wl.bits(case.k_new) if with_new else None, wl.bits(case.v_new) if with_new else None,
        case.block_table, case.cache_seqlens, case.softmax_scale if scale is None else scale, sel=sel)
    return out, lse, err, k, v


@pytest.mark.parametrize("with_new", [True, False])
def test_tiny_matches_sdpa_on_dense_gather(oracle_mod, with_new):
    case = wl.tiny()
    out, lse, err, _, _ = _run_decode(oracle_mod, case, with_new)
    assert err == 0
    k0, v0 = wl.bits(case.k_cache), wl.bits(case.v_cache)
    q = wl.bits(case.q)
    for b in range(case.batch):
        L = int(case.cache_seqlens[b])
        kd, vd = _dense(case, k0, v0, b, L)
        if with_new:  # append then attend: the new token is logical position L
            kd = np.concatenate([kd, wl.bits(case.k_new)[b][None]])
            vd = np.concatenate([vd, wl.bits(case.v_new)[b][None]])
        if kd.shape[0] == 0:
            assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
            continue
        ref, ref_lse = _sdpa(q[b], kd, vd, case.group, case.softmax_scale)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-12, atol=1e-12)


def _random_case(seed, B, Hq, Hkv, D, P, layout, lens, extra_pages=5):
    g = torch.Generator().manual_seed(seed)
    lens = np.asarray(lens, np.int32)
    needed = (np.maximum(lens, 0) + 1 + P - 1) // P
    NP = int(needed.sum()) + 1 + extra_pages
    max_blocks = int(needed.max()) + 1
    order = (torch.randperm(NP - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = wl.assign_pages(needed, NP, max_blocks, order)
    case = wl.PagedCase("rand", B, Hq, Hkv, D, P, NP, layout, max_blocks, bt, lens, 1.0 / math.sqrt(D),
                        q=wl._randn_bf16((B, Hq, D), g, "cpu"))
    case.k_new = wl._randn_bf16((B, Hkv, D), g, "cpu")
    case.v_new = wl._randn_bf16((B, Hkv, D), g, "cpu")
    wl._fill_cache(case, g, "cpu", "cpu")
    return case


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("Hq,Hkv,D,P", [(8, 1, 32, 4), (6, 6, 16, 8), (16, 2, 128, 32), (4, 2, 256, 1)])
def test_shapes_match_sdpa(oracle_mod, layout, Hq, Hkv, D, P):
    case = _random_case(11 + D + P, 3, Hq, Hkv, D, P, layout, [0, 5, 37])
    out, lse, err, _, _ = _run_decode(oracle_mod, case)
    assert err == 0
    k0, v0 = wl.bits(case.k_cache), wl.bits(case.v_cache)
    for b in range(3):
        L = int(case.cache_seqlens[b])
        kd, vd = _dense(case, k0, v0, b, L)
        kd = np.concatenate([kd, wl.bits(case.k_new)[b][None]])
        vd = np.concatenate([vd, wl.bits(case.v_new)[b][None]])
        ref, ref_lse = _sdpa(wl.bits(case.q)[b], kd, vd, case.group, case.softmax_scale)
        np.testing.assert_allclose(out[b], ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=1e-12, atol=1e-12)


def test_scale_zero_gives_mean_of_values(oracle_mod):
    case = wl.tiny()
    out, lse, _, _, _ = _run_decode(oracle_mod, case, scale=0.0)
    k0, v0 = wl.bits(case.k_cache), wl.bits(case.v_cache)
    for b in range(case.batch):
        L = int(case.cache_seqlens[b])
        _, vd = _dense(case, k0, v0, b, L)
        vd = np.concatenate([vd, wl.bits(case.v_new)[b][None]])
        mean = wl_f64(vd).mean(axis=0)  # [Hkv, D]
        for h in range(case.num_q_heads):
            np.testing.assert_allclose(out[b, h], mean[h // case.group], rtol=1e-13, atol=1e-14)
            assert lse[b, h] == pytest.approx(math.log(L + 1), rel=1e-14)


def test_constant_values_give_that_row(oracle_mod):
    case = wl.tiny()
    row = wl.bits(case.v_new)[0, 0].copy()  # one bf16 row, used for every V
    v = wl.bits(case.v_cache).copy()
    live = ~np.isnan(wl_f64(v))
    v[live] = np.broadcast_to(row, v.shape)[live]
    case.v_cache = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16)
    case.v_new = torch.from_numpy(np.broadcast_to(row, wl.bits(case.v_new).shape).copy().view(np.int16)).view(torch.bfloat16)
    out, _, _, _, _ = _run_decode(oracle_mod, case)
    for b in range(case.batch):
        for h in range(case.num_q_heads):
            np.testing.assert_allclose(out[b, h], wl_f64(row), rtol=1e-14, atol=0)


def test_single_key_returns_value_exactly(oracle_mod):
    case = wl.tiny()
    case.cache_seqlens = np.zeros(case.batch, np.int32)  # L=0: only the appended token
    out, lse, err, _, _ = _run_decode(oracle_mod, case)
    assert err == 0
    vn = wl_f64(wl.bits(case.v_new))
    for h in range(case.num_q_heads):
        assert np.array_equal(out[:, h], vn[:, h // case.group])
    assert np.all(lse == 0.0) or np.allclose(lse, np.einsum(
        "bhd,bhd->bh", wl_f64(wl.bits(case.q)),
        np.repeat(wl_f64(wl.bits(case.k_new)), case.group, axis=1)) * case.softmax_scale, rtol=1e-13)


def test_page_permutation_is_bit_invariant(oracle_mod):
    case = wl.tiny()
    out0, lse0, _, _, _ = _run_decode(oracle_mod, case)
    g = torch.Generator().manual_seed(99)
    perm = np.concatenate([[0], torch.randperm(case.num_pages - 1, generator=g).numpy() + 1])
    k, v = wl.bits(case.k_cache), wl.bits(case.v_cache)
    k2, v2 = np.empty_like(k), np.empty_like(v)
    k2[perm], v2[perm] = k, v  # physical page p moves to perm[p]
    case.block_table = np.where(case.block_table > 0, perm[case.block_table], 0).astype(np.int32)
    case.k_cache = torch.from_numpy(k2.view(np.int16)).view(torch.bfloat16)
    case.v_cache = torch.from_numpy(v2.view(np.int16)).view(torch.bfloat16)
    out1, lse1, _, _, _ = _run_decode(oracle_mod, case)
    assert out0.tobytes() == out1.tobytes()
    assert lse0.tobytes() == lse1.tobytes()


def test_append_changes_only_the_new_slot(oracle_mod):
    case = wl.tiny()
    before_k, before_v = wl.bits(case.k_cache), wl.bits(case.v_cache)
    _, _, _, k, v = _run_decode(oracle_mod, case)
    kn, vn = wl.bits(case.k_new), wl.bits(case.v_new)
    changed = np.argwhere(np.any(k != before_k, axis=-1))  # (page, slot, head)
    assert len(changed) == case.batch * case.num_kv_heads
    # every changed (page, slot) was a NaN slot and now holds exactly one row's new token
    seen = set()
    for page, slot, h in changed:
        assert np.all(np.isnan(wl_f64(before_k[page, slot, h])))
        b = [r for r in range(case.batch) if page in case.block_table[r]][0]
        assert np.array_equal(k[page, slot, h], kn[b, h])
        assert np.array_equal(v[page, slot, h], vn[b, h])
        seen.add((b, h))
    assert len(seen) == case.batch * case.num_kv_heads
    mask = np.ones(k.shape[:3], bool)
    mask[tuple(changed.T)] = False
    assert hashlib.sha256(k[mask].tobytes()).digest() == hashlib.sha256(before_k[mask].tobytes()).digest()
    assert hashlib.sha256(v[mask].tobytes()).digest() == hashlib.sha256(before_v[mask].tobytes()).digest()


def test_standalone_append_with_indptr(oracle_mod):
    case = _random_case(5, 3, 4, 2, 16, 4, 0, [3, 0, 9], extra_pages=8)
    n_new = np.array([2, 5, 1], np.int32)
    indptr = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    needed = (case.cache_seqlens + n_new + case.page_size - 1) // case.page_size
    assert np.all(needed <= case.max_blocks)
    # give row 1 the extra pages it needs beyond the single-token reservation
    free = sorted(set(range(1, case.num_pages)) - set(case.block_table.ravel().tolist()))
    for b in range(3):
        for j in range(case.max_blocks):
            if j < needed[b] and case.block_table[b, j] == 0:
                case.block_table[b, j] = free.pop(0)
    g = torch.Generator().manual_seed(3)
    kn = wl.bits(wl._randn_bf16((int(indptr[-1]), 2, 16), g, "cpu"))
    vn = wl.bits(wl._randn_bf16((int(indptr[-1]), 2, 16), g, "cpu"))
    k, v = wl.bits(case.k_cache).copy(), wl.bits(case.v_cache).copy()
    err, _ = oracle_mod.append(_desc(oracle_mod, case), k, v, kn, vn, indptr, case.block_table,
                               case.cache_seqlens)
    assert err == 0
    for b in range(3):
        for i in range(n_new[b]):
            t = int(case.cache_seqlens[b]) + i
            page, slot = case.block_table[b, t // 4], t % 4
            assert np.array_equal(k[page, slot], kn[indptr[b] + i])
            assert np.array_equal(v[page, slot], vn[indptr[b] + i])
    n_changed = np.count_nonzero(np.any(k != wl.bits(case.k_cache), axis=-1))
    assert n_changed == int(indptr[-1]) * 2


def test_inactive_and_empty_rows(oracle_mod):
    case = wl.tiny()
    case.cache_seqlens = np.array([-1, 0, 1, -7], np.int32)  # row 2 keeps its one cached token
    before = wl.bits(case.k_cache).copy()
    out, lse, err, k, _ = _run_decode(oracle_mod, case, with_new=False)
    assert err == 0
    for b in (0, 1, 3):  # inactive, and empty attend-only row: out 0, lse -inf, never NaN
        assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
    assert np.all(np.isfinite(out[2]))
    out2, lse2, err2, k2, _ = _run_decode(oracle_mod, case, with_new=True)
    assert np.all(out2[0] == 0) and np.all(out2[3] == 0)
    changed = np.count_nonzero(np.any(k2 != before, axis=-1))
    assert changed == 2 * case.num_kv_heads  # rows 1 and 2 only
    assert np.array_equal(out2[1], np.repeat(wl_f64(wl.bits(case.v_new))[1], case.group, axis=0))


def test_bad_pages_zero_the_row_and_flag(oracle_mod):
    case = wl.tiny()
    case.block_table = case.block_table.copy()
    case.block_table[1, 1] = 0  # null page used by a live token
    case.block_table[2, 0] = case.num_pages  # out of range
    before = wl.bits(case.k_cache).copy()
    out, lse, err, k, _ = _run_decode(oracle_mod, case)
    assert err == oracle_mod.ERR_PAGE
    for b in (1, 2):
        assert np.all(out[b] == 0) and np.all(np.isneginf(lse[b]))
    assert np.all(np.isfinite(out[0])) and np.all(np.isfinite(out[3]))
    changed = np.count_nonzero(np.any(k != before, axis=-1))
    assert changed == 2 * case.num_kv_heads  # rows 0 and 3 appended, 1 and 2 dropped


def test_overflow_row_flags(oracle_mod):
    case = wl.tiny()
    case.cache_seqlens = case.cache_seqlens.copy()
    case.cache_seqlens[3] = case.max_blocks * case.page_size  # L+1 does not fit
    out, lse, err, _, _ = _run_decode(oracle_mod, case)
    assert err == oracle_mod.ERR_OVERFLOW
    assert np.all(out[3] == 0) and np.all(np.isneginf(lse[3]))


def test_selection_matches_full(oracle_mod):
    case = wl.tiny()
    full, full_lse, _, _, _ = _run_decode(oracle_mod, case)
    sel = [(0, 3), (2, 1), (3, 0)]
    part, part_lse, _, _, _ = _run_decode(oracle_mod, case, sel=sel)
    for b, h in sel:
        assert np.array_equal(part[b, h], full[b, h]) and part_lse[b, h] == full_lse[b, h]
    assert np.isnan(part[1]).all()


def test_threads_do_not_change_bits(oracle_mod):
    case = wl.tiny()
    k, v = wl.bits(case.k_cache).copy(), wl.bits(case.v_cache).copy()
    args = (wl.bits(case.q), wl.bits(case.k_new), wl.bits(case.v_new), case.block_table, case.cache_seqlens,
            case.softmax_scale)
    d = _desc(oracle_mod, case)
    o1, l1, _, _ = oracle_mod.decode(d, k.copy(), v.copy(), *args, nthreads=1)
    o4, l4, _, _ = oracle_mod.decode(d, k.copy(), v.copy(), *args, nthreads=4)
    assert o1.tobytes() == o4.tobytes() and l1.tobytes() == l4.tobytes()


def test_standalone_append_checks_only_destination_pages(oracle_mod):
    case = wl.tiny()
    case.block_table = case.block_table.copy()
    case.block_table[3, 0] = 0  # a page row 3 reads, but an append at 64 does not touch
    k = wl.bits(case.k_cache).copy()
    v = wl.bits(case.v_cache).copy()
    d = _desc(oracle_mod, case)
    err, err_rows = oracle_mod.append(d, k, v, wl.bits(case.k_new), wl.bits(case.v_new), None,
                                      case.block_table, case.cache_seqlens)
    assert err == 0
    page = case.block_table[3, 64 // case.page_size]
    assert np.array_equal(k[page, 0], wl.bits(case.k_new)[3])
    case.block_table[3, 64 // case.page_size] = case.num_pages + 3  # now the destination is bad
    k2 = wl.bits(case.k_cache).copy()
    err, err_rows = oracle_mod.append(d, k2, v.copy(), wl.bits(case.k_new), wl.bits(case.v_new), None,
                                      case.block_table, case.cache_seqlens)
    assert err == oracle_mod.ERR_PAGE and list(err_rows) == [0, 0, 0, oracle_mod.ERR_PAGE]
    assert np.array_equal(k2[page], wl.bits(case.k_cache)[page])  # row 3 wrote nothing
