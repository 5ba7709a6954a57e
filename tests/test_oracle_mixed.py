"""Pins for the fp64 oracle's mixed step (CPU only): chunked prefill rows,
multi-token decode rows and single-token decode rows in one batch.

Each test ties ``oracle.mixed`` to something other than itself:
* torch's fp64 scaled_dot_product_attention (is_causal) on a dense gather
  that numpy builds from the ORIGINAL pool plus the new tokens: query i of a
  row with q new tokens over kv keys is row kv - q + i of a kv x kv causal
  problem (end alignment, FlashInfer page, code analysis part 1);
  torch.logsumexp under the same mask for lse;
* the append definition: after the call the pool equals a numpy scatter of
  k_new / v_new into slots L .. L+q-1, bit for bit, and nothing else moved;
* closed forms: one new token on an empty cache returns v_new exactly with
  lse = scale * q.k; a first chunk (L = 0) is plain causal attention;
* the row fates of the interface (inactive, too long, reversed range, bad
  page, overflow).
"""
import math

import numpy as np
import pytest
import torch

from paged_kv_decode_append_gb300 import workloads as wl


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _desc(oracle, case):
    return oracle.CacheDesc(case.num_pages, case.page_size, case.num_kv_heads, case.head_dim, case.layout)


def _run(oracle, case, with_new=True, max_qlen=None, sel=None, k=None, v=None):
    k = wl.bits(case.k_cache).copy() if k is None else k
    v = wl.bits(case.v_cache).copy() if v is None else v
    out, lse, err, rows = oracle.mixed(_desc(oracle, case), k, v, wl.bits(case.q),
                                       wl.bits(case.k_new) if with_new else None,
                                       wl.bits(case.v_new) if with_new else None, case.qo_indptr,
                                       case.block_table, case.cache_seqlens, case.softmax_scale,
                                       max_qlen=max_qlen, sel=sel)
    return out, lse, err, rows, k, v


def _token(pool, layout, page, slot):
    return pool[page, slot] if layout == wl.NHD else pool[page, :, slot]


def _dense(case, b, with_new):
    """[kv, Hkv, D] bits of row b's keys and values in logical order: cached
    tokens gathered by numpy from the original pools, then the new tokens."""
    L = int(case.cache_seqlens[b])
    kp, vp = wl.bits(case.k_cache), wl.bits(case.v_cache)
    ks = [_token(kp, case.layout, case.block_table[b, t // case.page_size], t % case.page_size) for t in range(L)]
    vs = [_token(vp, case.layout, case.block_table[b, t // case.page_size], t % case.page_size) for t in range(L)]
    lo, hi = case.qo_indptr[b], case.qo_indptr[b + 1]
    if with_new:
        ks += list(wl.bits(case.k_new)[lo:hi])
        vs += list(wl.bits(case.v_new)[lo:hi])
    return np.stack(ks), np.stack(vs)


def _sdpa_tail(case, b, with_new, seed=1):
    """fp64 out [q, Hq, D] and lse [q, Hq] of row b's queries as the last q
    rows of a kv x kv causal problem (filler queries above them)."""
    k_bits, v_bits = _dense(case, b, with_new)
    kv = k_bits.shape[0]
    lo, hi = case.qo_indptr[b], case.qo_indptr[b + 1]
    qn = hi - lo
    G = case.group
    filler = torch.randn(kv - qn, case.num_q_heads, case.head_dim, dtype=torch.float64,
                         generator=torch.Generator().manual_seed(seed))
    q = torch.cat([filler, torch.from_numpy(_f64(wl.bits(case.q)[lo:hi]))]).permute(1, 0, 2)[None]
    k = torch.from_numpy(_f64(k_bits)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    v = torch.from_numpy(_f64(v_bits)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=case.softmax_scale)
    s = (q[0, :, kv - qn:, None, :] * k[0, :, None]).sum(-1) * case.softmax_scale  # [Hq, q, kv]
    mask = torch.arange(kv)[None, :] <= (kv - qn + torch.arange(qn))[:, None]
    lse = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
    return out[0, :, kv - qn:].permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
@pytest.mark.parametrize("Hq,Hkv,D,P", [(4, 2, 16, 4), (8, 2, 32, 8), (6, 6, 8, 16)])
def test_rows_match_tail_of_square_causal_sdpa(oracle_mod, layout, Hq, Hkv, D, P):
    # decode (q=1), speculative (q=3, 4), a chunk on a cache (q=9), a first chunk (L=0)
    q_lens, cache = [1, 3, 9, 4, 7, 1], [13, 5, 20, 0, 0, 31]
    case = wl.mixed_step(11, q_lens, cache, Hq, Hkv, D, P, layout=layout)
    out, lse, err, rows, _, _ = _run(oracle_mod, case)
    assert err == 0 and not rows.any()
    for b in range(case.batch):
        lo, hi = case.qo_indptr[b], case.qo_indptr[b + 1]
        ref, ref_lse = _sdpa_tail(case, b, True)
        np.testing.assert_allclose(out[lo:hi], ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[lo:hi], ref_lse, rtol=1e-12, atol=1e-12)


def test_attend_only_matches_sdpa(oracle_mod):
    # the caller appended already: kv = L and query i sees L - q + i + 1 keys
    case = wl.mixed_step(12, [2, 5, 1], [9, 5, 4], 4, 1, 16, 4)
    out, lse, err, _, _, _ = _run(oracle_mod, case, with_new=False)
    assert err == 0
    for b in range(case.batch):
        lo, hi = case.qo_indptr[b], case.qo_indptr[b + 1]
        ref, ref_lse = _sdpa_tail(case, b, False)
        np.testing.assert_allclose(out[lo:hi], ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[lo:hi], ref_lse, rtol=1e-12, atol=1e-12)


def test_first_chunk_is_plain_causal(oracle_mod):
    case = wl.mixed_step(13, [17], [0], 4, 2, 16, 8)
    out, _, _, _, _, _ = _run(oracle_mod, case)
    q = torch.from_numpy(_f64(wl.bits(case.q))).permute(1, 0, 2)[None]
    k = torch.from_numpy(_f64(wl.bits(case.k_new))).permute(1, 0, 2).repeat_interleave(2, 0)[None]
    v = torch.from_numpy(_f64(wl.bits(case.v_new))).permute(1, 0, 2).repeat_interleave(2, 0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=case.softmax_scale)
    np.testing.assert_allclose(out, ref[0].permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)


def test_one_token_on_empty_cache_is_exact(oracle_mod):
    case = wl.mixed_step(14, [1, 1], [0, 0], 4, 2, 16, 4)
    out, lse, _, _, _, _ = _run(oracle_mod, case)
    vnew = _f64(wl.bits(case.v_new))  # [2, Hkv, D]
    knew = _f64(wl.bits(case.k_new))
    qv = _f64(wl.bits(case.q))  # [2, Hq, D]
    for t in range(2):
        for h in range(4):
            assert np.array_equal(out[t, h], vnew[t, h // 2])
            assert lse[t, h] == pytest.approx(case.softmax_scale * float(qv[t, h] @ knew[t, h // 2]), rel=1e-14)


def test_append_writes_exactly_the_new_slots(oracle_mod):
    case = wl.mixed_step(15, [1, 6, 0, 3], [7, 2, 4, -1], 4, 2, 16, 4, layout=wl.HND)
    _, _, err, _, k, v = _run(oracle_mod, case)
    assert err == 0
    k_ref, v_ref = wl.bits(case.k_cache).copy(), wl.bits(case.v_cache).copy()
    kn, vn = wl.bits(case.k_new), wl.bits(case.v_new)
    for b in range(case.batch):
        L = int(case.cache_seqlens[b])
        if L < 0:
            continue
        for i, t in enumerate(range(case.qo_indptr[b], case.qo_indptr[b + 1])):
            pos = L + i
            page, slot = case.block_table[b, pos // case.page_size], pos % case.page_size
            k_ref[page, :, slot] = kn[t]
            v_ref[page, :, slot] = vn[t]
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_single_token_rows_equal_fused_decode(oracle_mod):
    case = wl.mixed_step(16, [1, 1, 1], [5, 0, 12], 4, 2, 16, 4)
    out, lse, _, _, _, _ = _run(oracle_mod, case)
    k, v = wl.bits(case.k_cache).copy(), wl.bits(case.v_cache).copy()
    out_d, lse_d, _, _ = oracle_mod.decode(_desc(oracle_mod, case), k, v, wl.bits(case.q), wl.bits(case.k_new),
                                           wl.bits(case.v_new), case.block_table, case.cache_seqlens,
                                           case.softmax_scale)
    assert np.array_equal(out, out_d) and np.array_equal(lse, lse_d)


def test_page_permutation_is_bit_invariant(oracle_mod):
    case = wl.mixed_step(17, [2, 5], [9, 3], 4, 2, 16, 4)
    out, lse, _, _, _, _ = _run(oracle_mod, case)
    perm = np.concatenate([[0], np.random.default_rng(0).permutation(case.num_pages - 1) + 1]).astype(np.int32)
    k2, v2 = np.empty_like(wl.bits(case.k_cache)), np.empty_like(wl.bits(case.v_cache))
    k2[perm], v2[perm] = wl.bits(case.k_cache), wl.bits(case.v_cache)
    case.block_table = np.where(case.block_table > 0, perm[case.block_table], 0).astype(np.int32)
    out2, lse2, _, _, _, _ = _run(oracle_mod, case, k=k2, v=v2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_row_fates(oracle_mod):
    # rows: ok, inactive, too long, bad cached page, bad destination page
    case = wl.mixed_step(18, [2, 3, 6, 2, 2], [8, -1, 4, 9, 6], 4, 2, 16, 4)
    case.block_table = case.block_table.copy()
    case.block_table[3, 0] = 0                    # row 3: a cached token's page
    dest = int(case.block_table[4, 1])            # row 4: the page of its new tokens 6 and 7
    case.block_table[4, 1] = case.num_pages
    out, lse, err, rows, k, v = _run(oracle_mod, case, max_qlen=5)
    assert list(rows) == [0, 0, oracle_mod.ERR_QLEN, oracle_mod.ERR_PAGE, oracle_mod.ERR_PAGE]
    assert err == oracle_mod.ERR_QLEN | oracle_mod.ERR_PAGE
    ip = case.qo_indptr
    assert np.all(np.isfinite(out[ip[0]:ip[1]])) and np.all(out[ip[0]:ip[1]] != 0)
    for b in (1, 2, 3, 4):
        assert np.all(out[ip[b]:ip[b + 1]] == 0) and np.all(np.isneginf(lse[ip[b]:ip[b + 1]]))
    kp = wl.bits(case.k_cache)

    def slot(b, pos):
        return k[case.block_table[b, pos // 4], :, pos % 4] if case.layout == wl.HND else \
            k[case.block_table[b, pos // 4], pos % 4]
    # too long: no append; bad cached page: the append still lands (its own pages are fine)
    assert np.array_equal(k[case.block_table[2, 1]], kp[case.block_table[2, 1]])
    kn = wl.bits(case.k_new)
    assert np.array_equal(slot(3, 9), kn[ip[3]]) and np.array_equal(slot(3, 10), kn[ip[3] + 1])
    # bad destination page: nothing of the row is written
    assert np.array_equal(k[dest], kp[dest])


def test_reversed_range_writes_nothing(oracle_mod):
    case = wl.mixed_step(19, [2, 2, 2], [3, 3, 3], 4, 2, 16, 4)
    case.qo_indptr = np.array([0, 4, 2, 6], np.int32)  # row 1 is reversed
    out, lse, err, rows, _, _ = _run(oracle_mod, case)
    assert rows[1] == oracle_mod.ERR_QLEN and err & oracle_mod.ERR_QLEN
    assert rows[0] == 0 and rows[2] == 0


def test_overflow_row(oracle_mod):
    case = wl.mixed_step(20, [4, 1], [6, 2], 4, 2, 16, 4)
    case.max_blocks = case.block_table.shape[1]
    case.cache_seqlens = case.cache_seqlens.copy()
    case.cache_seqlens[0] = 4 * case.max_blocks - 2  # 4 new tokens do not fit
    out, lse, err, rows, _, _ = _run(oracle_mod, case)
    assert rows[0] == oracle_mod.ERR_OVERFLOW and rows[1] == 0
    assert np.all(out[0:4] == 0) and np.all(np.isneginf(lse[0:4]))
