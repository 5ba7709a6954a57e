"""Pins for the fp64 oracle's ragged end-aligned causal prefill (CPU only).

* The visited pair count equals the printed closed form Hq * sum q(2kv-q+1)/2
  on the two workloads the FlashInfer page prints (tests/golden).
* Query i of q over kv keys sees kv - q + i + 1 keys (printed rule, golden).
* q == kv reduces to torch's fp64 SDPA with is_causal=True; q < kv equals
  the last q rows of a kv x kv causal SDPA (end alignment).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from paged_kv_decode_append_gb300 import workloads as wl

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "printed_values.json")))


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(seed, q_lens, kv_lens, Hq, Hkv, D, P, layout=wl.HND, extra_pages=3):
    g = torch.Generator().manual_seed(seed)
    q_lens = np.asarray(q_lens, np.int32)
    kv_lens = np.asarray(kv_lens, np.int32)
    B = len(q_lens)
    indptr = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    needed = (kv_lens + P - 1) // P
    NP = int(needed.sum()) + 1 + extra_pages
    order = (torch.randperm(NP - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = wl.assign_pages(needed, NP, int(needed.max()), order)
    case = wl.PagedCase("p", B, Hq, Hkv, D, P, NP, layout, int(needed.max()), bt, np.zeros(B, np.int32),
                        1.0 / math.sqrt(D), q=wl._randn_bf16((int(indptr[-1]), Hq, D), g, "cpu"),
                        qo_indptr=indptr, kv_lens=kv_lens)
    wl._fill_cache(case, g, "cpu", "cpu")
    return case


def _run(oracle, case, sel=None):
    d = oracle.CacheDesc(case.num_pages, case.page_size, case.num_kv_heads, case.head_dim, case.layout)
    return oracle.prefill(d, wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.q), case.qo_indptr,
                          case.kv_lens, case.block_table, case.softmax_scale, sel=sel)


def _dense_row(case, which, b):
    pool = wl.bits(case.k_cache if which == "k" else case.v_cache)
    toks = []
    for t in range(int(case.kv_lens[b])):
        page, slot = case.block_table[b, t // case.page_size], t % case.page_size
        toks.append(pool[page, :, slot] if case.layout == wl.HND else pool[page, slot])
    return np.stack(toks)  # [kv, Hkv, D]


@pytest.mark.parametrize("entry", GOLDEN["causal_pairs"], ids=lambda e: f"Hq{e['num_q_heads']}")
def test_pair_count_matches_printed_formula(oracle_mod, entry):
    # Pair counts do not depend on D or Hkv; a small head keeps the oracle fast.
    Hq = entry["num_q_heads"]
    case = _case(7, entry["q_lens"], entry["kv_lens"], Hq, Hq // 4 if Hq % 4 == 0 else Hq, 4, 16)
    _, _, pairs, _ = _run(oracle_mod, case)
    assert pairs == entry["pairs"]
    assert (pairs >= GOLDEN["admission_threshold"]["value"]) == entry["admitted"]


@pytest.mark.parametrize("c", GOLDEN["visible_keys"]["cases"], ids=lambda c: f"q{c['q']}kv{c['kv']}")
def test_visible_keys_per_query(oracle_mod, c):
    case = _case(3, [c["q"]], [c["kv"]], 2, 1, 8, 4)
    for i, want in enumerate(c["visible"]):
        _, _, pairs, _ = _run(oracle_mod, case, sel=[(i, 1)])
        assert pairs == want


def test_q_equals_kv_is_standard_causal(oracle_mod):
    case = _case(21, [13, 1, 40], [13, 1, 40], 8, 2, 32, 8)
    out, lse, pairs, _ = _run(oracle_mod, case)
    assert pairs == 8 * sum(q * (q + 1) // 2 for q in (13, 1, 40))
    q_all = _f64(wl.bits(case.q))
    for b in range(case.batch):
        lo, hi = case.qo_indptr[b], case.qo_indptr[b + 1]
        q = torch.from_numpy(q_all[lo:hi]).permute(1, 0, 2)[None]  # [1, Hq, q, D]
        k = torch.from_numpy(_f64(_dense_row(case, "k", b))).permute(1, 0, 2).repeat_interleave(4, 0)[None]
        v = torch.from_numpy(_f64(_dense_row(case, "v", b))).permute(1, 0, 2).repeat_interleave(4, 0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=case.softmax_scale)
        np.testing.assert_allclose(out[lo:hi], ref[0].permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("layout", [wl.HND, wl.NHD])
def test_end_aligned_matches_tail_of_square_causal(oracle_mod, layout):
    q_lens, kv_lens = [5, 1, 17], [29, 9, 17]
    case = _case(8, q_lens, kv_lens, 6, 3, 16, 4, layout=layout)
    out, lse, pairs, _ = _run(oracle_mod, case)
    assert pairs == 6 * sum(q * (2 * kv - q + 1) // 2 for q, kv in zip(q_lens, kv_lens))
    q_all = _f64(wl.bits(case.q))
    g = torch.Generator().manual_seed(1)
    for b in range(case.batch):
        lo, hi = case.qo_indptr[b], case.qo_indptr[b + 1]
        kv, qn = int(kv_lens[b]), hi - lo
        # a kv x kv causal problem whose last qn query rows are this request's queries
        filler = torch.randn(kv - qn, 6, 16, generator=g, dtype=torch.float64)
        q_full = torch.cat([filler, torch.from_numpy(q_all[lo:hi])]).permute(1, 0, 2)[None]
        k = torch.from_numpy(_f64(_dense_row(case, "k", b))).permute(1, 0, 2).repeat_interleave(2, 0)[None]
        v = torch.from_numpy(_f64(_dense_row(case, "v", b))).permute(1, 0, 2).repeat_interleave(2, 0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(q_full, k, v, is_causal=True,
                                                               scale=case.softmax_scale)
        np.testing.assert_allclose(out[lo:hi], ref[0, :, kv - qn:].permute(1, 0, 2).numpy(), rtol=1e-11,
                                   atol=1e-12)
        scores = (q_full[0, :, kv - qn:, None, :] * k[0, :, None]).sum(-1) * case.softmax_scale
        mask = torch.arange(kv)[None, :] <= (kv - qn + torch.arange(qn))[:, None]
        ref_lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
        np.testing.assert_allclose(lse[lo:hi], ref_lse.permute(1, 0).numpy(), rtol=1e-12, atol=1e-12)


def test_malformed_request_rejected(oracle_mod):
    case = _case(2, [4], [4], 2, 1, 8, 4)
    case.kv_lens = np.array([3], np.int32)  # q > kv is outside the end-aligned rule
    _, _, pairs, _ = _run(oracle_mod, case)
    assert pairs == -1


def test_bad_page_zeroes_row(oracle_mod):
    case = _case(2, [3, 2], [9, 5], 2, 1, 8, 4)
    case.block_table = case.block_table.copy()
    case.block_table[0, 1] = 0
    out, lse, pairs, err_rows = _run(oracle_mod, case)
    assert pairs == -2 and err_rows[0] == oracle_mod.ERR_PAGE and err_rows[1] == 0
    assert np.all(out[0:3] == 0) and np.all(np.isneginf(lse[0:3]))
    assert np.all(np.isfinite(out[3:]))


def test_pool_bytes_printed_example():
    g = GOLDEN["pool_bytes"]
    total = g["num_pages"] * g["page_size"] * g["layers"] * 2 * g["num_kv_heads"] * g["head_dim"] * g["bytes_per_value"]
    assert total == g["total_bytes"]
    # the page prints the decimal-GB value truncated to two places (2.936 -> 2.93)
    assert math.floor(total / 1e7) / 100 == g["printed_gb"]
