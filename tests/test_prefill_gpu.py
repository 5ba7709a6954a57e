"""GPU parity of the ragged causal paged prefill (pkv_prefill_attn) with the
fp64 oracle: outputs within max-abs / max-rel 1e-2, lse within 1e-2, error
rows zeroed with the matching bit, results independent of the physical page
placement and of repetition."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_append_gb300 as pkv
from paged_kv_decode_append_gb300 import workloads as wl

from gpu_util import assert_close, assert_lse_close, desc_of

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _tensors(case):
    return (torch.as_tensor(case.qo_indptr, device=DEV), torch.as_tensor(case.kv_lens, device=DEV),
            torch.as_tensor(case.block_table, device=DEV))


def _run_gpu(case, qo=None, kvl=None, bt=None):
    qo0, kvl0, bt0 = _tensors(case)
    qo = qo0 if qo is None else qo
    kvl = kvl0 if kvl is None else kvl
    bt = bt0 if bt is None else bt
    q = case.q.to(DEV)
    T, Hq, _ = q.shape
    out = torch.full_like(q, float("nan"))
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.pkv_prefill_attn(case.k_cache, case.v_cache, q, qo, kvl, bt, case.softmax_scale, out=out, lse=lse,
                         err_flag=err, layout=case.layout)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(err.item())


def _run_oracle(case, sel=None, kv_lens=None, block_table=None):
    return oracle.prefill(desc_of(case), wl.bits(case.k_cache), wl.bits(case.v_cache), wl.bits(case.q),
                          case.qo_indptr, case.kv_lens if kv_lens is None else kv_lens,
                          case.block_table if block_table is None else block_table, case.softmax_scale, sel=sel)


SHAPES = [
    # D, Hq, Hkv, P, layout, q_lens, kv_lens
    (256, 48, 6, 16, wl.HND, [65, 1, 130, 17], [65, 100, 700, 17]),   # G 8, the ragged-prefill geometry
    (128, 32, 8, 16, wl.NHD, [33, 64, 5], [200, 64, 1000]),           # G 4
    (64, 4, 2, 8, wl.HND, [129, 3], [300, 3]),                        # G 2, page 8
    (128, 16, 16, 64, wl.HND, [200, 1], [250, 70]),                   # G 1: 128 queries per tile
    (256, 16, 1, 128, wl.NHD, [40, 9], [1000, 9]),                    # G 16: 8 queries per tile
    (64, 8, 1, 256, wl.NHD, [100], [600]),                            # page 256
    (128, 8, 2, 32, wl.HND, [64, 128, 63, 16], [64, 300, 127, 16]),   # tile-boundary lengths
    # CTA-pair kernel edges: page 8 boxes, page 256, key counts whose last
    # 128-key step leaves the odd CTA's K tile empty (kv % 128 in 1..64) or partial
    (256, 16, 2, 8, wl.NHD, [70, 33], [193, 33]),
    (128, 32, 8, 256, wl.HND, [100, 7], [640, 65]),
    (128, 32, 4, 16, wl.NHD, [129, 256, 1], [129, 320, 129]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"D{s[0]}-G{s[1] // s[2]}-P{s[3]}-{'HND' if s[4] else 'NHD'}")
def test_parity_with_oracle(shape):
    D, Hq, Hkv, P, layout, ql, kl = shape
    case = wl.small_prefill(100 + D + P, ql, kl, Hq, Hkv, D, P, layout, device=DEV)
    out, lse, err = _run_gpu(case)
    ref, ref_lse, pairs, _ = _run_oracle(case)
    assert err == 0 and pairs > 0
    assert_close(out, ref)
    assert_lse_close(lse, ref_lse)


def test_ragged_prefill_workload_sampled():
    """The B=8, Hq=48, Hkv=6, D=256, page-16 HND workload at full size, checked
    on sampled (query, head) rows: every request's first and last query, the
    query-tile boundaries, and random ones."""
    case = wl.ragged_prefill(device=DEV)
    out, lse, err = _run_gpu(case)
    assert err == 0
    rng = np.random.default_rng(0)
    Hq = case.num_q_heads
    toks = []
    for b in range(case.batch):
        s, e = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        toks += [s, e - 1, s + 15, s + 16, min(s + 64, e - 1)]
        toks += list(rng.integers(s, e, 12))
    sel = np.array([(t, h) for t in toks for h in rng.choice(Hq, 6, replace=False)], np.int32).reshape(-1)
    ref, ref_lse, pairs, _ = _run_oracle(case, sel=sel)
    t_idx, h_idx = sel[0::2], sel[1::2]
    assert_close(out[t_idx, h_idx], ref[t_idx, h_idx])
    assert_lse_close(lse[t_idx, h_idx], ref_lse[t_idx, h_idx])


def test_bad_page_and_overflow_zero_their_rows():
    case = wl.small_prefill(7, [20, 30, 10], [40, 90, 10], 8, 2, 128, 16, wl.HND, device=DEV)
    bt = case.block_table.copy()
    bt[1, 3] = 0                                   # a page request 1 needs
    kvl = case.kv_lens.copy()
    kvl[2] = case.max_blocks * case.page_size + 1  # more keys than the table can hold
    out, lse, err = _run_gpu(case, kvl=torch.as_tensor(kvl, device=DEV), bt=torch.as_tensor(bt, device=DEV))
    assert err == pkv.api.ERR_PAGE | pkv.api.ERR_OVERFLOW
    ref, ref_lse, pairs, err_rows = _run_oracle(case, kv_lens=kvl, block_table=bt)
    assert pairs == -2 and list(err_rows) == [0, oracle.ERR_PAGE, oracle.ERR_OVERFLOW]
    assert_close(out, ref)
    assert_lse_close(lse, ref_lse)
    assert not out[20:].any() and np.isneginf(lse[20:]).all()


def test_more_queries_than_keys_is_flagged():
    case = wl.small_prefill(9, [20, 30], [40, 90], 8, 2, 64, 16, wl.NHD, device=DEV)
    kvl = case.kv_lens.copy()
    kvl[0] = 10                                     # 20 queries over 10 keys
    out, lse, err = _run_gpu(case, kvl=torch.as_tensor(kvl, device=DEV))
    assert err == pkv.api.ERR_QLEN
    assert not out[:20].any() and np.isneginf(lse[:20]).all()
    ref, ref_lse, _, _ = _run_oracle(case)          # request 1 is unaffected
    assert_close(out[20:], ref[20:])
    assert_lse_close(lse[20:], ref_lse[20:])


def test_decreasing_indptr_runs_nothing():
    case = wl.small_prefill(11, [20, 30, 10], [40, 90, 10], 8, 2, 64, 16, wl.NHD, device=DEV)
    qo = case.qo_indptr.copy()
    qo[2] = 10                                      # request 1 would be 20 -> 10
    out, lse, err = _run_gpu(case, qo=torch.as_tensor(qo, device=DEV))
    assert err == pkv.api.ERR_QLEN
    assert not out[:60].any() and np.isneginf(lse[:60]).all()


def test_empty_requests_and_rows_nobody_owns():
    case = wl.small_prefill(13, [0, 25, 0], [0, 40, 7], 4, 4, 64, 16, wl.HND, device=DEV)
    out, lse, err = _run_gpu(case)
    ref, ref_lse, _, _ = _run_oracle(case)
    assert err == 0
    assert_close(out, ref)
    assert_lse_close(lse, ref_lse)


def test_bit_identical_across_calls_and_page_placement():
    D, Hq, Hkv, P = 128, 16, 2, 16
    case = wl.small_prefill(21, [70, 33], [300, 100], Hq, Hkv, D, P, wl.HND, extra_pages=40, device=DEV)
    a, la, _ = _run_gpu(case)
    b, lb, _ = _run_gpu(case)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)) and np.array_equal(la, lb)
    # move every page to another physical slot
    perm = np.random.default_rng(1).permutation(np.arange(1, case.num_pages)).astype(np.int32)
    mapping = np.concatenate([[0], perm]).astype(np.int32)
    k2 = torch.empty_like(case.k_cache)
    v2 = torch.empty_like(case.v_cache)
    idx = torch.as_tensor(mapping, device=DEV, dtype=torch.long)
    k2[idx] = case.k_cache
    v2[idx] = case.v_cache
    bt2 = mapping[case.block_table]
    case2 = wl.PagedCase(**{**case.__dict__, "k_cache": k2, "v_cache": v2, "block_table": bt2})
    c, lc, _ = _run_gpu(case2)
    assert np.array_equal(a.view(np.uint32), c.view(np.uint32)) and np.array_equal(la, lc)
