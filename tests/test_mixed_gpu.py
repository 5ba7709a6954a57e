"""GPU parity of the mixed step (pkv_mixed_attn) with the fp64 oracle:
single-token decode rows, multi-token decode rows (split-KV decode kernel,
(query, head) columns with per-column causal limits) and prefill chunks
(tensor-core prefill kernel over L + q keys) in one call.  The appended cache
is bit-exact; outputs within max-abs / max-rel 1e-2 and lse within 1e-2 of
the oracle; every row fate (inactive, too long, reversed range, bad page,
overflow) matches; repeated calls and graph replays are bit-identical."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_append_gb300 as pkv
from paged_kv_decode_append_gb300 import workloads as wl

from gpu_util import assert_close, assert_lse_close, desc_of

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _dev(case):
    return (torch.as_tensor(case.qo_indptr, device=DEV), torch.as_tensor(case.block_table, device=DEV),
            torch.as_tensor(case.cache_seqlens, device=DEV))


def _run_gpu(case, max_qlen, dq, with_new=True, ws=None, qo=None):
    qo0, bt, sl = _dev(case)
    qo = qo0 if qo is None else qo
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    q = case.q.to(DEV)
    T, Hq, _ = q.shape
    out = torch.full_like(q, float("nan"))
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kn = case.k_new.to(DEV) if with_new else None
    vn = case.v_new.to(DEV) if with_new else None
    pkv.pkv_mixed_attn(kc, vc, q, kn, vn, qo, bt, sl, case.softmax_scale, max_qlen, dq, out=out, lse=lse,
                       workspace=ws, err_flag=err, layout=case.layout)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy(), int(err.item()), kc, vc


def _run_oracle(case, max_qlen, with_new=True, qo_indptr=None, sel=None):
    k, v = wl.bits(case.k_cache).copy(), wl.bits(case.v_cache).copy()
    out, lse, err, rows = oracle.mixed(desc_of(case), k, v, wl.bits(case.q),
                                       wl.bits(case.k_new) if with_new else None,
                                       wl.bits(case.v_new) if with_new else None,
                                       case.qo_indptr if qo_indptr is None else qo_indptr, case.block_table,
                                       case.cache_seqlens, case.softmax_scale, max_qlen=max_qlen, sel=sel)
    return out, lse, err, rows, k, v


def _compare(case, got, ref, check_cache=True):
    out, lse, err, kc, vc = got
    rout, rlse, rerr, _, rk, rv = ref
    assert err == rerr, (err, rerr)
    if check_cache:
        assert np.array_equal(wl.bits(kc), rk) and np.array_equal(wl.bits(vc), rv), "appended cache differs"
    written = ~np.isnan(rlse)  # query rows (and heads) some row owns
    assert np.array_equal(~np.isnan(lse), written), "rows written differ from the rows owned"
    zero = np.isneginf(rlse)
    assert np.all(out[zero] == 0) and np.all(np.isneginf(lse[zero]))
    live = written & ~zero
    if live.any():
        assert_close(out[live], rout[live])
        assert_lse_close(lse[live], rlse[live])


# D, Hq, Hkv, P, layout
GEOMS = [
    (128, 32, 8, 16, wl.NHD),   # Qwen3-shaped, G 4
    (128, 32, 8, 16, wl.HND),
    (256, 48, 6, 16, wl.HND),   # G 8
    (64, 8, 8, 8, wl.NHD),      # G 1
    (64, 16, 1, 32, wl.HND),    # G 16
    (128, 8, 4, 128, wl.NHD),   # G 2, page 128
]
# q_lens / cache lens: decode, speculative (2, 3, 4, 7), a chunk on a cache,
# a first chunk, an inactive row, a row with no query
Q_LENS = [1, 4, 37, 2, 1, 129, 3, 0, 7, 1]
CACHE = [300, 45, 260, 1, 0, 0, 999, 17, 64, -1]


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"D{g[0]}-G{g[1] // g[2]}-P{g[3]}-{'HND' if g[4] else 'NHD'}")
@pytest.mark.parametrize("dq", [None, 1, 8], ids=["dq-default", "dq1", "dq8"])
def test_parity_mixed_batch(geom, dq):
    D, Hq, Hkv, P, layout = geom
    case = wl.mixed_step(200 + D + P + Hq, Q_LENS, CACHE, Hq, Hkv, D, P, layout, device=DEV)
    dq = pkv.default_decode_max_qlen(Hq, Hkv) if dq is None else dq
    _compare(case, _run_gpu(case, 256, dq), _run_oracle(case, 256))


@pytest.mark.parametrize("max_qlen,dq", [(8, 8), (4, 8)], ids=["no-prefill", "long-row-zeroed-by-decode"])
def test_decode_kernel_alone(max_qlen, dq):
    """No row longer than the decode limit: the prefill kernel is not launched;
    a row past max_qlen is zeroed by the decode kernel (PKV_ERR_QLEN)."""
    case = wl.mixed_step(31, [1, 8, 3, 6, 2], [513, 40, 0, 77, 1500], 32, 8, 128, 16, wl.NHD, device=DEV)
    _compare(case, _run_gpu(case, max_qlen, dq), _run_oracle(case, max_qlen))


def test_small_pages_decode_only():
    """Pages of 4 tokens (no prefill kernel): every row on the decode kernel."""
    case = wl.mixed_step(32, [1, 5, 2, 8], [50, 3, 0, 200], 16, 4, 64, 4, wl.HND, device=DEV)
    _compare(case, _run_gpu(case, 8, 8), _run_oracle(case, 8))


def test_attend_only():
    """k_new / v_new NULL: the queries' own tokens are cached already, so the
    cache lengths include them (kv = L); one row has fewer keys than queries."""
    q_lens = [1, 4, 50, 3, 5]
    case = wl.mixed_step(33, q_lens, [31, 13, 130, 5, 3], 32, 8, 128, 16, wl.HND, device=DEV)
    got = _run_gpu(case, 64, 4, with_new=False)
    ref = _run_oracle(case, 64, with_new=False)
    _compare(case, got, ref)


def test_long_rows_split_across_ctas():
    """Multi-token rows long enough to be split over many CTAs: the appended
    tokens (and so the column masks) sit in the last slice of each unit."""
    case = wl.mixed_step(34, [4, 3, 1, 2], [9000, 4100, 7000, 31], 32, 8, 128, 16, wl.NHD, extra_pages=0,
                         device=DEV)
    _compare(case, _run_gpu(case, 4, 4), _run_oracle(case, 4))


@pytest.mark.parametrize("geom", [(64, 16, 2, 32, wl.HND), (256, 16, 2, 16, wl.NHD), (128, 32, 8, 16, wl.HND)],
                         ids=["D64-G8", "D256-G8", "D128-G4"])
def test_wide_units_split_across_ctas(geom):
    """Units of 9..16 (query, head) columns (one consumer warp per 8 columns,
    over one K/V pass) on rows long enough to be split over many CTAs: their
    partials are written and merged in two 8-column passes; a row of 24
    columns takes a 16-column and an 8-column unit."""
    D, Hq, Hkv, P, layout = geom
    G = Hq // Hkv
    q_lens = [16 // G, 24 // G, 1, 12 // G if G < 8 else 2, 16 // G]
    case = wl.mixed_step(36 + D, q_lens, [9000, 4100, 7000, 31, 0], Hq, Hkv, D, P, layout, extra_pages=0,
                         device=DEV)
    dq = 24 // G
    _compare(case, _run_gpu(case, dq, dq), _run_oracle(case, dq))


def test_row_fates_match_oracle():
    # ok, inactive, too long, bad cached page (decode row), bad destination
    # page (prefill row), overflow, bad cached page (prefill row)
    case = wl.mixed_step(35, [2, 3, 20, 2, 12, 3, 9], [8, -1, 4, 90, 6, 10, 40], 32, 8, 128, 16, wl.NHD,
                         device=DEV)
    case.block_table = case.block_table.copy()
    case.block_table[3, 1] = 0                      # tokens 16..31 of row 3
    case.block_table[4, 1] = case.num_pages + 5     # tokens 16, 17: new tokens of row 4
    case.block_table[6, 0] = case.num_pages         # tokens 0..15 of row 6
    case.cache_seqlens = case.cache_seqlens.copy()
    case.cache_seqlens[5] = 16 * case.block_table.shape[1] - 1
    _compare(case, _run_gpu(case, 16, 4), _run_oracle(case, 16))


@pytest.mark.parametrize("max_qlen", [8, 2], ids=["with-prefill", "decode-only"])
def test_query_range_past_total_q(max_qlen):
    """Row 2's range ends past total_q: PKV_ERR_QLEN, no append, nothing
    written for it; the other rows are unaffected."""
    case = wl.mixed_step(36, [2, 2, 2], [10, 10, 10], 32, 8, 128, 16, wl.NHD, device=DEV)
    bad = np.array([0, 2, 4, 9], np.int32)
    got = _run_gpu(case, max_qlen, 1, qo=torch.as_tensor(bad, device=DEV))
    ref = _run_oracle(case, max_qlen, qo_indptr=bad)
    assert ref[2] == oracle.ERR_QLEN
    _compare(case, got, ref)


def test_decreasing_indptr_sets_the_flag():
    case = wl.mixed_step(36, [2, 2, 2], [10, 10, 10], 32, 8, 128, 16, wl.NHD, device=DEV)
    got = _run_gpu(case, 8, 4, qo=torch.as_tensor(np.array([0, 4, 2, 6], np.int32), device=DEV))
    assert got[2] & oracle.ERR_QLEN


def test_repeat_and_page_permutation_are_bit_identical():
    case = wl.mixed_step(37, Q_LENS, CACHE, 32, 8, 128, 16, wl.HND, device=DEV)
    ws = pkv.mixed_workspace(case.batch, case.q.shape[0], case.block_table.shape[1], 32, 256, 4,
                             pkv.cache_desc(case.k_cache, case.layout), DEV)
    a = _run_gpu(case, 256, 4, ws=ws)
    b = _run_gpu(case, 256, 4, ws=ws)
    assert np.array_equal(a[0], b[0], equal_nan=True) and np.array_equal(a[1], b[1], equal_nan=True)
    # the same logical cache on other physical pages
    perm = torch.as_tensor(np.concatenate([[0], np.random.default_rng(1).permutation(case.num_pages - 1) + 1]),
                           device=DEV)
    k2, v2 = torch.empty_like(case.k_cache), torch.empty_like(case.v_cache)
    k2[perm], v2[perm] = case.k_cache, case.v_cache
    case.k_cache, case.v_cache = k2, v2
    case.block_table = np.where(case.block_table > 0, perm.cpu().numpy()[case.block_table], 0).astype(np.int32)
    c = _run_gpu(case, 256, 4, ws=ws)
    assert np.array_equal(a[0], c[0], equal_nan=True) and np.array_equal(a[1], c[1], equal_nan=True)


def test_graph_capture_replays_identically():
    case = wl.mixed_step(38, Q_LENS, CACHE, 32, 8, 128, 16, wl.NHD, device=DEV)
    qo, bt, sl = _dev(case)
    q, kn, vn = case.q.to(DEV), case.k_new.to(DEV), case.v_new.to(DEV)
    ws = pkv.mixed_workspace(case.batch, q.shape[0], bt.shape[1], 32, 256, 4,
                             pkv.cache_desc(case.k_cache, case.layout), DEV)
    out = torch.empty_like(q)
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    eager = pkv.pkv_mixed_attn(kc, vc, q, kn, vn, qo, bt, sl, case.softmax_scale, 256, 4, workspace=ws).clone()
    kc2, vc2 = case.k_cache.clone(), case.v_cache.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pkv.pkv_mixed_attn(kc2, vc2, q, kn, vn, qo, bt, sl, case.softmax_scale, 256, 4, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert torch.equal(kc2.view(torch.int16), kc.view(torch.int16))


def test_speculative_decode_qwen3_layer_sampled():
    """B=64 rows of 4 speculative tokens on cached lengths U[512, 1024],
    Qwen3-shaped (Hq=32, Hkv=8, D=128, page 16, shuffled pages) -- the decode
    kernel's multi-query path at full size, checked on sampled rows."""
    g = np.random.default_rng(5)
    B = 64
    case = wl.mixed_step(39, [4] * B, g.integers(512, 1025, B), 32, 8, 128, 16, wl.NHD, device=DEV)
    out, lse, err, kc, vc = _run_gpu(case, 4, 4)
    assert err == 0
    rows = g.choice(case.q.shape[0], 24, replace=False)
    sel = [(int(t), int(h)) for t in rows for h in (0, 3, 17, 31)]
    rout, rlse, rerr, _, rk, rv = _run_oracle(case, 4, sel=sel)
    assert rerr == 0
    assert np.array_equal(wl.bits(kc), rk) and np.array_equal(wl.bits(vc), rv)
    t, h = np.array(sel).T
    assert_close(out[t, h], rout[t, h])
    assert_lse_close(lse[t, h], rlse[t, h])


def _bench_workload_sampled(case, rows, max_qlen, tokens_per_row=None, seed=0):
    """The full workload on the GPU in the bench's launch configuration (the
    library's default decode_max_qlen); the oracle on a host copy of only the
    sampled rows' pages, taken before the call (the oracle appends itself).
    Checks the rows' appended slots bit for bit and sampled (token, head)
    outputs within tolerance."""
    dq = pkv.default_decode_max_qlen(case.num_q_heads, case.num_kv_heads)
    ql = np.diff(case.qo_indptr)
    need = case.cache_seqlens[rows] + ql[rows]
    k0, v0, bt_sub = wl.compact_rows(case.k_cache, case.v_cache, case.block_table, rows, need, case.page_size)
    out, lse, err, kc, vc = _run_gpu(case, max_qlen, dq)
    assert err == 0
    toks = [np.arange(case.qo_indptr[b], case.qo_indptr[b + 1]) for b in rows]
    idx = np.concatenate(toks)
    qo_sub = np.concatenate([[0], np.cumsum(ql[rows])]).astype(np.int32)
    d = oracle.CacheDesc(k0.shape[0], case.page_size, case.num_kv_heads, case.head_dim, case.layout)
    rng = np.random.default_rng(seed)
    sel = []
    for i, t in enumerate(toks):
        pick = t if tokens_per_row is None or len(t) <= tokens_per_row else \
            np.unique(np.concatenate([[t[0], t[-1]], rng.choice(t, tokens_per_row - 2, replace=False)]))
        base = int(qo_sub[i]) - int(t[0])
        sel += [(int(x) + base, h) for x in pick for h in rng.choice(case.num_q_heads, 4, replace=False)]
    k_or, v_or = k0.copy(), v0.copy()
    rout, rlse, rerr, _ = oracle.mixed(d, k_or, v_or, wl.bits(case.q)[idx], wl.bits(case.k_new)[idx],
                                       wl.bits(case.v_new)[idx], qo_sub, bt_sub, case.cache_seqlens[rows],
                                       case.softmax_scale, max_qlen=max_qlen, sel=sel)
    assert rerr == 0
    k1, v1, _ = wl.compact_rows(kc, vc, case.block_table, rows, need, case.page_size)
    assert np.array_equal(k1, k_or) and np.array_equal(v1, v_or), "appended slots differ"
    t_sub, h = np.array(sel).T
    assert_close(out[idx[t_sub], h], rout[t_sub, h])
    assert_lse_close(lse[idx[t_sub], h], rlse[t_sub, h])


def test_spec_decode_bench_workload_sampled():
    """bench.py --workload spec: B=32 rows of 4 tokens, Qwen3-shaped, page 16,
    65,536-page shuffled pool; decode kernel (multi-query rows)."""
    case = wl.spec_decode(device=DEV)
    _bench_workload_sampled(case, [0, 7, 13, 22, 31], 4)


def test_chunked_bench_workload_sampled():
    """bench.py --workload chunked: 4 chunks of 496 tokens on prefixes
    U[0,2048] + 60 decode rows; chunks on the prefill kernel, decode rows on
    the decode kernel, in one call."""
    case = wl.chunked_mix(device=DEV)
    _bench_workload_sampled(case, [0, 3, 4, 30, 63], 496, tokens_per_row=12)
