"""GPU parity of the fused append + decode kernel against the fp64 oracle.

Outputs within max-abs 1e-2 / max-rel 1e-2 (see gpu_util); appended cache
bytes and page routing bit-exact (sha256 of whole pools).
"""
import hashlib
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_append_gb300 as pkv
from paged_kv_decode_append_gb300 import workloads as wl

from gpu_util import assert_close, assert_lse_close, desc_of, f32, oracle_decode_compact

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _sha(t: torch.Tensor) -> str:
    return hashlib.sha256(wl.bits(t).tobytes()).hexdigest()


def _run(case, with_new=True, layout=None, err=None, workspace=None):
    layout = case.layout if layout is None else layout
    bt = torch.as_tensor(case.block_table, device=DEV)
    sl = torch.as_tensor(case.cache_seqlens, device=DEV)
    lse = torch.empty(case.batch, case.num_q_heads, dtype=torch.float32, device=DEV)
    out = pkv.pkv_decode_attn(case.k_cache, case.v_cache, case.q,
                              case.k_new if with_new else None, case.v_new if with_new else None,
                              bt, sl, case.softmax_scale, lse=lse, err_flag=err, workspace=workspace,
                              layout=layout)
    torch.cuda.synchronize()
    return out, lse


def _oracle_full(case, with_new=True):
    """Oracle on full host copies of the pools; returns out, lse, err, k, v."""
    k, v = wl.bits(case.k_cache).copy(), wl.bits(case.v_cache).copy()
    out, lse, err, err_rows = oracle.decode(desc_of(case), k, v, wl.bits(case.q),
                                            wl.bits(case.k_new) if with_new else None,
                                            wl.bits(case.v_new) if with_new else None,
                                            case.block_table, case.cache_seqlens, case.softmax_scale)
    return out, lse, err, k, v


@pytest.mark.parametrize("with_new", [True, False])
def test_tiny_parity_and_bit_exact_append(with_new):
    case = wl.tiny(device=DEV)
    ref_out, ref_lse, ref_err, ref_k, ref_v = _oracle_full(case, with_new)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = _run(case, with_new, err=err)
    assert ref_err == 0 and int(err.item()) == 0
    assert_close(f32(out), ref_out)
    assert_lse_close(lse.cpu().numpy(), ref_lse)
    assert hashlib.sha256(ref_k.tobytes()).hexdigest() == _sha(case.k_cache)
    assert hashlib.sha256(ref_v.tobytes()).hexdigest() == _sha(case.v_cache)


def test_qwen3_layer_full_parity():
    case = wl.qwen3_decode(device=DEV)
    ref_out, ref_lse, ref_err, _ = oracle_decode_compact(case)
    out, lse = _run(case)
    assert ref_err == 0
    assert_close(f32(out), ref_out)
    assert_lse_close(lse.cpu().numpy(), ref_lse)
    # appended slots: each row's token L_b holds k_new / v_new bit for bit
    kb, vb = wl.bits(case.k_cache), wl.bits(case.v_cache)
    for b in range(case.batch):
        L = int(case.cache_seqlens[b])
        page, slot = case.block_table[b, L // 16], L % 16
        assert np.array_equal(kb[page, slot], wl.bits(case.k_new)[b])
        assert np.array_equal(vb[page, slot], wl.bits(case.v_new)[b])


def test_skewed_full_parity():
    case = wl.skewed_decode(device=DEV)
    ref_out, ref_lse, ref_err, _ = oracle_decode_compact(case)
    out, lse = _run(case)
    assert ref_err == 0
    assert_close(f32(out), ref_out)
    assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("batch,contiguous", [(8, True), (64, False), (256, True)])
def test_batch_sweep_steps(batch, contiguous):
    """Three consecutive decode steps over two layer caches sharing one block
    table; the oracle replays the same appends on its own copies."""
    sw = wl.batch_sweep(batch, device=DEV, contiguous=contiguous, layers=2)
    bt = torch.as_tensor(sw.block_table, device=DEV)
    desc = pkv.cache_desc(sw.k_caches[0])
    ws = pkv.decode_workspace(batch, sw.max_blocks, 32, desc, DEV)
    host_k = [wl.bits(k).copy() for k in sw.k_caches]
    host_v = [wl.bits(v).copy() for v in sw.v_caches]
    od = oracle.CacheDesc(sw.num_pages, sw.page_size, 8, 128, wl.NHD)
    for step in range(3):
        lens = (sw.prompt_lens + step).astype(np.int32)
        sl = torch.as_tensor(lens, device=DEV)
        for layer, (q, kn, vn) in enumerate(wl.sweep_step_inputs(sw, step, DEV)):
            lse = torch.empty(batch, 32, dtype=torch.float32, device=DEV)
            out = pkv.pkv_decode_attn(sw.k_caches[layer], sw.v_caches[layer], q, kn, vn, bt, sl,
                                      sw.softmax_scale, lse=lse, workspace=ws)
            ref_out, ref_lse, err, _ = oracle.decode(od, host_k[layer], host_v[layer], wl.bits(q), wl.bits(kn),
                                                     wl.bits(vn), sw.block_table, lens, sw.softmax_scale)
            assert err == 0
            assert_close(f32(out), ref_out)
            assert_lse_close(lse.cpu().numpy(), ref_lse)
    for layer in range(2):
        assert hashlib.sha256(host_k[layer].tobytes()).hexdigest() == _sha(sw.k_caches[layer])
        assert hashlib.sha256(host_v[layer].tobytes()).hexdigest() == _sha(sw.v_caches[layer])


@pytest.mark.parametrize("batch,contiguous", [(8, False), (16, True), (32, False), (64, True), (128, False),
                                              (256, True)])
def test_batch_sweep_full_cycle(batch, contiguous):
    """All 512 decode steps of the sweep on two layer caches: outputs against
    the oracle at steps 0, 255 and 511 (on compact host copies of the GPU's
    cache at that step), and every one of the 512 appended tokens of every row
    bit-exact at the end (compact rows against a host scatter)."""
    steps, check = wl.SWEEP_DECODE_STEPS, (0, 255, 511)
    sw = wl.batch_sweep(batch, device=DEV, contiguous=contiguous, layers=2)
    bt = torch.as_tensor(sw.block_table, device=DEV)
    desc = pkv.cache_desc(sw.k_caches[0])
    ws = pkv.decode_workspace(batch, sw.max_blocks, 32, desc, DEV)
    rows = list(range(batch))
    cap = sw.prompt_lens + steps
    expect = [wl.compact_rows(sw.k_caches[layer], sw.v_caches[layer], sw.block_table, rows, cap, sw.page_size)
              for layer in range(2)]
    P = sw.page_size
    for step in range(steps):
        lens = (sw.prompt_lens + step).astype(np.int32)
        sl = torch.as_tensor(lens, device=DEV)
        for layer, (q, kn, vn) in enumerate(wl.sweep_step_inputs(sw, step, DEV, layers=2)):
            # the host scatter of this step's appended token
            ek, ev, ebt = expect[layer]
            pg = ebt[np.arange(batch), lens // P]
            ek[pg, lens % P] = wl.bits(kn)
            ev[pg, lens % P] = wl.bits(vn)
            if step in check:
                hk, hv, hbt = wl.compact_rows(sw.k_caches[layer], sw.v_caches[layer], sw.block_table, rows, lens + 1, P)
                od = oracle.CacheDesc(hk.shape[0], P, 8, 128, wl.NHD)
                ref_out, ref_lse, err, _ = oracle.decode(od, hk, hv, wl.bits(q), wl.bits(kn), wl.bits(vn), hbt, lens,
                                                         sw.softmax_scale)
                assert err == 0
            lse = torch.empty(batch, 32, dtype=torch.float32, device=DEV)
            out = pkv.pkv_decode_attn(sw.k_caches[layer], sw.v_caches[layer], q, kn, vn, bt, sl, sw.softmax_scale,
                                      lse=lse, workspace=ws, flags=pkv.api.DECODE_OVERLAP_PROLOGUE)
            if step in check:
                assert_close(f32(out), ref_out)
                assert_lse_close(lse.cpu().numpy(), ref_lse)
    for layer in range(2):
        gk, gv, _ = wl.compact_rows(sw.k_caches[layer], sw.v_caches[layer], sw.block_table, rows, cap, P)
        ek, ev, _ = expect[layer]
        assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


@pytest.mark.parametrize("use_plan", [False, True])
def test_decode_step_graph_with_padded_bucket(use_plan):
    """Three layers captured once as a decode-step graph for the 16-row bucket
    of 13 live rows (rows 13..15 inactive), replayed for two steps with the
    inputs rewritten in place.  Every layer's live rows match the fp64 oracle
    (which replays the same appends on its own host copies) within tolerance
    and direct calls bit for bit; padding rows are exactly 0 with lse -inf;
    the appended tokens are bit-exact against the oracle's copies."""
    live, layers = 13, 3
    bucket = pkv.pkv_decode_bucket(live)
    assert bucket == 16
    sw = wl.batch_sweep(live, device=DEV, contiguous=False, layers=layers)
    bt_live = sw.block_table
    bt = torch.zeros(bucket, sw.max_blocks, dtype=torch.int32, device=DEV)
    bt[:live] = torch.as_tensor(bt_live, device=DEV)
    desc = pkv.cache_desc(sw.k_caches[0])
    flags = pkv.api.DECODE_OVERLAP_PROLOGUE | pkv.api.DECODE_EARLY_KV
    if use_plan:  # layer 0 makes the step plan, layers 1.. reuse it
        flags |= pkv.api.DECODE_USE_PLAN
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kc_g = [k.clone() for k in sw.k_caches]
    vc_g = [v.clone() for v in sw.v_caches]
    # graph buffers (bucket rows), written in place every step
    q = [torch.zeros(bucket, 32, 128, dtype=torch.bfloat16, device=DEV) for _ in range(layers)]
    kn = [torch.zeros(bucket, 8, 128, dtype=torch.bfloat16, device=DEV) for _ in range(layers)]
    vn = [torch.zeros(bucket, 8, 128, dtype=torch.bfloat16, device=DEV) for _ in range(layers)]
    out = [torch.empty(bucket, 32, 128, dtype=torch.bfloat16, device=DEV) for _ in range(layers)]
    lse = [torch.empty(bucket, 32, dtype=torch.float32, device=DEV) for _ in range(layers)]
    seq = torch.full((bucket,), -1, dtype=torch.int32, device=DEV)
    ws = pkv.decode_workspace(bucket, sw.max_blocks, 32, desc, DEV)
    step_graph = pkv.DecodeStep(kc_g, vc_g, q, kn, vn, bt, seq, sw.softmax_scale, out, lse=lse, workspace=ws,
                                err_flag=err, flags=flags)
    ws_ref = pkv.decode_workspace(live, sw.max_blocks, 32, desc, DEV)
    bt_ref = torch.as_tensor(bt_live, device=DEV)
    rows = list(range(live))
    need = sw.prompt_lens + 2  # the pages both steps touch
    host = [wl.compact_rows(kc_g[layer], vc_g[layer], bt_live, rows, need, sw.page_size) for layer in range(layers)]
    od = oracle.CacheDesc(host[0][0].shape[0], sw.page_size, 8, 128, wl.NHD)
    for step in range(2):
        lens = torch.as_tensor((sw.prompt_lens + step).astype(np.int32), device=DEV)
        ins = wl.sweep_step_inputs(sw, step, DEV, layers=layers)
        seq[:live] = lens
        for layer, (qq, kk, vv) in enumerate(ins):
            q[layer][:live] = qq
            kn[layer][:live] = kk
            vn[layer][:live] = vv
        step_graph.launch()
        torch.cuda.synchronize()
        for layer, (qq, kk, vv) in enumerate(ins):
            hk, hv, hbt = host[layer]  # the oracle appends into its copies as well
            o_out, o_lse, o_err, _ = oracle.decode(od, hk, hv, wl.bits(qq), wl.bits(kk), wl.bits(vv), hbt,
                                                   lens.cpu().numpy(), sw.softmax_scale)
            assert o_err == 0
            assert_close(f32(out[layer][:live]), o_out, what=f"graph step {step} layer {layer}")
            assert_lse_close(lse[layer][:live].cpu().numpy(), o_lse)
            ref_lse = torch.empty(live, 32, dtype=torch.float32, device=DEV)
            ref = pkv.pkv_decode_attn(sw.k_caches[layer], sw.v_caches[layer], qq, kk, vv, bt_ref, lens,
                                      sw.softmax_scale, lse=ref_lse, workspace=ws_ref)
            torch.cuda.synchronize()
            assert torch.equal(out[layer][:live].view(torch.int16), ref.view(torch.int16))
            assert torch.equal(lse[layer][:live].view(torch.int32), ref_lse.view(torch.int32))
            assert not out[layer][live:].float().any()
            assert torch.isneginf(lse[layer][live:]).all()
    for layer in range(layers):
        assert torch.equal(kc_g[layer].view(torch.int16), sw.k_caches[layer].view(torch.int16))
        assert torch.equal(vc_g[layer].view(torch.int16), sw.v_caches[layer].view(torch.int16))
        gk, gv, _ = wl.compact_rows(kc_g[layer], vc_g[layer], bt_live, rows, need, sw.page_size)
        assert np.array_equal(gk, host[layer][0]) and np.array_equal(gv, host[layer][1])
    assert int(err.item()) == 0


def _plan_flags(layer):
    base = pkv.api.DECODE_OVERLAP_PROLOGUE | pkv.api.DECODE_EARLY_KV
    return base | (pkv.api.DECODE_MAKE_PLAN if layer == 0 else pkv.api.DECODE_USE_PLAN)


@pytest.mark.parametrize("batch,contiguous", [(8, False), (64, False), (256, True)])
def test_step_plan_reuse_is_bit_identical(batch, contiguous):
    """Three layers per step, layer 0 with PKV_DECODE_MAKE_PLAN and layers 1-2
    with PKV_DECODE_USE_PLAN, against the same calls planning for themselves
    (flags 0) on copies of the pools: the same work split, so outputs, lse and
    appended caches are bit-identical, and no error bit is raised.  One layer
    of the first step is also checked against the oracle."""
    layers = 3
    sw = wl.batch_sweep(batch, device=DEV, contiguous=contiguous, layers=layers)
    bt = torch.as_tensor(sw.block_table, device=DEV)
    desc = pkv.cache_desc(sw.k_caches[0])
    ws_p = pkv.decode_workspace(batch, sw.max_blocks, 32, desc, DEV)
    ws_r = pkv.decode_workspace(batch, sw.max_blocks, 32, desc, DEV)
    kc = [k.clone() for k in sw.k_caches]
    vc = [v.clone() for v in sw.v_caches]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    rows = list(range(batch))
    for step in (0, 1, 7):
        lens = (sw.prompt_lens + step).astype(np.int32)
        sl = torch.as_tensor(lens, device=DEV)
        ins = wl.sweep_step_inputs(sw, step, DEV, layers=layers)
        if step == 0:
            hk, hv, hbt = wl.compact_rows(sw.k_caches[1], sw.v_caches[1], sw.block_table, rows, lens + 1,
                                          sw.page_size)
        outs = []
        for layer, (q, kn, vn) in enumerate(ins):
            lse = torch.empty(batch, 32, dtype=torch.float32, device=DEV)
            o = pkv.pkv_decode_attn(kc[layer], vc[layer], q, kn, vn, bt, sl, sw.softmax_scale, lse=lse,
                                    workspace=ws_p, err_flag=err, flags=_plan_flags(layer))
            outs.append((o, lse))
        for layer, (q, kn, vn) in enumerate(ins):
            lse = torch.empty(batch, 32, dtype=torch.float32, device=DEV)
            o = pkv.pkv_decode_attn(sw.k_caches[layer], sw.v_caches[layer], q, kn, vn, bt, sl, sw.softmax_scale,
                                    lse=lse, workspace=ws_r)
            torch.cuda.synchronize()
            assert torch.equal(outs[layer][0].view(torch.int16), o.view(torch.int16))
            assert torch.equal(outs[layer][1].view(torch.int32), lse.view(torch.int32))
            if step == 0 and layer == 1:
                od = oracle.CacheDesc(hk.shape[0], sw.page_size, 8, 128, wl.NHD)
                r_out, r_lse, r_err, _ = oracle.decode(od, hk, hv, wl.bits(q), wl.bits(kn), wl.bits(vn), hbt, lens,
                                                       sw.softmax_scale)
                assert r_err == 0
                assert_close(f32(outs[layer][0]), r_out, what="plan reuse")
                assert_lse_close(outs[layer][1].cpu().numpy(), r_lse)
    assert int(err.item()) == 0
    for layer in range(layers):
        assert torch.equal(kc[layer].view(torch.int16), sw.k_caches[layer].view(torch.int16))
        assert torch.equal(vc[layer].view(torch.int16), sw.v_caches[layer].view(torch.int16))


def test_step_plan_reuse_skewed_split_units():
    """The skewed batch (one 32,768-token row split over many CTAs, combined by
    log-sum-exp): a second layer that reuses the first layer's plan gives the
    bits of a self-planned call, within tolerance of the oracle."""
    case = wl.skewed_decode(device=DEV)
    bt = torch.as_tensor(case.block_table, device=DEV)
    sl = torch.as_tensor(case.cache_seqlens, device=DEV)
    desc = pkv.cache_desc(case.k_cache)
    ws = pkv.decode_workspace(case.batch, case.max_blocks, 32, desc, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref_out, ref_lse, ref_err, _ = oracle_decode_compact(case)
    k2, v2 = case.k_cache.clone(), case.v_cache.clone()
    # layer 0 (makes the plan) on the copy, layer 1 (reuses it) on the original pools
    pkv.pkv_decode_attn(k2, v2, case.q, case.k_new, case.v_new, bt, sl, case.softmax_scale, workspace=ws,
                        err_flag=err, flags=_plan_flags(0))
    lse = torch.empty(case.batch, 32, dtype=torch.float32, device=DEV)
    out = pkv.pkv_decode_attn(case.k_cache, case.v_cache, case.q, case.k_new, case.v_new, bt, sl,
                              case.softmax_scale, lse=lse, workspace=ws, err_flag=err, flags=_plan_flags(1))
    lse_r = torch.empty(case.batch, 32, dtype=torch.float32, device=DEV)
    ws_r = pkv.decode_workspace(case.batch, case.max_blocks, 32, desc, DEV)
    out_r = pkv.pkv_decode_attn(k2, v2, case.q, None, None, bt, sl + 1, case.softmax_scale, lse=lse_r,
                                workspace=ws_r)  # attend-only over the copy that layer 0 appended to
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and ref_err == 0
    assert_close(f32(out), ref_out, what="skewed plan reuse")
    assert_lse_close(lse.cpu().numpy(), ref_lse)
    assert torch.equal(k2.view(torch.int16), case.k_cache.view(torch.int16))
    assert_close(f32(out_r), f32(out).astype(np.float64), what="attend-only after the append")


def test_step_plan_mismatch_and_stale_lengths_raise_plan_bit():
    """A plan made for another call shape (attend-only, no new token) is not
    used by a fused append + decode call: that call plans for itself, gives
    the exact outputs and sets PKV_ERR_PLAN.  A plan whose lengths differ
    from cache_seqlens is detected (PKV_ERR_PLAN set)."""
    sw = wl.batch_sweep(16, device=DEV, contiguous=False, layers=2)
    bt = torch.as_tensor(sw.block_table, device=DEV)
    desc = pkv.cache_desc(sw.k_caches[0])
    ws = pkv.decode_workspace(16, sw.max_blocks, 32, desc, DEV)
    lens = torch.as_tensor(sw.prompt_lens.astype(np.int32), device=DEV)
    (q, kn, vn), _ = wl.sweep_step_inputs(sw, 0, DEV, layers=2)
    kc, vc = sw.k_caches[0].clone(), sw.v_caches[0].clone()
    # an attend-only plan, then a fused call that asks for a plan (same workspace layout)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.pkv_decode_attn(kc, vc, q, None, None, bt, lens, sw.softmax_scale, workspace=ws, err_flag=err,
                        flags=pkv.api.DECODE_MAKE_PLAN)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kc, vc = sw.k_caches[0].clone(), sw.v_caches[0].clone()
    kr, vr = sw.k_caches[0].clone(), sw.v_caches[0].clone()
    out = pkv.pkv_decode_attn(kc, vc, q, kn, vn, bt, lens, sw.softmax_scale, workspace=ws, err_flag=err,
                              flags=pkv.api.DECODE_USE_PLAN)
    ref = pkv.pkv_decode_attn(kr, vr, q, kn, vn, bt, lens, sw.softmax_scale)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.api.ERR_PLAN
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(kc.view(torch.int16), kr.view(torch.int16))
    # a plan of these sizes, then lengths one longer without a new plan
    err.zero_()
    kc, vc = sw.k_caches[0].clone(), sw.v_caches[0].clone()
    pkv.pkv_decode_attn(kc, vc, q, kn, vn, bt, lens, sw.softmax_scale, workspace=ws, err_flag=err,
                        flags=pkv.api.DECODE_MAKE_PLAN)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    pkv.pkv_decode_attn(kc, vc, q, kn, vn, bt, lens + 1, sw.softmax_scale, workspace=ws, err_flag=err,
                        flags=pkv.api.DECODE_USE_PLAN)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.api.ERR_PLAN


def _random_case(seed, B, Hq, Hkv, D, P, lens, layout=wl.NHD, spare=7):
    g = torch.Generator().manual_seed(seed)
    lens = np.asarray(lens, np.int32)
    needed = (np.maximum(lens, 0) + 1 + P - 1) // P
    NP = int(needed.sum()) + 1 + spare
    max_blocks = int(needed.max()) + 1
    order = (torch.randperm(NP - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = wl.assign_pages(needed, NP, max_blocks, order)
    case = wl.PagedCase("rand", B, Hq, Hkv, D, P, NP, layout, max_blocks, bt, lens, 1.0 / math.sqrt(D),
                        q=wl._randn_bf16((B, Hq, D), g, "cpu").to(DEV))
    case.k_new = wl._randn_bf16((B, Hkv, D), g, "cpu").to(DEV)
    case.v_new = wl._randn_bf16((B, Hkv, D), g, "cpu").to(DEV)
    wl._fill_cache(case, g, DEV, "cpu")
    return case


SHAPES = [  # (Hq, Hkv, D, P)
    (32, 8, 128, 16), (32, 8, 128, 128), (4, 2, 64, 16), (8, 8, 64, 1), (16, 2, 64, 8),
    (64, 4, 64, 32), (8, 4, 256, 64), (8, 1, 256, 256), (16, 16, 128, 4), (32, 2, 128, 32),
]


@pytest.mark.parametrize("layout", [wl.NHD, wl.HND])
@pytest.mark.parametrize("Hq,Hkv,D,P", SHAPES)
def test_shapes_and_ragged_tails(layout, Hq, Hkv, D, P):
    lens = [0, 1, 31, 32, 33, 95, 257, 700]
    case = _random_case(100 + D + P + Hq, len(lens), Hq, Hkv, D, P, lens, layout)
    ref_out, ref_lse, ref_err, ref_k, ref_v = _oracle_full(case)
    out, lse = _run(case)
    assert ref_err == 0
    assert_close(f32(out), ref_out)
    assert_lse_close(lse.cpu().numpy(), ref_lse)
    assert hashlib.sha256(ref_k.tobytes()).hexdigest() == _sha(case.k_cache)
    assert hashlib.sha256(ref_v.tobytes()).hexdigest() == _sha(case.v_cache)


def test_single_key_is_exact():
    case = wl.tiny(device=DEV)
    case.cache_seqlens = np.zeros(case.batch, np.int32)
    out, lse = _run(case)
    want = wl.bits(case.v_new).repeat(case.group, axis=1)
    assert np.array_equal(wl.bits(out), want)  # 1 key: softmax weight exactly 1


def test_inactive_and_empty_rows():
    case = wl.tiny(device=DEV)
    case.cache_seqlens = np.array([-1, 0, 1, -5], np.int32)  # row 2 keeps its one cached token
    before = _sha(case.k_cache)
    out, lse = _run(case, with_new=False)
    o = f32(out)
    assert np.all(o[[0, 1, 3]] == 0) and np.all(np.isneginf(lse.cpu().numpy()[[0, 1, 3]]))
    assert np.all(np.isfinite(o[2]))
    assert _sha(case.k_cache) == before  # attend-only writes nothing


def test_bad_pages_and_overflow_flag_and_zero_rows():
    case = wl.tiny(device=DEV)
    case.block_table = case.block_table.copy()
    case.block_table[1, 1] = 0                     # null page used by a live token
    case.block_table[2, 0] = case.num_pages + 5    # out of range
    case.cache_seqlens = case.cache_seqlens.copy()
    case.cache_seqlens[3] = case.max_blocks * case.page_size  # L + 1 does not fit
    ref_out, ref_lse, ref_err, ref_k, ref_v = _oracle_full(case)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = _run(case, err=err)
    assert int(err.item()) == ref_err == (oracle.ERR_PAGE | oracle.ERR_OVERFLOW)
    o = f32(out)
    assert np.all(o[1:] == 0) and np.all(np.isneginf(lse.cpu().numpy()[1:]))
    assert_close(o[0], ref_out[0])
    assert hashlib.sha256(ref_k.tobytes()).hexdigest() == _sha(case.k_cache)
    assert hashlib.sha256(ref_v.tobytes()).hexdigest() == _sha(case.v_cache)


def test_page_permutation_bit_identical():
    case = wl.qwen3_decode(device=DEV, batch=8, num_pages=4096)
    out0, lse0 = _run(case, with_new=False)
    g = torch.Generator().manual_seed(5)
    perm = np.concatenate([[0], torch.randperm(case.num_pages - 1, generator=g).numpy() + 1])
    inv = torch.as_tensor(np.argsort(perm), device=DEV)
    case.k_cache = case.k_cache[inv].contiguous()  # physical page p -> perm[p]
    case.v_cache = case.v_cache[inv].contiguous()
    case.block_table = np.where(case.block_table > 0, perm[case.block_table], 0).astype(np.int32)
    out1, lse1 = _run(case, with_new=False)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_workspace_reuse_is_stable():
    case = wl.skewed_decode(device=DEV, batch=16, long_len=8192)
    desc = pkv.cache_desc(case.k_cache)
    ws = pkv.decode_workspace(case.batch, case.max_blocks, case.num_q_heads, desc, DEV)
    a, la = _run(case, with_new=False, workspace=ws)
    b, lb = _run(case, with_new=False, workspace=ws)
    assert torch.equal(a, b) and torch.equal(la, lb)
    assert int(ws[:4 * case.batch * 8].view(torch.int32).abs().sum().item()) == 0  # tickets back at zero


def test_large_batch_limit():
    lens = np.random.default_rng(0).integers(0, 40, 1024).astype(np.int32)
    case = _random_case(9, 1024, 8, 2, 64, 16, lens)
    ref_out, ref_lse, ref_err, _, _ = _oracle_full(case)
    out, lse = _run(case)
    assert_close(f32(out), ref_out)
    assert_lse_close(lse.cpu().numpy(), ref_lse)
    with pytest.raises(pkv.PkvError):
        big = _random_case(9, 1025, 8, 2, 64, 16, np.zeros(1025, np.int32))
        _run(big)


@pytest.mark.parametrize("graph", [False, True])
def test_overlap_prologue_launch_is_bit_identical(graph):
    """Back-to-back layers sharing one workspace, launched with programmatic
    dependent launch -- alone, and with the K/V stream started before the
    preceding kernel completes -- eagerly and inside a CUDA graph, give the
    same bits as plain launches."""
    layers = 3
    sw = wl.batch_sweep(32, device=DEV, contiguous=False, layers=layers)
    bt = torch.as_tensor(sw.block_table, device=DEV)
    sl = torch.as_tensor(sw.prompt_lens.astype(np.int32), device=DEV)  # step 0: the prompt is cached
    desc = pkv.cache_desc(sw.k_caches[0])
    ins = wl.sweep_step_inputs(sw, 0, DEV)
    results = []
    flag_sets = (0, pkv.api.DECODE_OVERLAP_PROLOGUE, pkv.api.DECODE_OVERLAP_PROLOGUE | pkv.api.DECODE_EARLY_KV)
    for flags in flag_sets:
        kc = [k.clone() for k in sw.k_caches]
        vc = [v.clone() for v in sw.v_caches]
        ws = pkv.decode_workspace(32, sw.max_blocks, 32, desc, DEV)
        outs = [torch.empty(32, 32, 128, dtype=torch.bfloat16, device=DEV) for _ in range(layers)]
        lses = [torch.empty(32, 32, dtype=torch.float32, device=DEV) for _ in range(layers)]

        def step():
            for layer, (q, kn, vn) in enumerate(ins):
                pkv.pkv_decode_attn(kc[layer], vc[layer], q, kn, vn, bt, sl, sw.softmax_scale, out=outs[layer],
                                    lse=lses[layer], workspace=ws, flags=flags)

        if graph and flags:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step()
            g.replay()
        else:
            step()
        torch.cuda.synchronize()
        results.append((outs, lses, kc, vc))
    o0, l0, k0, v0 = results[0]
    for o1, l1, k1, v1 in results[1:]:
        for layer in range(layers):
            assert torch.isfinite(o0[layer].float()).all()
            assert torch.equal(o0[layer].view(torch.int16), o1[layer].view(torch.int16))
            assert torch.equal(l0[layer].view(torch.int32), l1[layer].view(torch.int32))
            assert torch.equal(k0[layer].view(torch.int16), k1[layer].view(torch.int16))
            assert torch.equal(v0[layer].view(torch.int16), v1[layer].view(torch.int16))
