"""pkv_decode_attn_noalloc gives what pkv_decode_attn gives (GPU).

The no-allocation entry point serves callers that may not allocate device
memory themselves, for instance code running inside a host framework that
owns all device memory and forbids its plug-ins to allocate, or a serving
loop that must not call the allocator after start-up.  It takes no workspace
and uses an array compiled into the library instead.  Here two calls in a row
(the second attends the token the first appended) are compared, through the
C ABI, with the same two calls made with a caller workspace.

This file is named to be collected last, so that a run stopping at its first
failure has run every other test before it.  It passes on its own in a fresh
process as well as after the other tests (the array is cleared where it must
be by every call, not by test order).
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_decode_append_gb300 as pkv
from paged_kv_decode_append_gb300 import workloads as wl

from gpu_util import assert_close, assert_lse_close, f32

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _two_steps(case, call):
    """Runs two consecutive decode steps on private copies of the caches."""
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    bt = torch.as_tensor(case.block_table, device=DEV)
    outs = []
    for step in range(2):
        sl = torch.as_tensor((case.cache_seqlens + step).astype(np.int32), device=DEV)
        g = torch.Generator().manual_seed(50 + step)
        q = wl._randn_bf16(tuple(case.q.shape), g, "cpu").to(DEV)
        kn = wl._randn_bf16(tuple(case.k_new.shape), g, "cpu").to(DEV)
        vn = wl._randn_bf16(tuple(case.v_new.shape), g, "cpu").to(DEV)
        lse = torch.empty(case.batch, case.num_q_heads, dtype=torch.float32, device=DEV)
        out = call(kc, vc, q, kn, vn, bt, sl, lse)
        torch.cuda.synchronize()
        outs.append((f32(out), lse.cpu().numpy()))
    return outs, kc, vc


@pytest.mark.parametrize("maker", ["qwen3", "skewed"])
def test_noalloc_matches_workspace_entry_point(maker):
    case = (wl.qwen3_decode(device=DEV, batch=16, num_pages=4096) if maker == "qwen3"
            else wl.skewed_decode(device=DEV, batch=8, long_len=4096, num_pages=4096))
    # leave room for the second step's token in every row
    assert np.all((case.cache_seqlens + 2) <= case.max_blocks * case.page_size)

    def with_workspace(kc, vc, q, kn, vn, bt, sl, lse):
        return pkv.pkv_decode_attn(kc, vc, q, kn, vn, bt, sl, case.softmax_scale, lse=lse)

    def no_alloc(kc, vc, q, kn, vn, bt, sl, lse):
        out = torch.empty_like(q)
        return pkv.api.pkv_decode_attn_noalloc(kc, vc, q, kn, vn, bt, sl, case.softmax_scale, out=out, lse=lse)

    ref, k_ref, v_ref = _two_steps(case, with_workspace)
    got, k_got, v_got = _two_steps(case, no_alloc)
    for (o_ref, l_ref), (o_got, l_got) in zip(ref, got):
        assert np.all(np.isfinite(o_ref))
        assert_close(o_got, o_ref.astype(np.float64))
        assert_lse_close(l_got, l_ref.astype(np.float64))
    assert torch.equal(k_ref.view(torch.int16), k_got.view(torch.int16))
    assert torch.equal(v_ref.view(torch.int16), v_got.view(torch.int16))
