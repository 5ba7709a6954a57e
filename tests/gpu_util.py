"""Helpers shared by the GPU parity tests: run the oracle on the same seeded
inputs and compare within the stated tolerance."""
import os

import numpy as np
import torch

import oracle
from paged_kv_decode_append_gb300 import workloads as wl

# Attention outputs (bf16 in, fp32 accumulate, bf16 out) must be within
# max-abs 1e-2 and max-rel 1e-2 of the fp64 oracle.  Relative error is taken
# over elements with |ref| >= 1e-2 (below that, fp32 rounding of the softmax
# sum dominates any relative measure).  One allowance on the abs bound: the
# output format is bf16, whose rounding alone moves a value by up to half an
# ulp, 2^-9 |ref| relative; from |ref| >= 4 that half-ulp is 2^-6 > 1e-2, so
# there (and only there) the abs bound is 1e-2 plus the half-ulp of ref.
ATOL = 1e-2
RTOL = 1e-2
REL_FLOOR = 1e-2
LSE_ATOL = 1e-2
ULP_FROM = 4.0

# (test, what, max-abs, max-rel, elements) of every comparison in this
# session; conftest prints them after the run so the margins show in the log.
MARGINS = []


def _record(what, max_abs, max_rel, n):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    MARGINS.append((test, what, max_abs, max_rel, n))
    print(f"{test} {what}: max-abs {max_abs:.3e} max-rel {max_rel:.3e} over {n} elements")


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = "out"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    big = np.abs(ref) >= REL_FLOOR
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    _record(what, max_abs, max_rel, int(err.size))
    bound = np.where(np.abs(ref) >= ULP_FROM, ATOL + bf16_half_ulp(ref), ATOL)
    excess = err - bound
    assert not (excess > 0).any(), (f"{what}: max-abs {max_abs:.3e} > {ATOL} "
                                    f"(+ bf16 output half-ulp where |ref| >= {ULP_FROM})")
    assert max_rel <= RTOL, f"{what}: max-rel {max_rel:.3e} > {RTOL}"
    return max_abs, max_rel


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significand bits)."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 8)


def assert_lse_close(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    inf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf), "lse: -inf pattern differs"
    if (~inf).any():
        err = float(np.abs(got[~inf] - ref[~inf]).max())
        _record("lse", err, 0.0, int((~inf).sum()))
        assert err <= LSE_ATOL, f"lse: max-abs {err:.3e}"


def f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def desc_of(case):
    return oracle.CacheDesc(case.num_pages, case.page_size, case.num_kv_heads, case.head_dim, case.layout)


def oracle_decode_compact(case, rows=None, with_new=True, sel=None):
    """Oracle decode for `rows` using a compact host copy of only the pages
    those rows touch (large pools stay on the device).  Returns out, lse
    indexed by position in `rows`, plus the compact inputs."""
    rows = list(range(case.batch)) if rows is None else list(rows)
    L = case.cache_seqlens[rows]
    need = np.maximum(L, 0) + (1 if with_new else 0)
    k, v, bt = wl.compact_rows(case.k_cache, case.v_cache, case.block_table, rows, need, case.page_size)
    d = oracle.CacheDesc(k.shape[0], case.page_size, case.num_kv_heads, case.head_dim, case.layout)
    q = wl.bits(case.q)[rows]
    kn = wl.bits(case.k_new)[rows] if with_new else None
    vn = wl.bits(case.v_new)[rows] if with_new else None
    out, lse, err, err_rows = oracle.decode(d, k, v, q, kn, vn, bt, L, case.softmax_scale, sel=sel)
    return out, lse, err, err_rows
