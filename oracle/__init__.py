"""fp64 CPU oracle for paged KV append, decode attention, causal prefill and
the mixed step (chunked prefill and multi-token decode rows in one batch).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library (``paged_kv_decode_append_gb300``) never imports, loads or
calls it, and the two share no code: the oracle is ``oracle.c`` (plain C,
fp64, loops in logical token order) plus this ctypes wrapper.

What it follows (page title, section):

* "mini-infer系统实战-06 True PagedAttention", sections 1 and 3: one call
  appends the new token's K/V at index ``cache_seqlens[b]`` via
  ``block_table`` and attends over the paged cache
  ``[num_blocks, block_size, num_kv_heads, head_dim]``.  The oracle is the
  gather formulation that the page replaces: it gathers keys/values in
  logical order and applies textbook softmax attention in fp64.
* "[flashinfer] H100 D256 paged attention cuDNN auto-dispatch", code
  analysis part 1: end-aligned causal rule (query i of q sees kv-q+i+1 keys)
  and the pair count ``Hq * sum q(2kv-q+1)/2``; HND page layout.
* "flex_attention + paged KV + CUDA graphs vs vLLM", "What broke
  correctness": page 0 is a null slot; a row with no visible key gives
  out = 0 and lse = -inf, never NaN.  Same page, "What's left on the
  table": vLLM interleaves prefill chunks and decode tokens within one step;
  ``mixed`` is that step (append every row's new tokens, then the
  end-aligned causal rule over the grown cache).

Pins (tests under ``tests/test_oracle_*.py``) tie it to torch's fp64 SDPA on
dense gathers, closed forms (scale 0, constant V, one key), page-permutation
invariance and the printed pair-count formula.

All bf16 data is passed as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

NHD = 0
HND = 1
ERR_PAGE = 1
ERR_OVERFLOW = 2
ERR_QLEN = 8


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc into ``oracle/liboracle.so``.

    ``-ffp-contract=off`` keeps the fp64 arithmetic identical on x86 and Arm
    (no fused multiply-add contraction).  OpenMP is used when gcc has it.
    """
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no C compiler found to build the oracle")
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = [cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cache(ctypes.Structure):
    _fields_ = [
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("layout", ctypes.c_int32),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        lib.oracle_append.argtypes = [P, P, P, P, P, P, P, i32, P, i32, P]
        lib.oracle_append.restype = i32
        lib.oracle_decode.argtypes = [P, P, P, P, P, P, P, i32, P, i32, i32, ctypes.c_double,
                                      P, i32, P, P, P, i32]
        lib.oracle_decode.restype = i32
        lib.oracle_prefill.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, ctypes.c_double,
                                       P, i32, P, P, P, i32]
        lib.oracle_prefill.restype = ctypes.c_int64
        i64 = ctypes.c_int64
        lib.oracle_mixed.argtypes = [P, P, P, P, P, P, P, i64, P, i32, P, i32, i32, i64, ctypes.c_double,
                                     P, i32, P, P, P, i32]
        lib.oracle_mixed.restype = i32
        lib.oracle_max_threads.argtypes = [i32]
        lib.oracle_max_threads.restype = i32
        _lib = lib
    return _lib


@dataclass(frozen=True)
class CacheDesc:
    """Physical page pool geometry: ``num_pages`` pages of ``page_size`` tokens,
    ``num_kv_heads`` heads of ``head_dim`` values; layout NHD
    ``[pages, page_size, Hkv, D]`` or HND ``[pages, Hkv, page_size, D]``."""

    num_pages: int
    page_size: int
    num_kv_heads: int
    head_dim: int
    layout: int = NHD

    def _c(self) -> _Cache:
        return _Cache(self.num_pages, self.page_size, self.num_kv_heads, self.head_dim, self.layout)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a, name):
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"{name}: expected uint16 bf16 bit patterns, got {a.dtype}")
    return np.ascontiguousarray(a)


def _i32(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _sel(sel):
    if sel is None:
        return None, 0
    s = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 2))
    return s, s.shape[0]


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def append(desc: CacheDesc, k_cache, v_cache, k_new, v_new, append_indptr, block_table, cache_seqlens):
    """In-place bit-copy append into ``k_cache``/``v_cache`` (uint16 arrays).

    Returns ``(err_bits, err_rows)``."""
    lib = _load()
    c = desc._c()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k_new, v_new = _u16(k_new, "k_new"), _u16(v_new, "v_new")
    bt, sl, ip = _i32(block_table), _i32(cache_seqlens), _i32(append_indptr)
    B = sl.shape[0]
    err_rows = np.zeros(B, np.int32)
    err = lib.oracle_append(ctypes.byref(c), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                            _ptr(ip), _ptr(bt), bt.shape[1], _ptr(sl), B, _ptr(err_rows))
    return err, err_rows


def decode(desc: CacheDesc, k_cache, v_cache, q, k_new, v_new, block_table, cache_seqlens,
           softmax_scale, sel=None, nthreads: int = 0):
    """Fused append + decode attention in fp64.

    ``k_cache``/``v_cache`` are modified in place (the append), so pass copies
    when the originals are still needed.  ``q`` is ``[B, Hq, D]``; ``k_new``
    and ``v_new`` are ``[B, Hkv, D]`` or both None (attend only).  ``sel`` is an
    optional ``[n, 2]`` list of (row, q-head) pairs to compute.  Returns
    ``(out [B,Hq,D] f64, lse [B,Hq] f64, err_bits, err_rows)``; entries not in
    ``sel`` are left as NaN.
    """
    lib = _load()
    c = desc._c()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    q = _u16(q, "q")
    k_new, v_new = _u16(k_new, "k_new"), _u16(v_new, "v_new")
    bt, sl = _i32(block_table), _i32(cache_seqlens)
    B, Hq, D = q.shape
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    err_rows = np.zeros(B, np.int32)
    s, ns = _sel(sel)
    err = lib.oracle_decode(ctypes.byref(c), _ptr(k_cache), _ptr(v_cache), _ptr(q), _ptr(k_new),
                            _ptr(v_new), _ptr(bt), bt.shape[1], _ptr(sl), B, Hq,
                            float(softmax_scale), _ptr(s), ns, _ptr(out), _ptr(lse),
                            _ptr(err_rows), int(nthreads))
    return out, lse, err, err_rows


def prefill(desc: CacheDesc, k_cache, v_cache, q, qo_indptr, kv_lens, block_table, softmax_scale,
            sel=None, nthreads: int = 0):
    """Ragged end-aligned causal prefill in fp64 (no append).

    ``q`` is ``[total_q, Hq, D]``.  Returns ``(out, lse, pairs, err_rows)``
    where ``pairs`` counts the visited (query, key, head) triples (-1 for
    malformed requests, -2 when a row has a data error)."""
    lib = _load()
    c = desc._c()
    q = _u16(q, "q")
    ip, kl, bt = _i32(qo_indptr), _i32(kv_lens), _i32(block_table)
    T, Hq, D = q.shape
    B = kl.shape[0]
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    err_rows = np.zeros(B, np.int32)
    s, ns = _sel(sel)
    pairs = lib.oracle_prefill(ctypes.byref(c), _ptr(np.ascontiguousarray(k_cache)),
                               _ptr(np.ascontiguousarray(v_cache)), _ptr(q), _ptr(ip), _ptr(kl),
                               _ptr(bt), bt.shape[1], B, Hq, float(softmax_scale), _ptr(s), ns,
                               _ptr(out), _ptr(lse), _ptr(err_rows), int(nthreads))
    return out, lse, int(pairs), err_rows


def mixed(desc: CacheDesc, k_cache, v_cache, q, k_new, v_new, qo_indptr, block_table, cache_seqlens,
          softmax_scale, max_qlen=None, sel=None, nthreads: int = 0):
    """One step of a mixed batch in fp64: row b appends its
    ``qo_indptr[b+1] - qo_indptr[b]`` new tokens (when ``k_new``/``v_new``
    ``[total_q, Hkv, D]`` are given) after its ``cache_seqlens[b]`` cached
    ones, then its query i sees keys ``0 .. kv_b - q_b + i`` (end aligned).

    ``k_cache``/``v_cache`` are modified in place (pass copies).  ``q`` is
    ``[total_q, Hq, D]``; ``max_qlen`` (default: no limit) is the longest
    query range accepted.  Returns ``(out [total_q,Hq,D], lse [total_q,Hq],
    err_bits, err_rows)``; entries not computed (not in ``sel``, or owned by
    no row) are NaN."""
    lib = _load()
    c = desc._c()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    q = _u16(q, "q")
    k_new, v_new = _u16(k_new, "k_new"), _u16(v_new, "v_new")
    ip, bt, sl = _i32(qo_indptr), _i32(block_table), _i32(cache_seqlens)
    T, Hq, D = q.shape
    B = sl.shape[0]
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    err_rows = np.zeros(B, np.int32)
    s, ns = _sel(sel)
    mq = (1 << 62) if max_qlen is None else int(max_qlen)
    err = lib.oracle_mixed(ctypes.byref(c), _ptr(k_cache), _ptr(v_cache), _ptr(q), _ptr(k_new), _ptr(v_new),
                           _ptr(ip), T, _ptr(bt), bt.shape[1], _ptr(sl), B, Hq, mq, float(softmax_scale),
                           _ptr(s), ns, _ptr(out), _ptr(lse), _ptr(err_rows), int(nthreads))
    return out, lse, err, err_rows


def max_threads(nthreads: int = 0) -> int:
    """Threads the oracle's parallel loops use for ``nthreads`` (0 = default)."""
    return int(_load().oracle_max_threads(int(nthreads)))
