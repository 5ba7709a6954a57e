"""Python binding of the C ABI (``include/pkv.h``): same names, torch tensors
in, argument marshalling only.  Every step of the computation runs in the
library's CUDA kernels; there is no Python or CPU fallback, and a missing or
unloadable library raises.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib
from ._lib import CacheDesc

NHD = 0
HND = 1

OK, EINVAL, EUNSUPPORTED, ECUDA, ENOPAGES, EWORKSPACE, ETOOBIG = range(7)
DECODE_OVERLAP_PROLOGUE = 1  # pkv_decode_attn_ex flags (see include/pkv.h)
DECODE_EARLY_KV = 2
DECODE_MAKE_PLAN = 4
DECODE_USE_PLAN = 8
ERR_PAGE, ERR_OVERFLOW, ERR_TIMEOUT, ERR_QLEN, ERR_PLAN = 1, 2, 4, 8, 16


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _lib.load().pkv_status_str(status).decode()
        super().__init__(f"{what}: {msg} (status {status})")


def _check(status: int, what: str) -> None:
    if status != OK:
        raise PkvError(status, what)


def cache_desc(k_cache: torch.Tensor, layout: int = NHD) -> CacheDesc:
    """Descriptor of a pool tensor: NHD ``[pages, P, Hkv, D]`` or HND
    ``[pages, Hkv, P, D]``."""
    if k_cache.dim() != 4:
        raise ValueError("cache must be 4-D")
    if layout == NHD:
        n, p, h, d = k_cache.shape
    else:
        n, h, p, d = k_cache.shape
    return CacheDesc(n, p, h, d, layout)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _bf16(t, name):
    if t is None:
        return
    if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: expected a contiguous CUDA bfloat16 tensor")


def _i32(t, name):
    if t is None:
        return
    if t.dtype != torch.int32 or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name}: expected a contiguous CUDA int32 tensor")


def pkv_decode_workspace_size(batch: int, max_blocks: int, num_q_heads: int, desc: CacheDesc) -> int:
    return int(_lib.load().pkv_decode_workspace_size(batch, max_blocks, num_q_heads, ctypes.byref(desc)))


def decode_workspace(batch: int, max_blocks: int, num_q_heads: int, desc: CacheDesc, device) -> torch.Tensor:
    """A zero-filled workspace for pkv_decode_attn (reusable across calls)."""
    n = pkv_decode_workspace_size(batch, max_blocks, num_q_heads, desc)
    if n == 0:
        raise PkvError(EUNSUPPORTED, "pkv_decode_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def pkv_append(k_cache, v_cache, k_new, v_new, block_table, cache_seqlens, append_indptr=None, err_flag=None,
               layout: int = NHD) -> None:
    """Bit-copy ``k_new``/``v_new`` ``[T, Hkv, D]`` into their page slots."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new")):
        _bf16(t, n)
    for t, n in ((block_table, "block_table"), (cache_seqlens, "cache_seqlens"), (append_indptr, "append_indptr"),
                 (err_flag, "err_flag")):
        _i32(t, n)
    desc = cache_desc(k_cache, layout)
    st = _lib.load().pkv_append(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new),
                                k_new.shape[0], _ptr(append_indptr), _ptr(block_table), block_table.shape[1],
                                _ptr(cache_seqlens), cache_seqlens.shape[0], _ptr(err_flag),
                                _stream(k_cache.device))
    _check(st, "pkv_append")


def pkv_decode_attn(k_cache, v_cache, q, k_new, v_new, block_table, cache_seqlens, softmax_scale: float,
                    out=None, lse=None, workspace=None, err_flag=None, layout: int = NHD,
                    flags: int = 0) -> torch.Tensor:
    """Fused append + decode attention; returns ``out`` ``[B, Hq, D]`` bf16.
    ``flags`` (e.g. DECODE_OVERLAP_PROLOGUE) selects ``pkv_decode_attn_ex``."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (q, "q"), (k_new, "k_new"), (v_new, "v_new"),
                 (out, "out")):
        _bf16(t, n)
    for t, n in ((block_table, "block_table"), (cache_seqlens, "cache_seqlens"), (err_flag, "err_flag")):
        _i32(t, n)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse: expected contiguous float32")
    desc = cache_desc(k_cache, layout)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = decode_workspace(B, block_table.shape[1], Hq, desc, q.device)
    args = (ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(block_table),
            block_table.shape[1], _ptr(cache_seqlens), B, Hq, float(softmax_scale), _ptr(out), _ptr(lse),
            _ptr(workspace), workspace.numel(), _ptr(err_flag), _stream(q.device))
    if flags:
        _check(_lib.load().pkv_decode_attn_ex(*args, int(flags)), "pkv_decode_attn_ex")
    else:
        _check(_lib.load().pkv_decode_attn(*args), "pkv_decode_attn")
    return out


def pkv_decode_attn_noalloc(k_cache, v_cache, q, k_new, v_new, block_table, cache_seqlens, softmax_scale: float,
                            out=None, lse=None, err_flag=None, layout: int = NHD) -> torch.Tensor:
    """pkv_decode_attn for callers that cannot allocate device memory: no
    workspace argument, the library's built-in scratch is used instead (see
    include/pkv.h for its size limit and sharing rules).  Pass ``out`` to
    avoid the allocation of a fresh output tensor here."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (q, "q"), (k_new, "k_new"), (v_new, "v_new"),
                 (out, "out")):
        _bf16(t, n)
    for t, n in ((block_table, "block_table"), (cache_seqlens, "cache_seqlens"), (err_flag, "err_flag")):
        _i32(t, n)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse: expected contiguous float32")
    desc = cache_desc(k_cache, layout)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    st = _lib.load().pkv_decode_attn_noalloc(
        ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(block_table),
        block_table.shape[1], _ptr(cache_seqlens), B, Hq, float(softmax_scale), _ptr(out), _ptr(lse), _ptr(err_flag),
        _stream(q.device))
    _check(st, "pkv_decode_attn_noalloc")
    return out


def pkv_decode_bucket(batch: int) -> int:
    """Graph batch size serving ``batch`` rows (0 if out of range)."""
    return int(_lib.load().pkv_decode_bucket(batch))


class DecodeStep:
    """``pkv_decode_step_*``: every layer's fused append + decode of one step
    captured once as a CUDA graph.  The tensors given here are baked in:
    write each step's inputs (``q``, ``k_new``, ``v_new``, ``cache_seqlens``)
    into them, then call :meth:`launch`."""

    def __init__(self, k_caches, v_caches, q, k_new, v_new, block_table, cache_seqlens, softmax_scale: float, out,
                 lse=None, workspace=None, err_flag=None, layout: int = NHD, flags: int = 0):
        layers = len(k_caches)
        if not (len(v_caches) == len(q) == len(out) == layers) or layers < 1:
            raise ValueError("one k / v cache, q and out per layer")
        for lst, n in ((k_caches, "k_caches"), (v_caches, "v_caches"), (q, "q"), (out, "out"),
                       (k_new or [], "k_new"), (v_new or [], "v_new")):
            for t in lst:
                _bf16(t, n)
        for t, n in ((block_table, "block_table"), (cache_seqlens, "cache_seqlens"), (err_flag, "err_flag")):
            _i32(t, n)
        desc = cache_desc(k_caches[0], layout)
        B, Hq, D = q[0].shape
        if workspace is None:
            workspace = decode_workspace(B, block_table.shape[1], Hq, desc, q[0].device)
        arr = ctypes.c_void_p * layers

        def ptrs(lst):
            return None if lst is None else arr(*[t.data_ptr() if t is not None else None for t in lst])

        self._keep = (k_caches, v_caches, q, k_new, v_new, block_table, cache_seqlens, out, lse, workspace, err_flag)
        self._lib = _lib.load()
        handle = ctypes.c_void_p()
        st = self._lib.pkv_decode_step_create(
            ctypes.byref(desc), layers, ptrs(k_caches), ptrs(v_caches), ptrs(q), ptrs(k_new), ptrs(v_new),
            _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens), B, Hq, float(softmax_scale), ptrs(out),
            ptrs(lse), _ptr(workspace), workspace.numel(), _ptr(err_flag), int(flags), ctypes.byref(handle))
        _check(st, "pkv_decode_step_create")
        self._h = handle
        self.device = q[0].device

    def launch(self) -> None:
        _check(self._lib.pkv_decode_step_launch(self._h, _stream(self.device)), "pkv_decode_step_launch")

    def __del__(self):
        if getattr(self, "_h", None):
            self._lib.pkv_decode_step_destroy(self._h)
            self._h = None


def pkv_prefill_workspace_size(batch: int, total_q: int, num_q_heads: int, desc: CacheDesc) -> int:
    return int(_lib.load().pkv_prefill_workspace_size(batch, total_q, num_q_heads, ctypes.byref(desc)))


def prefill_workspace(batch: int, total_q: int, num_q_heads: int, desc: CacheDesc, device) -> torch.Tensor:
    """A workspace for pkv_prefill_attn (needs no initialisation)."""
    n = pkv_prefill_workspace_size(batch, total_q, num_q_heads, desc)
    if n == 0:
        raise PkvError(EUNSUPPORTED, "pkv_prefill_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def pkv_prefill_attn(k_cache, v_cache, q, qo_indptr, kv_lens, block_table, softmax_scale: float, out=None,
                     lse=None, workspace=None, err_flag=None, layout: int = NHD) -> torch.Tensor:
    """Ragged end-aligned causal prefill over the paged cache; ``q`` is
    ``[total_q, Hq, D]``, request b owns rows ``qo_indptr[b]:qo_indptr[b+1]``
    and sees ``kv_lens[b]`` keys.  Returns ``out`` ``[total_q, Hq, D]`` bf16."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (q, "q"), (out, "out")):
        _bf16(t, n)
    for t, n in ((qo_indptr, "qo_indptr"), (kv_lens, "kv_lens"), (block_table, "block_table"),
                 (err_flag, "err_flag")):
        _i32(t, n)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse: expected contiguous float32")
    desc = cache_desc(k_cache, layout)
    total_q, Hq, D = q.shape
    B = kv_lens.shape[0]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = prefill_workspace(B, total_q, Hq, desc, q.device)
    st = _lib.load().pkv_prefill_attn(
        ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(q), _ptr(qo_indptr), _ptr(kv_lens),
        _ptr(block_table), block_table.shape[1], B, Hq, total_q, float(softmax_scale), _ptr(out), _ptr(lse),
        _ptr(workspace), workspace.numel(), _ptr(err_flag), _stream(q.device))
    _check(st, "pkv_prefill_attn")
    return out


def pkv_mixed_workspace_size(batch: int, total_q: int, max_blocks: int, num_q_heads: int, max_qlen: int,
                             decode_max_qlen: int, desc: CacheDesc) -> int:
    return int(_lib.load().pkv_mixed_workspace_size(batch, total_q, max_blocks, num_q_heads, max_qlen,
                                                    decode_max_qlen, ctypes.byref(desc)))


def default_decode_max_qlen(num_q_heads: int, num_kv_heads: int) -> int:
    """Longest row the decode kernel takes by default in a mixed step: up to
    16 (query, head) columns of a kv head (two decode units)."""
    return max(1, 16 // max(1, num_q_heads // num_kv_heads))


def mixed_workspace(batch: int, total_q: int, max_blocks: int, num_q_heads: int, max_qlen: int,
                    decode_max_qlen: int, desc: CacheDesc, device) -> torch.Tensor:
    """A zero-filled workspace for pkv_mixed_attn (reusable across calls)."""
    n = pkv_mixed_workspace_size(batch, total_q, max_blocks, num_q_heads, max_qlen, decode_max_qlen, desc)
    if n == 0:
        raise PkvError(EUNSUPPORTED, "pkv_mixed_workspace_size")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def pkv_mixed_attn(k_cache, v_cache, q, k_new, v_new, qo_indptr, block_table, cache_seqlens, softmax_scale: float,
                   max_qlen: int, decode_max_qlen: int | None = None, out=None, lse=None, workspace=None,
                   err_flag=None, layout: int = NHD) -> torch.Tensor:
    """One step of a mixed batch: row b appends its ``qo_indptr[b+1] -
    qo_indptr[b]`` new tokens (``k_new``/``v_new`` ``[total_q, Hkv, D]``, or
    both None when already appended) after its ``cache_seqlens[b]`` cached
    ones, then its query i attends keys ``0 .. kv_b - q_b + i``.  Rows of up
    to ``decode_max_qlen`` queries run on the decode kernel, longer ones on
    the prefill kernel.  Returns ``out`` ``[total_q, Hq, D]`` bf16."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (q, "q"), (k_new, "k_new"), (v_new, "v_new"),
                 (out, "out")):
        _bf16(t, n)
    for t, n in ((qo_indptr, "qo_indptr"), (block_table, "block_table"), (cache_seqlens, "cache_seqlens"),
                 (err_flag, "err_flag")):
        _i32(t, n)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise ValueError("lse: expected contiguous float32")
    desc = cache_desc(k_cache, layout)
    total_q, Hq, D = q.shape
    B = cache_seqlens.shape[0]
    if decode_max_qlen is None:
        decode_max_qlen = default_decode_max_qlen(Hq, desc.num_kv_heads)
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = mixed_workspace(B, total_q, block_table.shape[1], Hq, max_qlen, decode_max_qlen, desc,
                                    q.device)
    st = _lib.load().pkv_mixed_attn(
        ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(qo_indptr),
        _ptr(block_table), block_table.shape[1], _ptr(cache_seqlens), B, Hq, total_q, int(max_qlen),
        int(decode_max_qlen), float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _ptr(err_flag), _stream(q.device))
    _check(st, "pkv_mixed_attn")
    return out


def pkv_pool_bytes(desc: CacheDesc) -> int:
    return int(_lib.load().pkv_pool_bytes(ctypes.byref(desc)))


def pkv_validate_host(desc: CacheDesc, block_table: np.ndarray, seqlens: np.ndarray, extra_tokens: int):
    """Host check of a block table; returns (status, first bad row or -1)."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    bad = ctypes.c_int32(-1)
    st = _lib.load().pkv_validate_host(ctypes.byref(desc), bt.ctypes.data_as(_lib.I32P), bt.shape[1],
                                       sl.ctypes.data_as(_lib.I32P), sl.shape[0], extra_tokens, ctypes.byref(bad))
    return st, bad.value


class PagePool:
    """Host page pool (``pkv_pool_*``): pages 1..num_pages-1, page 0 never
    handed out; a fresh pool hands pages out in ascending order."""

    def __init__(self, num_pages: int):
        self._lib = _lib.load()
        self._p = self._lib.pkv_pool_create(num_pages)
        if not self._p:
            raise PkvError(EINVAL, "pkv_pool_create")

    def __del__(self):
        if getattr(self, "_p", None):
            self._lib.pkv_pool_destroy(self._p)
            self._p = None

    @property
    def num_free(self) -> int:
        return int(self._lib.pkv_pool_num_free(self._p))

    def alloc(self, n: int) -> np.ndarray:
        out = np.zeros(max(n, 0), np.int32)
        _check(self._lib.pkv_pool_alloc(self._p, n, out.ctypes.data_as(_lib.I32P)), "pkv_pool_alloc")
        return out

    def free(self, pages) -> None:
        pages = np.ascontiguousarray(pages, dtype=np.int32)
        _check(self._lib.pkv_pool_free(self._p, pages.ctypes.data_as(_lib.I32P), pages.size), "pkv_pool_free")

    def shuffle(self, seed: int) -> None:
        _check(self._lib.pkv_pool_shuffle(self._p, seed), "pkv_pool_shuffle")

    def reserve(self, row: np.ndarray, page_size: int, cur_len: int, new_len: int) -> None:
        """Extend one block-table row (an int32 numpy view) from cur_len to new_len tokens."""
        assert row.dtype == np.int32 and row.flags.c_contiguous
        _check(self._lib.pkv_table_reserve(self._p, row.ctypes.data_as(_lib.I32P), row.size, page_size, cur_len,
                                           new_len), "pkv_table_reserve")

    def release(self, row: np.ndarray, page_size: int, length: int) -> None:
        assert row.dtype == np.int32 and row.flags.c_contiguous
        _check(self._lib.pkv_table_release(self._p, row.ctypes.data_as(_lib.I32P), row.size, page_size, length),
               "pkv_table_release")
