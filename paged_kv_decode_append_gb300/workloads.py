"""Seeded synthetic inputs for the paged-KV decode/prefill workloads.

This module only draws random numbers and lays pages out: it holds none of
the attention arithmetic.  The tests, the benchmark and the oracle checks all
take their inputs from here, so the CUDA path and the oracle see identical
bytes.

Workload shapes follow the pages' workloads:

* ``tiny``     -- 4 rows, Hq=4, Hkv=2, D=64, page 16, lengths {17,33,1,64},
                  24 physical pages (page 0 null) handed out by a seeded shuffle.
* ``qwen3``    -- one Qwen3-4B-shaped attention layer (Hq=32, Hkv=8, D=128),
                  B=32, page 16, lengths uniform in [512, 1024], pages drawn at
                  random from a 65,536-page pool ("flex_attention + paged KV +
                  CUDA graphs vs vLLM", Setup: Qwen3-4B-Base, bf16).
* ``sweep``    -- the batch sweep of the same page's "Batch-size sweep" table:
                  B in {8..256}, page 128, prompt uniform in [64, 512], then up
                  to 512 decode steps over 36 per-layer caches that share one
                  block table; contiguous or shuffled page layout.
* ``skewed``   -- B=64, page 16, row 0 holds 32,768 tokens, the others
                  clip(floor(lognormal(6.5, 0.8)), 128, 4096).
* ``prefill``  -- ragged causal prefill, B=8, Hq=48, Hkv=6, D=256, page 16 HND,
                  q uniform in [65, 1023], kv = q + uniform [0, 2048]
                  ("[flashinfer] H100 D256 paged attention cuDNN
                  auto-dispatch": HND, page 16, D=256, Hq up to 48).
* ``spec``     -- speculative decode on the Qwen3-shaped layer: B=32 rows of
                  4 new tokens on cached lengths U[512, 1024].
* ``chunked``  -- a chunked-prefill serving step on the same layer: 4 chunks
                  of 496 tokens on prefixes U[0, 2048] plus 60 decode rows on
                  U[512, 1024] ("flex_attention + paged KV + CUDA graphs vs
                  vLLM", "What's left on the table": prefill chunks and decode
                  tokens interleaved in one step).

Values are float32 N(0, 1) draws rounded to bf16 (round to nearest even).
Every cache slot that holds no token yet -- page 0, unused pages, and the
slots at or past a row's length, including the slot the next append fills --
holds a bf16 NaN, so any read of a slot outside a row's live tokens poisons
the result instead of passing silently.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

NHD = 0
HND = 1
BF16_NAN_BITS = 0x7FC0

SWEEP_BATCHES = (8, 16, 32, 64, 128, 256)
SWEEP_LAYERS = 36
SWEEP_DECODE_STEPS = 512


@dataclass
class PagedCase:
    """One paged-attention problem.  Host copies are numpy; tensors live on
    ``device``.  ``cache_seqlens`` are lengths BEFORE the append."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    layout: int
    max_blocks: int
    block_table: np.ndarray  # int32 [B, max_blocks]; unused entries 0
    cache_seqlens: np.ndarray  # int32 [B]
    softmax_scale: float
    q: torch.Tensor  # bf16 [B, Hq, D] (decode) or [total_q, Hq, D] (prefill)
    k_new: torch.Tensor | None = None  # bf16 [B, Hkv, D]
    v_new: torch.Tensor | None = None
    k_cache: torch.Tensor | None = None  # bf16 pool, NHD or HND
    v_cache: torch.Tensor | None = None
    qo_indptr: np.ndarray | None = None  # prefill / mixed step, int32 [B+1]
    kv_lens: np.ndarray | None = None  # prefill only, int32 [B]
    extra: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def pool_shape(self) -> tuple:
        if self.layout == NHD:
            return (self.num_pages, self.page_size, self.num_kv_heads, self.head_dim)
        return (self.num_pages, self.num_kv_heads, self.page_size, self.head_dim)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn_bf16(shape, g: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def _nan_pool(shape, device) -> torch.Tensor:
    return torch.full(shape, BF16_NAN_BITS, dtype=torch.int16, device=device).view(torch.bfloat16)


def scatter_tokens(pool: torch.Tensor, layout: int, page_size: int, pages: np.ndarray,
                   slots: np.ndarray, values: torch.Tensor) -> None:
    """Write ``values`` ``[n, Hkv, D]`` into the pool at (pages[i], slots[i])."""
    n_pages, _, _, D = pool.shape
    if layout == NHD:
        Hkv = pool.shape[2]
        flat = pool.view(n_pages * page_size, Hkv, D)
        idx = torch.as_tensor(pages.astype(np.int64) * page_size + slots, device=pool.device)
        flat[idx] = values
    else:
        Hkv = pool.shape[1]
        perm = pool.permute(0, 2, 1, 3)  # [pages, P, Hkv, D] view
        pg = torch.as_tensor(pages.astype(np.int64), device=pool.device)
        sl = torch.as_tensor(slots.astype(np.int64), device=pool.device)
        perm[pg, sl] = values


def assign_pages(needed: np.ndarray, num_pages: int, max_blocks: int, order: np.ndarray) -> np.ndarray:
    """Block table whose row b takes the next ``needed[b]`` pages of ``order``."""
    B = needed.shape[0]
    bt = np.zeros((B, max_blocks), np.int32)
    pos = 0
    for b in range(B):
        n = int(needed[b])
        bt[b, :n] = order[pos:pos + n]
        pos += n
    if pos > len(order):
        raise ValueError("page pool too small")
    return bt


def _fill_cache(case: PagedCase, g: torch.Generator, device, data_device) -> None:
    """Allocate NaN pools and write seeded tokens 0..L_b-1 of every row."""
    case.k_cache = _nan_pool(case.pool_shape(), device)
    case.v_cache = _nan_pool(case.pool_shape(), device)
    lens = case.kv_lens if case.kv_lens is not None else case.cache_seqlens
    rows = [np.arange(max(int(L), 0), dtype=np.int64) for L in lens]
    b_idx = np.concatenate([np.full(len(r), b, np.int64) for b, r in enumerate(rows)]) if rows else np.zeros(0, np.int64)
    t_idx = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    if t_idx.size == 0:
        return
    pages = case.block_table[b_idx, t_idx // case.page_size]
    slots = t_idx % case.page_size
    n = t_idx.size
    kv_shape = (n, case.num_kv_heads, case.head_dim)
    k = _randn_bf16(kv_shape, g, data_device).to(device)
    v = _randn_bf16(kv_shape, g, data_device).to(device)
    scatter_tokens(case.k_cache, case.layout, case.page_size, pages, slots, k)
    scatter_tokens(case.v_cache, case.layout, case.page_size, pages, slots, v)


def tiny(device="cpu", seed: int = 0) -> PagedCase:
    """B=4, Hq=4, Hkv=2, D=64, page 16, lengths {17,33,1,64}, 24 pages."""
    g = _gen(seed)
    B, Hq, Hkv, D, P, NP = 4, 4, 2, 64, 16, 24
    L = np.array([17, 33, 1, 64], np.int32)
    needed = (L + 1 + P - 1) // P
    max_blocks = int(needed.max())
    order = (torch.randperm(NP - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = assign_pages(needed, NP, max_blocks, order)
    case = PagedCase("tiny", B, Hq, Hkv, D, P, NP, NHD, max_blocks, bt, L, 1.0 / math.sqrt(D),
                     q=_randn_bf16((B, Hq, D), g, "cpu").to(device))
    case.k_new = _randn_bf16((B, Hkv, D), g, "cpu").to(device)
    case.v_new = _randn_bf16((B, Hkv, D), g, "cpu").to(device)
    _fill_cache(case, g, device, "cpu")
    return case


def qwen3_decode(device="cpu", seed: int = 1, batch: int = 32, num_pages: int = 65536,
                 min_len: int = 512, max_len: int = 1024) -> PagedCase:
    """One Qwen3-4B-shaped layer: B=32, Hq=32, Hkv=8, D=128, page 16,
    lengths uniform in [512, 1024], pages from a seeded permutation of the
    65,536-page pool."""
    g = _gen(seed)
    Hq, Hkv, D, P = 32, 8, 128, 16
    L = torch.randint(min_len, max_len + 1, (batch,), generator=g).numpy().astype(np.int32)
    max_blocks = (max_len + 1 + P - 1) // P
    needed = (L + 1 + P - 1) // P
    order = (torch.randperm(num_pages - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = assign_pages(needed, num_pages, max_blocks, order)
    case = PagedCase("qwen3", batch, Hq, Hkv, D, P, num_pages, NHD, max_blocks, bt, L,
                     1.0 / math.sqrt(D), q=_randn_bf16((batch, Hq, D), g, "cpu").to(device))
    case.k_new = _randn_bf16((batch, Hkv, D), g, "cpu").to(device)
    case.v_new = _randn_bf16((batch, Hkv, D), g, "cpu").to(device)
    _fill_cache(case, g, device, "cpu")
    return case


def skewed_decode(device="cpu", seed: int = 3, batch: int = 64, long_len: int = 32768,
                  num_pages: int = 65536) -> PagedCase:
    """B=64, page 16: row 0 holds 32,768 tokens, rows 1.. hold
    clip(floor(lognormal(6.5, 0.8)), 128, 4096); pages shuffled in a 65,536
    page pool."""
    g = _gen(seed)
    Hq, Hkv, D, P = 32, 8, 128, 16
    ln = torch.empty(batch - 1, dtype=torch.float64).log_normal_(6.5, 0.8, generator=g)
    rest = np.clip(np.floor(ln.numpy()), 128, 4096).astype(np.int32)
    L = np.concatenate([[long_len], rest]).astype(np.int32)
    max_blocks = (int(L.max()) + 1 + P - 1) // P
    needed = (L + 1 + P - 1) // P
    order = (torch.randperm(num_pages - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = assign_pages(needed, num_pages, max_blocks, order)
    case = PagedCase("skewed", batch, Hq, Hkv, D, P, num_pages, NHD, max_blocks, bt, L,
                     1.0 / math.sqrt(D), q=_randn_bf16((batch, Hq, D), g, "cpu").to(device))
    case.k_new = _randn_bf16((batch, Hkv, D), g, "cpu").to(device)
    case.v_new = _randn_bf16((batch, Hkv, D), g, "cpu").to(device)
    _fill_cache(case, g, device, "cpu")
    return case


def _serving_case(name: str, g: torch.Generator, q_lens: np.ndarray, L: np.ndarray, num_pages: int,
                  device) -> PagedCase:
    """A Qwen3-4B-shaped mixed step (Hq=32, Hkv=8, D=128, page 16, NHD): row b
    holds L[b] cached tokens and brings q_lens[b] new ones; pages for all of
    them from a seeded permutation of the num_pages pool."""
    Hq, Hkv, D, P = 32, 8, 128, 16
    B = len(q_lens)
    indptr = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(indptr[-1])
    needed = (L + q_lens + P - 1) // P
    max_blocks = int(needed.max())
    order = (torch.randperm(num_pages - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = assign_pages(needed, num_pages, max_blocks, order)
    case = PagedCase(name, B, Hq, Hkv, D, P, num_pages, NHD, max_blocks, bt, L.astype(np.int32),
                     1.0 / math.sqrt(D), q=_randn_bf16((T, Hq, D), g, "cpu").to(device), qo_indptr=indptr)
    case.k_new = _randn_bf16((T, Hkv, D), g, "cpu").to(device)
    case.v_new = _randn_bf16((T, Hkv, D), g, "cpu").to(device)
    _fill_cache(case, g, device, "cpu")
    return case


def spec_decode(device="cpu", seed: int = 6, batch: int = 32, q_len: int = 4, min_len: int = 512,
                max_len: int = 1024, num_pages: int = 65536) -> PagedCase:
    """Speculative decode on the Qwen3-4B-shaped layer: B=32 rows of q_len=4
    new tokens each on cached lengths uniform in [512, 1024], 65,536-page
    shuffled pool."""
    g = _gen(seed)
    L = torch.randint(min_len, max_len + 1, (batch,), generator=g).numpy().astype(np.int32)
    return _serving_case("spec", g, np.full(batch, q_len, np.int32), L, num_pages, device)


def chunked_mix(device="cpu", seed: int = 7, decode_rows: int = 60, chunks: int = 4, chunk_len: int = 496,
                num_pages: int = 65536) -> PagedCase:
    """A chunked-prefill serving step on the Qwen3-4B-shaped layer: `chunks`
    prefill chunks of chunk_len tokens on cached prefixes uniform in
    [0, 2048] (rows 0..chunks-1), then decode_rows single-token rows on
    lengths uniform in [512, 1024] -- 2,044 new tokens in all, 65,536-page
    shuffled pool."""
    g = _gen(seed)
    L_chunk = torch.randint(0, 2048 + 1, (chunks,), generator=g).numpy()
    L_dec = torch.randint(512, 1024 + 1, (decode_rows,), generator=g).numpy()
    q = np.concatenate([np.full(chunks, chunk_len), np.ones(decode_rows)]).astype(np.int32)
    L = np.concatenate([L_chunk, L_dec]).astype(np.int32)
    return _serving_case("chunked", g, q, L, num_pages, device)


def ragged_prefill(device="cpu", seed: int = 4, batch: int = 8, num_pages: int = 4096,
                   q_range=(65, 1023), extra_kv: int = 2048, num_q_heads: int = 48,
                   num_kv_heads: int = 6, head_dim: int = 256, page_size: int = 16,
                   layout: int = HND) -> PagedCase:
    """Ragged end-aligned causal prefill: B=8, Hq=48, Hkv=6, D=256, page 16
    HND, q uniform in [65, 1023], kv = q + uniform [0, 2048]."""
    g = _gen(seed)
    P = page_size
    qn = torch.randint(q_range[0], q_range[1] + 1, (batch,), generator=g).numpy().astype(np.int32)
    kv = (qn + torch.randint(0, extra_kv + 1, (batch,), generator=g).numpy()).astype(np.int32)
    indptr = np.concatenate([[0], np.cumsum(qn)]).astype(np.int32)
    needed = (kv + P - 1) // P
    max_blocks = int(needed.max())
    order = (torch.randperm(num_pages - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = assign_pages(needed, num_pages, max_blocks, order)
    total_q = int(indptr[-1])
    case = PagedCase("prefill", batch, num_q_heads, num_kv_heads, head_dim, P, num_pages, layout,
                     max_blocks, bt, np.zeros(batch, np.int32), 1.0 / math.sqrt(head_dim),
                     q=_randn_bf16((total_q, num_q_heads, head_dim), g, "cpu").to(device),
                     qo_indptr=indptr, kv_lens=kv)
    _fill_cache(case, g, device, "cpu")
    return case


def small_prefill(seed: int, q_lens, kv_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                  page_size: int, layout: int = HND, extra_pages: int = 3, device="cpu") -> PagedCase:
    """A ragged prefill problem of chosen lengths: request b has q_lens[b]
    queries over kv_lens[b] cached keys; pages from a seeded permutation,
    every slot without a token NaN."""
    g = _gen(seed)
    q_lens = np.asarray(q_lens, np.int32)
    kv_lens = np.asarray(kv_lens, np.int32)
    B = len(q_lens)
    P = page_size
    indptr = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    needed = (np.maximum(kv_lens, 0) + P - 1) // P
    num_pages = int(needed.sum()) + 1 + extra_pages
    max_blocks = max(int(needed.max()), 1)
    order = (torch.randperm(num_pages - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = assign_pages(needed, num_pages, max_blocks, order)
    case = PagedCase("prefill", B, num_q_heads, num_kv_heads, head_dim, P, num_pages, layout, max_blocks, bt,
                     np.zeros(B, np.int32), 1.0 / math.sqrt(head_dim),
                     q=_randn_bf16((int(indptr[-1]), num_q_heads, head_dim), g, "cpu").to(device),
                     qo_indptr=indptr, kv_lens=kv_lens)
    _fill_cache(case, g, device, "cpu")
    return case


def mixed_step(seed: int, q_lens, cache_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
               page_size: int, layout: int = NHD, extra_pages: int = 3, device="cpu") -> PagedCase:
    """One step of a mixed batch: row b holds cache_lens[b] cached tokens
    (negative: an inactive row) and brings q_lens[b] new tokens -- q, k_new
    and v_new are [sum q_lens, H, D] with row b's tokens at qo_indptr[b] ..
    qo_indptr[b+1]-1.  Pages for cache_lens[b] + q_lens[b] tokens come from a
    seeded permutation; every slot without a cached token is NaN."""
    g = _gen(seed)
    q_lens = np.asarray(q_lens, np.int32)
    L = np.asarray(cache_lens, np.int32)
    B = len(q_lens)
    P = page_size
    indptr = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    T = int(indptr[-1])
    needed = (np.maximum(L, 0) + np.where(L >= 0, q_lens, 0) + P - 1) // P
    num_pages = int(needed.sum()) + 1 + extra_pages
    max_blocks = max(int(needed.max()) if B else 1, 1)
    order = (torch.randperm(num_pages - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = assign_pages(needed, num_pages, max_blocks, order)
    case = PagedCase("mixed", B, num_q_heads, num_kv_heads, head_dim, P, num_pages, layout, max_blocks, bt, L,
                     1.0 / math.sqrt(head_dim), q=_randn_bf16((T, num_q_heads, head_dim), g, "cpu").to(device),
                     qo_indptr=indptr)
    case.k_new = _randn_bf16((T, num_kv_heads, head_dim), g, "cpu").to(device)
    case.v_new = _randn_bf16((T, num_kv_heads, head_dim), g, "cpu").to(device)
    _fill_cache(case, g, device, "cpu")
    return case


@dataclass
class SweepCase:
    """The batch sweep: ``layers`` per-layer K/V pools that share one block
    table; row b starts with ``prompt_lens[b]`` tokens and grows by one per
    decode step."""

    batch: int
    layers: int
    contiguous: bool
    page_size: int
    num_pages: int
    max_blocks: int
    block_table: np.ndarray
    prompt_lens: np.ndarray
    k_caches: list
    v_caches: list
    num_q_heads: int = 32
    num_kv_heads: int = 8
    head_dim: int = 128
    softmax_scale: float = 1.0 / math.sqrt(128)


def batch_sweep(batch: int, device="cuda", contiguous: bool = True, layers: int = SWEEP_LAYERS,
                decode_steps: int = SWEEP_DECODE_STEPS, seed: int | None = None,
                data_device=None, fill_decode: bool = False) -> SweepCase:
    """Batch-sweep state: prompt K/V pre-filled in every layer's pool, every
    slot past the prompt NaN.  Pages for prompt + ``decode_steps`` tokens are
    reserved up front, sequentially (contiguous) or from a seeded permutation
    (shuffled).  Random draws for the caches are made on ``data_device``
    (default: ``device``) so multi-GB pools fill quickly.

    fill_decode: also fill the ``decode_steps`` slots after the prompt with
    seeded tokens, as earlier decode steps would have appended them, so that
    any decode step can be run first and attends finite values only."""
    seed = 2 if seed is None else seed
    g = _gen(seed)
    data_device = device if data_device is None else data_device
    gd = _gen(seed, data_device)
    P, Hkv, D = 128, 8, 128
    prompt = torch.randint(64, 512 + 1, (batch,), generator=g).numpy().astype(np.int32)
    max_blocks = (512 + decode_steps + P - 1) // P
    needed = (prompt + decode_steps + P - 1) // P
    num_pages = int(needed.sum()) + 1
    if contiguous:
        order = np.arange(1, num_pages, dtype=np.int32)
    else:
        order = (torch.randperm(num_pages - 1, generator=g).numpy() + 1).astype(np.int32)
    bt = assign_pages(needed, num_pages, max_blocks, order)
    filled = prompt + (decode_steps if fill_decode else 0)
    b_idx = np.concatenate([np.full(int(n), b, np.int64) for b, n in enumerate(filled)])
    t_idx = np.concatenate([np.arange(int(n), dtype=np.int64) for n in filled])
    pages, slots = bt[b_idx, t_idx // P], t_idx % P
    shape = (num_pages, P, Hkv, D)
    ks, vs = [], []
    for _ in range(layers):
        kc, vc = _nan_pool(shape, device), _nan_pool(shape, device)
        scatter_tokens(kc, NHD, P, pages, slots, _randn_bf16((t_idx.size, Hkv, D), gd, data_device).to(device))
        scatter_tokens(vc, NHD, P, pages, slots, _randn_bf16((t_idx.size, Hkv, D), gd, data_device).to(device))
        ks.append(kc)
        vs.append(vc)
    return SweepCase(batch, layers, contiguous, P, num_pages, max_blocks, bt, prompt, ks, vs)


def sweep_step_inputs(sw: SweepCase, step: int, device="cuda", layers=None):
    """Per-layer (q, k_new, v_new) for decode step ``step`` (seed 1000*B + step)."""
    g = _gen(1000 * sw.batch + step, device)
    n = sw.layers if layers is None else layers
    B, Hq, Hkv, D = sw.batch, sw.num_q_heads, sw.num_kv_heads, sw.head_dim
    out = []
    for _ in range(n):
        out.append((_randn_bf16((B, Hq, D), g, device), _randn_bf16((B, Hkv, D), g, device),
                    _randn_bf16((B, Hkv, D), g, device)))
    return out


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def compact_rows(k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: np.ndarray, rows,
                 lens_needed, page_size: int):
    """Host copy of only the pages that ``rows`` use (for the first
    ``lens_needed[b]`` tokens), renumbered 1..n with page 0 kept as a null
    page.  Returns ``(k_pages, v_pages, block_table_rows)``: a small pool
    with the same geometry and a block table restricted to ``rows``."""
    rows = list(rows)
    max_blocks = block_table.shape[1]
    bt = np.zeros((len(rows), max_blocks), np.int32)
    src = [0]
    for i, b in enumerate(rows):
        nb = min((int(lens_needed[i]) + page_size - 1) // page_size, max_blocks)
        for j in range(nb):
            src.append(int(block_table[b, j]))
            bt[i, j] = len(src) - 1
    idx = torch.as_tensor(np.array(src, np.int64), device=k_cache.device)
    k = bits(k_cache.index_select(0, idx))
    v = bits(v_cache.index_select(0, idx))
    return np.ascontiguousarray(k), np.ascontiguousarray(v), bt
