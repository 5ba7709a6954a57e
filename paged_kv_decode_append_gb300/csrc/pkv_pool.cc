// pkv_pool.cc -- host page pool and block-table helpers.
//
// "flex_attention + paged KV + CUDA graphs vs vLLM": pages are handed out
// from a pool in which page 0 is reserved as the null / padding slot ("Why
// this works", point 3), and on a fresh batch PageTable.reserve hands pages
// out sequentially, which is what makes a row's blocks contiguous ("What
// each option did", BLOCKS_ARE_CONTIGUOUS).  This pool does the same: a
// LIFO-free stack that starts as 1, 2, 3, ... so a fresh pool allocates in
// ascending order; pkv_pool_shuffle scatters it for the shuffled layout.
#include <stdint.h>
#include <stdlib.h>

#include <new>
#include <vector>

#include "pkv.h"

struct pkv_pool {
    int32_t num_pages;
    std::vector<int32_t> free_stack; // top = back(); next page handed out
    std::vector<uint8_t> is_free;    // by page id
};

namespace {

uint64_t splitmix64(uint64_t *state)
{
    uint64_t z = (*state += 0x9e3779b97f4a7c15ull);
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

int32_t blocks_for(int64_t len, int32_t page_size)
{
    return (int32_t)((len + page_size - 1) / page_size);
}

} // namespace

extern "C" {

pkv_pool *pkv_pool_create(int32_t num_pages)
{
    if (num_pages < 2)
        return nullptr;
    pkv_pool *p = new (std::nothrow) pkv_pool;
    if (p == nullptr)
        return nullptr;
    try {
        p->num_pages = num_pages;
        p->free_stack.reserve((size_t)num_pages - 1);
        for (int32_t i = num_pages - 1; i >= 1; --i) // pop order: 1, 2, 3, ...
            p->free_stack.push_back(i);
        p->is_free.assign((size_t)num_pages, 1);
        p->is_free[0] = 0;
    } catch (...) {
        delete p;
        return nullptr;
    }
    return p;
}

void pkv_pool_destroy(pkv_pool *pool)
{
    delete pool;
}

int32_t pkv_pool_num_free(const pkv_pool *pool)
{
    return pool == nullptr ? 0 : (int32_t)pool->free_stack.size();
}

pkv_status pkv_pool_alloc(pkv_pool *pool, int32_t n, int32_t *pages_out)
{
    if (pool == nullptr || n < 0 || (n > 0 && pages_out == nullptr))
        return PKV_EINVAL;
    if ((size_t)n > pool->free_stack.size())
        return PKV_ENOPAGES;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t page = pool->free_stack.back();
        pool->free_stack.pop_back();
        pool->is_free[(size_t)page] = 0;
        pages_out[i] = page;
    }
    return PKV_OK;
}

pkv_status pkv_pool_free(pkv_pool *pool, const int32_t *pages, int32_t n)
{
    if (pool == nullptr || n < 0 || (n > 0 && pages == nullptr))
        return PKV_EINVAL;
    // validate everything first (including duplicates within `pages`)
    std::vector<uint8_t> seen;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t page = pages[i];
        if (page < 1 || page >= pool->num_pages || pool->is_free[(size_t)page])
            return PKV_EINVAL;
    }
    seen.assign((size_t)pool->num_pages, 0);
    for (int32_t i = 0; i < n; ++i) {
        if (seen[(size_t)pages[i]])
            return PKV_EINVAL;
        seen[(size_t)pages[i]] = 1;
    }
    for (int32_t i = n - 1; i >= 0; --i) { // the first page returned is the next handed out
        pool->free_stack.push_back(pages[i]);
        pool->is_free[(size_t)pages[i]] = 1;
    }
    return PKV_OK;
}

pkv_status pkv_pool_shuffle(pkv_pool *pool, uint64_t seed)
{
    if (pool == nullptr)
        return PKV_EINVAL;
    uint64_t state = seed;
    std::vector<int32_t> &s = pool->free_stack;
    for (size_t i = s.size(); i > 1; --i) {
        const size_t j = (size_t)(splitmix64(&state) % i);
        const int32_t t = s[i - 1];
        s[i - 1] = s[j];
        s[j] = t;
    }
    return PKV_OK;
}

pkv_status pkv_table_reserve(pkv_pool *pool, int32_t *row, int32_t max_blocks, int32_t page_size, int32_t cur_len,
                             int32_t new_len)
{
    if (pool == nullptr || row == nullptr || max_blocks < 1 || page_size < 1 || cur_len < 0 || new_len < cur_len)
        return PKV_EINVAL;
    const int32_t have = blocks_for(cur_len, page_size);
    const int32_t need = blocks_for(new_len, page_size);
    if (need > max_blocks)
        return PKV_EINVAL;
    if (need == have)
        return PKV_OK;
    return pkv_pool_alloc(pool, need - have, row + have);
}

pkv_status pkv_table_release(pkv_pool *pool, int32_t *row, int32_t max_blocks, int32_t page_size, int32_t len)
{
    if (pool == nullptr || row == nullptr || max_blocks < 1 || page_size < 1 || len < 0)
        return PKV_EINVAL;
    const int32_t n = blocks_for(len, page_size);
    if (n > max_blocks)
        return PKV_EINVAL;
    const pkv_status st = pkv_pool_free(pool, row, n);
    if (st != PKV_OK)
        return st;
    for (int32_t i = 0; i < n; ++i)
        row[i] = 0;
    return PKV_OK;
}

pkv_status pkv_validate_host(const pkv_cache_desc *desc, const int32_t *block_table, int32_t max_blocks,
                             const int32_t *seqlens, int32_t batch, int32_t extra_tokens, int32_t *bad_row)
{
    if (bad_row != nullptr)
        *bad_row = -1;
    if (desc == nullptr || desc->page_size < 1 || desc->num_pages < 2 || max_blocks < 1 || batch < 0 ||
        extra_tokens < 0 || (batch > 0 && (block_table == nullptr || seqlens == nullptr)))
        return PKV_EINVAL;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t L = seqlens[b];
        if (L < 0)
            continue; // inactive row
        const int64_t len = L + extra_tokens;
        bool ok = len <= (int64_t)max_blocks * desc->page_size;
        for (int64_t k = 0; ok && k < blocks_for(len, desc->page_size); ++k) {
            const int32_t page = block_table[(int64_t)b * max_blocks + k];
            ok = page >= 1 && page < desc->num_pages;
        }
        if (!ok) {
            if (bad_row != nullptr)
                *bad_row = b;
            return PKV_EINVAL;
        }
    }
    return PKV_OK;
}

} // extern "C"
